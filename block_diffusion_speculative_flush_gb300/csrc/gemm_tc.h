// Weight-streaming matrix product on the sm_103a tensor cores (tcgen05 with
// TMEM accumulators, operands staged by TMA).  Internal interface.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dfl {

struct TcContext;

// err: device word the kernels set bit 4 of when a bounded wait expires.
int tc_create(TcContext** out, int num_sms, int* err);
void tc_destroy(TcContext* c);
const char* tc_last_error();

// Y[M][N] (fp32, row stride ldy) = X[M][K] . W[N][K]^T with bf16 X and W.
// Needs K % 64 == 0, ldx and ldw multiples of 8 elements and 16-byte aligned
// X / W; any M >= 1 and N >= 1.  The k order of every output element
// depends on N and K only (never on M), so a row's result does not change
// with the number of rows in the call.
int tc_gemm(TcContext* c, const void* X, int64_t ldx, const void* W, int64_t ldw, float* Y, int64_t ldy, int M, int N,
            int K, cudaStream_t st);

}  // namespace dfl
