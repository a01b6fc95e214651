// Weight-streaming matrix product on the sm_103a tensor cores (tcgen05 with
// TMEM accumulators, operands staged by TMA).  Internal interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfl {

struct TcContext;

// err: device word the kernels set bit 4 of when a bounded wait expires.
int tc_create(TcContext** out, int num_sms, int* err);
void tc_destroy(TcContext* c);
const char* tc_last_error();

enum TcMode {
  kF32 = 0,        // Y fp32 [M][ldy]: Y = X W^T
  kResidBf16 = 1,  // Y bf16 [M][ldy]: Y = bf16(Y + X W^T), the residual add
  kSwigluBf16 = 2  // Y bf16 [M][ldy]: Y = bf16(silu(X Wg^T) * (X Wu^T)), W = Wg, W2 = Wu
};

// Weight-streaming product with bf16 X [M][K] and W [N][K] (and W2 for
// SwiGLU, N = the intermediate width).  Needs K % 64 == 0, ldx and ldw
// multiples of 8 elements and 16-byte aligned operands; any M, N >= 1.  The
// k order of every output element depends on N and K only (never on M), so
// a row's result does not change with the number of rows in the call.
// With yseg (device table, kF32 only) output rows [j*seg_rows, (j+1)*seg_rows)
// go to the buffer yseg[j] (row stride ldy, 16-byte aligned) instead of
// Y + row * ldy; Y is then unused.  ws (kResidBf16 only, may be NULL): an
// fp32 [M][N] scratch that lets many-row calls use 256-wide tiles, holding
// the running sum of the K splits; its contents are overwritten.
// late_trigger: the next kernel in the stream starts only once this one's
// CTAs are past their wait for the previous kernel, so that everything
// enqueued before this call has finished when it starts.
int tc_gemm(TcContext* c, const void* X, int64_t ldx, const void* W, const void* W2, int64_t ldw, void* Y, int64_t ldy,
            int M, int N, int K, int mode, cudaStream_t st, void* const* yseg = nullptr, int seg_rows = 0,
            float* ws = nullptr, int late_trigger = 0);

// `groups` independent fp32 products of one shape in one persistent launch of
// 256-wide tiles: X stacked [groups * M][ldx], W stacked [groups * N][ldw],
// product g into Y + g * y_group (rows ldy apart).  Each product sums its K
// splits exactly as tc_gemm does for that shape, so its results are the same
// bits as a separate call's.
int tc_gemm_grouped(TcContext* c, const void* X, int64_t ldx, const void* W, int64_t ldw, float* Y, int64_t ldy,
                    int64_t y_group, int M, int N, int K, int groups, cudaStream_t st);

// TMA maps of a session's K/V cache for the attention kernel: out[0] views
// the K planes ([planes][cap][d], 64 x 64 boxes), out[1] the V^T planes
// ([planes][d][cap], 64-position x d boxes).  cap must be a multiple of 64.
int tc_encode_kv_maps(TcContext* c, const void* kv, int64_t cap, int d, int planes, CUtensorMap* out);

}  // namespace dfl
