// Device helpers shared by the DFlash kernels: storage conversions, warp and
// block reductions, the counter-based random numbers the round draws, and the
// RMSNorm row statistic.  Written for sm_103a.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfl {

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------------------
// storage <-> fp32
// ---------------------------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum over the whole block; every thread gets the result.  `red` must hold
// at least blockDim.x / 32 floats.  Summation order is fixed by the block
// shape, never by the data or by other rows.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float s = 0.f;
  for (int i = 0; i < nw; ++i) s += red[i];
  return s;
}

// (value, index) argmax with the lowest index winning ties.
struct ArgMax {
  float v;
  int32_t i;
};
__device__ __forceinline__ ArgMax better(ArgMax a, ArgMax b) {
  if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
  return a;
}
// ---------------------------------------------------------------------------
// the sampler's order: value descending, then id ascending
// ---------------------------------------------------------------------------
// Monotone map of a float to uint32 (a larger float gives a larger word;
// -0 is taken as +0); NaN maps to 0.
__device__ __forceinline__ uint32_t float_order(float s) {
  if (s != s) return 0u;
  uint32_t u = s == 0.f ? 0u : __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float float_of_order(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
// Key of entry v with scaled score s: a larger key comes first in the order;
// NaN keys are 0.  A truncated distribution keeps the entries whose key is at
// least its cut (cut 0: all entries).
__device__ __forceinline__ uint64_t order_key(float s, int v) {
  const uint32_t o = float_order(s);
  return o ? ((uint64_t)o << 32) | (uint64_t)(0xffffffffu - (uint32_t)v) : 0ull;
}

__device__ __forceinline__ ArgMax warp_argmax(ArgMax a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ArgMax b;
    b.v = __shfl_xor_sync(0xffffffffu, a.v, o);
    b.i = __shfl_xor_sync(0xffffffffu, a.i, o);
    a = better(a, b);
  }
  return a;
}

// ---------------------------------------------------------------------------
// Philox4x32-10: Salmon, Moraes, Dror & Shaw, "Parallel Random Numbers: As
// Easy as 1, 2, 3" (SC'11).  Ten rounds of two 32x32->64 multiplies by the
// paper's constants; the high halves are xored with the other two counter
// words and the key, the key advancing by the two Weyl constants between
// rounds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k.x += 0x9E3779B9u;
      k.y += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
  }
  return c;
}

enum : uint32_t { kStreamDraft = 0, kStreamAccept = 1, kStreamBonus = 2 };

// The random word for index v (a vocabulary entry, or 0 for a row's single
// draw): word v & 3 of Philox at counter (v >> 2, row | stream << 16, seq,
// round), key = seed.  One evaluation serves four consecutive indices.
__device__ __forceinline__ uint4 rand_block(uint64_t seed, uint32_t rnd, uint32_t stream, uint32_t seq, uint32_t row,
                                           uint32_t blk) {
  const uint4 c = make_uint4(blk, (row & 0xFFFFu) | (stream << 16), seq, rnd);
  const uint2 k = make_uint2((uint32_t)seed, (uint32_t)(seed >> 32));
  return philox4x32_10(c, k);
}
__device__ __forceinline__ uint32_t rand_u32(uint64_t seed, uint32_t rnd, uint32_t stream,
                                             uint32_t seq, uint32_t row, uint32_t v) {
  const uint4 r = rand_block(seed, rnd, stream, seq, row, v >> 2);
  const uint32_t w = v & 3u;
  return w == 0 ? r.x : w == 1 ? r.y : w == 2 ? r.z : r.w;
}

// u = ((x >> 9) + 0.5) * 2^-23: strictly inside (0, 1) and exact in fp32.
__device__ __forceinline__ float uniform_open(uint32_t x) {
  return ((float)(x >> 9) + 0.5f) * 1.1920928955078125e-07f;
}

// Gumbel noise -log(-log u).  The logarithms run on the special-function
// unit (__logf, relative error near 1e-6): a draw moves only where two scores
// agree to that precision.
__device__ __forceinline__ float gumbel_of(uint32_t x) { return -__logf(-__logf(uniform_open(x))); }

__device__ __forceinline__ float gumbel(uint64_t seed, uint32_t rnd, uint32_t stream, uint32_t seq,
                                        uint32_t row, uint32_t v) {
  return gumbel_of(rand_u32(seed, rnd, stream, seq, row, v));
}
__device__ __forceinline__ uint32_t word_of(const uint4& r, int w) {
  return w == 0 ? r.x : w == 1 ? r.y : w == 2 ? r.z : r.w;
}

// ---------------------------------------------------------------------------
// Bounded waits: a spin that runs past its limit records where it gave up in
// a device error word that the host reads after the call.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: every kernel lets the next one in the stream
// be scheduled early (trigger) and waits for the previous one to finish and
// flush its memory before reading anything it produced (wait).  Without the
// launch attribute both are no-ops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// p as the compiler must take it from here on: its value is opaque until this
// point, so no load through the result can be scheduled before it.  Pointers
// to what an earlier kernel of the chain writes pass through it right after
// the wait, and such data is read with plain (coherent) loads: a read-only
// (__ldg) load is only valid for memory that no kernel writes while this one
// runs, and with programmatic launch the previous kernel still runs when
// this one starts.
template <typename T>
__device__ __forceinline__ T* after_wait(T* p) {
  asm volatile("" : "+l"(p)::"memory");
  return p;
}

}  // namespace dfl
