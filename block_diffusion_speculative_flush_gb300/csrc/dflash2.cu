// DFlash2 on the GPU: the block-local dynamic convolution of each layer and
// the candidate selector that draws a block's tokens one position after the
// other, each conditioned on its predecessor (the DFlash2 commit note of
// ollama's mlxrunner/dflash.go, and the BlockSelector branch of selectBlock).
//
//  * k_dynconv: h_i += sum_j w_ij * x_{i-j}, x = RMSNorm(h; conv_norm), over
//    the block's own rows (the anchor's row is the first; nothing before it),
//    with per-row kernel weights w_i = softmax over the taps of one channel
//    group's entries of W_dc x_i (the product runs as an ordinary GEMM).
//  * k_topk_partial / k_topk_merge: the sel_candidates largest logits of
//    each block row in the sampler's order (value descending, then id), as a
//    per-chunk selection whose chunk of 4096 entries stays in registers, then
//    a merge of the chunks' candidates by one warp per row.
//  * k_select: one warp per session and one lane per candidate walks the
//    block's positions in order: score = logit + <A[prev], B[candidate]>
//    with prev the token chosen one position earlier (the anchor at the
//    first), Gumbel-max over the candidates at the request temperature (the
//    draft's Philox stream, keyed by the candidate's id), and the candidate
//    distribution softmax(score / T) kept for verification.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "launch.h"

namespace dfl {

namespace {

constexpr int kConvThreads = 256;
constexpr int kTopkThreads = 256;
constexpr int kTopkPer = 16;                         // entries per thread of a chunk
constexpr int kTopkChunk = kTopkThreads * kTopkPer;  // 4096

template <typename T>
__global__ void __launch_bounds__(kConvThreads) k_dynconv(T* __restrict__ h, const T* __restrict__ x,
                                                         const float* __restrict__ a, int nrows, int H, int G,
                                                         int taps) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x, i = row % nrows, gw = H / G;
  const float* ar = a + (int64_t)row * G * taps;
  const int nt = min(taps, i + 1);  // taps before the anchor's row read zeros
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    const float* ag = ar + (c / gw) * taps;
    float mx = -INFINITY;
    for (int j = 0; j < taps; ++j) mx = fmaxf(mx, ag[j]);
    float e[kMaxConvTaps], sum = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxConvTaps; ++j) {
      e[j] = j < taps ? expf(ag[j] - mx) : 0.f;
      sum += e[j];
    }
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxConvTaps; ++j)
      if (j < nt) acc += (e[j] / sum) * to_f(x[(int64_t)(row - j) * H + c]);
    T* hp = h + (int64_t)row * H + c;
    *hp = from_f<T>(to_f(*hp) + acc);
  }
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Candidates of one chunk of one row: the kc largest order keys among the
// chunk's entries, largest first (0: fewer comparable entries than kc).
__global__ void __launch_bounds__(kTopkThreads) k_topk_partial(const float* const* __restrict__ rows, int rows_per_seq,
                                                              int64_t ld, int V, int kc, uint64_t* __restrict__ part) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint64_t sm[kTopkThreads / 32];
  const int r = blockIdx.x, ch = blockIdx.y, nch = gridDim.y;
  const float* row = rows[r / rows_per_seq] + (int64_t)(r % rows_per_seq) * ld;
  uint64_t key[kTopkPer];
#pragma unroll
  for (int k = 0; k < kTopkPer; ++k) {
    const int v = ch * kTopkChunk + k * kTopkThreads + (int)threadIdx.x;
    key[k] = v < V ? order_key(row[v], v) : 0ull;
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint64_t* out = part + ((int64_t)r * nch + ch) * kc;
  for (int t = 0; t < kc; ++t) {
    uint64_t best = 0ull;
#pragma unroll
    for (int k = 0; k < kTopkPer; ++k) best = key[k] > best ? key[k] : best;
    best = warp_max_u64(best);
    if (lane == 0) sm[w] = best;
    __syncthreads();
    uint64_t win = 0ull;
#pragma unroll
    for (int i = 0; i < kTopkThreads / 32; ++i) win = sm[i] > win ? sm[i] : win;
    __syncthreads();
    if (threadIdx.x == 0) out[t] = win;
    // keys are distinct (the id is part of the key): the one holder drops it
#pragma unroll
    for (int k = 0; k < kTopkPer; ++k)
      if (win && key[k] == win) key[k] = 0ull;
  }
}

// One warp per row: the kc largest of the chunks' candidates, as ids and
// logits in the sampler's order.
__global__ void k_topk_merge(const uint64_t* __restrict__ part, int nch, int kc, int32_t* __restrict__ ids,
                             float* __restrict__ logit, int rows) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= rows) return;
  const uint64_t* p = part + (int64_t)r * nch * kc;
  const int m = nch * kc;
  uint64_t prev = ~0ull;
  for (int t = 0; t < kc; ++t) {
    uint64_t best = 0ull;
    for (int i = lane; i < m; i += 32)
      if (p[i] < prev && p[i] > best) best = p[i];
    best = warp_max_u64(best);
    prev = best;
    if (lane == 0) {
      ids[(int64_t)r * kc + t] = best ? (int32_t)(0xffffffffu - (uint32_t)best) : 0;
      logit[(int64_t)r * kc + t] = best ? float_of_order((uint32_t)(best >> 32)) : -INFINITY;
    }
  }
}

// One warp per session of the call (compact index j): positions 0..n-1 in
// order, lane c holding candidate c.
template <typename T>
__global__ void k_select(SelectArgs a) {
  pdl_trigger();
  pdl_wait();
  const int j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (j >= a.B) return;
  const int n = a.n, kc = a.kc, r = a.rank;
  const int caller = a.sess_map ? a.sess_map[j] : j;
  const uint32_t seq = a.seq_ids ? (uint32_t)a.seq_ids[j] : (uint32_t)j;
  const T* A = (const T*)a.sel_prev;
  const T* Bt = (const T*)a.sel_next;
  int prev = a.current[caller];
  if (prev < 0 || prev >= a.V) {
    if (lane == 0) atomicOr(a.err, 1);
    prev = 0;
  }
  const bool live = lane < kc;
  for (int i = 0; i < n; ++i) {
    const int64_t row = (int64_t)j * n + i;
    const int id = live ? a.cand_ids[row * kc + lane] : 0;
    float score = -INFINITY;
    if (live) {
      float dot = 0.f;
      const T* ap = A + (int64_t)prev * r;
      const T* bp = Bt + (int64_t)id * r;
      for (int k = 0; k < r; ++k) dot += to_f(ap[k]) * to_f(bp[k]);
      score = a.cand_logit[row * kc + lane] + dot;
    }
    float z = score;
    if (a.temperature > 0.f && live)
      z = score / a.temperature + gumbel(a.seed, a.rnd, kStreamDraft, seq, (uint32_t)(i + 1), (uint32_t)id);
    // argmax over the candidates, ties to the earlier candidate
    ArgMax best{live ? z : -INFINITY, live ? lane : INT32_MAX};
    best = warp_argmax(best);
    const int win = best.i >= 0 && best.i < kc ? best.i : 0;
    float prob;
    if (a.temperature > 0.f) {
      const float s = live ? score / a.temperature : -INFINITY;
      const float m = warp_max(s);
      const float e = live ? expf(s - m) : 0.f;
      prob = e / warp_sum(e);
    } else {
      prob = lane == win ? 1.f : 0.f;
    }
    const int tok = __shfl_sync(0xffffffffu, id, win);
    const float qt = __shfl_sync(0xffffffffu, prob, win);
    if (live) {
      a.sess_ids[j][i * kc + lane] = id;
      a.sess_probs[j][i * kc + lane] = prob;
    }
    if (lane == 0) {
      a.sess_tok[j][i] = tok;
      a.out_tokens[(int64_t)caller * n + i] = tok;
      a.out_q[(int64_t)caller * n + i] = qt;
    }
    prev = tok;
  }
}

}  // namespace

void launch_dynconv(DT dt, void* h, const void* x, const float* a, int rows, int nrows, int H, int G, int taps,
                    cudaStream_t st) {
  if (rows <= 0) return;
  if (dt == DT::BF16)
    launch_k(k_dynconv<bf16>, rows, kConvThreads, 0, st, (bf16*)h, (const bf16*)x, a, nrows, H, G, taps);
  else
    launch_k(k_dynconv<float>, rows, kConvThreads, 0, st, (float*)h, (const float*)x, a, nrows, H, G, taps);
}

int topk_chunks(int V) { return (V + kTopkChunk - 1) / kTopkChunk; }

void launch_topk_candidates(const float* const* rows, int rows_per_seq, int64_t ld, int V, int kc, int n_rows,
                            uint64_t* part, int32_t* ids, float* logit, cudaStream_t st) {
  if (n_rows <= 0) return;
  const int nch = topk_chunks(V);
  launch_k(k_topk_partial, dim3(n_rows, nch), kTopkThreads, 0, st, rows, rows_per_seq, ld, V, kc, part);
  launch_k(k_topk_merge, (unsigned)((n_rows + 3) / 4), 128, 0, st, (const uint64_t*)part, nch, kc, ids, logit, n_rows);
}

void launch_select(DT dt, const SelectArgs& a, cudaStream_t st) {
  if (a.B <= 0) return;
  const unsigned grid = (unsigned)((a.B + 3) / 4);
  if (dt == DT::BF16)
    launch_k(k_select<bf16>, grid, 128, 0, st, a);
  else
    launch_k(k_select<float>, grid, 128, 0, st, a);
}

}  // namespace dfl
