// A small fp32 target decoder on the GPU: the model that a DFlash draft
// speculates for.  It produces what the draft consumes (the hidden-state taps
// of every position: the embedding output and the residual stream after each
// attention and each MLP) and what verify consumes (raw next-token logits),
// and rolls its cache back after a rejection.
//
// The pages run the draft against a real target (ollama's mlxrunner, the
// mlxcel Laguna PR's verify forward with its 5-tap capture and rollback
// trim); here a random-init dense decoder stands in: RMSNorm, RoPE (rotate
// half), causal multi-head attention over its cache, SwiGLU MLP.  A forward
// over R rows appends them at positions start..start+R-1; every row attends
// to the cache and to the earlier rows of the call, so a multi-row verify
// forward and token-by-token decoding compute the same rows.
//
// It reuses the draft's CUDA-core kernels: the RMSNorm, the split-key
// attention and its merge (the new rows are the "block" rows, causal among
// themselves), the residual add, SwiGLU and the row copy for the taps; its
// matrix products are a skinny warp-per-column kernel (k_gemm_rows).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <vector>

#include "common.cuh"
#include "dflash.h"
#include "kernels.h"
#include "launch.h"

extern "C" int dflash__set_error(int code, const char* msg);

namespace dfl {
namespace {

inline unsigned cdivu(int64_t a, int64_t b) { return (unsigned)((a + b - 1) / b); }

// x[i] = E[tokens[i]]; an id outside [0, V) sets bit 1 of *err and reads row 0.
__global__ void k_gather_rows(const float* __restrict__ E, const int32_t* __restrict__ tokens, int V, int H,
                              float* __restrict__ x, int32_t* __restrict__ err) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  int t = tokens[r];
  if (t < 0 || t >= V) {
    if (threadIdx.x == 0) atomicOr(err, 1);
    t = 0;
  }
  for (int j = threadIdx.x; j < H; j += blockDim.x) x[(int64_t)r * H + j] = E[(int64_t)t * H + j];
}

// Per (row, head): rotate-half RoPE of q and k from the row's cos/sin table,
// q to Q [rows][nh][d], k and v into the cache at the row's position.  Cache
// planes as the draft's: K (2l)*nh + h is [cap][d], V (2l+1)*nh + h is
// [d][cap].
__global__ void k_target_qkv(const float* __restrict__ qkv, const float2* __restrict__ rope, int nh, int d,
                             int64_t start, int64_t cap, int layer, float* __restrict__ Q, float* __restrict__ kv) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, h = blockIdx.y;
  const int half = d / 2, qd = nh * d;
  const float* row = qkv + (int64_t)r * 3 * qd;
  const float2* rt = rope + (int64_t)r * half;
  const int64_t slot = (start + r) % cap;
  float* kp = kv + ((int64_t)(2 * layer) * nh + h) * cap * d + slot * d;
  float* vp = kv + ((int64_t)(2 * layer + 1) * nh + h) * cap * d + slot;
  for (int j = threadIdx.x; j < half; j += blockDim.x) {
    const float2 cs = rt[j];
    const float qa = row[h * d + j], qb = row[h * d + j + half];
    const float ka = row[qd + h * d + j], kb = row[qd + h * d + j + half];
    Q[((int64_t)r * nh + h) * d + j] = qa * cs.x - qb * cs.y;
    Q[((int64_t)r * nh + h) * d + j + half] = qb * cs.x + qa * cs.y;
    kp[j] = ka * cs.x - kb * cs.y;
    kp[j + half] = kb * cs.x + ka * cs.y;
  }
  for (int j = threadIdx.x; j < d; j += blockDim.x) vp[(int64_t)j * cap] = row[2 * qd + h * d + j];
}

// Y[M][N] = X[M][K] . W[N][K]^T for few rows: one warp per output column n,
// lanes striding K by float4 (lane l takes k = 4l + 128j), eight rows per
// pass, then a butterfly sum.  A row's arithmetic (its lane partition and the
// reduction tree) does not depend on M or on which pass holds it, so a
// multi-row forward and one-row forwards give bit-identical rows.  Rows are
// 16-byte aligned (K, ldx, ldw multiples of 4).
__global__ void __launch_bounds__(256) k_gemm_rows(const float* __restrict__ X, int64_t ldx,
                                                   const float* __restrict__ W, int64_t ldw, float* __restrict__ Y,
                                                   int64_t ldy, int M, int N, int K) {
  pdl_trigger();
  pdl_wait();
  X = after_wait(X);  // the previous kernel's rows
  const int lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (n >= N) return;
  const float4* w4 = reinterpret_cast<const float4*>(W + (int64_t)n * ldw);
  const int K4 = K >> 2;
  for (int m0 = 0; m0 < M; m0 += 8) {
    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = 0.f;
    for (int k = lane; k < K4; k += 32) {
      const float4 w = __ldg(w4 + k);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (m0 + r < M) {
          const float4 x = reinterpret_cast<const float4*>(X + (int64_t)(m0 + r) * ldx)[k];
          float a = acc[r];
          a = fmaf(x.x, w.x, a);
          a = fmaf(x.y, w.y, a);
          a = fmaf(x.z, w.z, a);
          a = fmaf(x.w, w.w, a);
          acc[r] = a;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float v = warp_sum(acc[r]);
      if (lane == 0 && m0 + r < M) Y[(int64_t)(m0 + r) * ldy + n] = v;
    }
  }
}

void launch_gemm_rows(const float* X, int64_t ldx, const float* W, int64_t ldw, float* Y, int64_t ldy, int M, int N,
                      int K, cudaStream_t st) {
  if (M <= 0 || N <= 0) return;
  launch_k(k_gemm_rows, (unsigned)((N + 7) / 8), 256, 0, st, X, ldx, W, ldw, Y, ldy, M, N, K);
}

// Greedy choice of each row (lowest index on a tie), for the speculative loop.
__global__ void k_row_argmax(const float* __restrict__ logits, int V, int32_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  ArgMax best{-INFINITY, INT32_MAX};
  for (int v = threadIdx.x; v < V; v += blockDim.x) best = better(best, ArgMax{logits[(int64_t)r * V + v], v});
  best = warp_argmax(best);
  __shared__ ArgMax sm[32];
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    ArgMax b = sm[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) b = better(b, sm[w]);
    out[r] = b.i < 0 || b.i >= V ? 0 : b.i;
  }
}

// Best two entries of a row by (value descending, id ascending); NaN never
// enters (both comparisons are false for it).
struct Top2 {
  ArgMax a, b;
};
__device__ __forceinline__ bool beats(ArgMax x, ArgMax y) { return x.v > y.v || (x.v == y.v && x.i < y.i); }
__device__ __forceinline__ void top2_insert(Top2& t, ArgMax x) {
  if (beats(x, t.a)) {
    t.b = t.a;
    t.a = x;
  } else if (beats(x, t.b)) {
    t.b = x;
  }
}
__device__ __forceinline__ Top2 top2_merge(Top2 p, Top2 q) {
  Top2 r = p;
  top2_insert(r, q.a);
  top2_insert(r, q.b);
  return r;
}
__device__ __forceinline__ Top2 shfl_top2(Top2 t, int o) {
  Top2 u;
  u.a.v = __shfl_xor_sync(0xffffffffu, t.a.v, o);
  u.a.i = __shfl_xor_sync(0xffffffffu, t.a.i, o);
  u.b.v = __shfl_xor_sync(0xffffffffu, t.b.v, o);
  u.b.i = __shfl_xor_sync(0xffffffffu, t.b.i, o);
  return u;
}

// One CTA per row: the count of differing bytes of the two fp32 encodings
// and the top two of each arm.
__global__ void __launch_bounds__(256) k_logits_compare(const float* __restrict__ block,
                                                        const float* __restrict__ chain, int V,
                                                        dflash_exactness_row* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const ArgMax none{-INFINITY, INT32_MAX};
  Top2 tb{none, none}, tc{none, none};
  int diff = 0;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    const float x = block[(int64_t)r * V + v], y = chain[(int64_t)r * V + v];
    const uint32_t d = __float_as_uint(x) ^ __float_as_uint(y);
    diff += ((d & 0xffu) != 0) + ((d & 0xff00u) != 0) + ((d & 0xff0000u) != 0) + ((d & 0xff000000u) != 0);
    top2_insert(tb, ArgMax{x, v});
    top2_insert(tc, ArgMax{y, v});
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tb = top2_merge(tb, shfl_top2(tb, o));
    tc = top2_merge(tc, shfl_top2(tc, o));
    diff += __shfl_xor_sync(0xffffffffu, diff, o);
  }
  __shared__ Top2 sb[8], sc[8];
  __shared__ int sd[8];
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    sb[w] = tb;
    sc[w] = tc;
    sd[w] = diff;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < (int)(blockDim.x >> 5); ++k) {
      tb = top2_merge(tb, sb[k]);
      tc = top2_merge(tc, sc[k]);
      diff += sd[k];
    }
    dflash_exactness_row o;
    o.differing_bytes = diff;
    o.block_top[0] = tb.a.i;
    o.block_top[1] = tb.b.i;
    o.chain_top[0] = tc.a.i;
    o.chain_top[1] = tc.b.i;
    o.block_val[0] = tb.a.v;
    o.block_val[1] = tb.b.v;
    o.chain_val[0] = tc.a.v;
    o.chain_val[1] = tc.b.v;
    out[r] = o;
  }
}

struct DevBuf {
  void* p = nullptr;
  size_t cap = 0;
  cudaError_t ensure(size_t bytes, cudaStream_t st) {
    if (bytes <= cap) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    if (p) {
      e = cudaStreamSynchronize(st);
      if (e == cudaSuccess) e = cudaFree(p);
      p = nullptr;
      cap = 0;
      if (e != cudaSuccess) return e;
    }
    e = cudaMalloc(&p, bytes);
    if (e == cudaSuccess) cap = bytes;
    return e;
  }
  template <typename T> T* as() const { return (T*)p; }
};

}  // namespace
}  // namespace dfl

using namespace dfl;

struct dflash_target {
  dflash_target_config cfg{};
  const float* E = nullptr;
  const float* U = nullptr;
  const float* nf = nullptr;
  struct Layer {
    const float *n1, *wo, *n2, *wd;
    float* wqkv;  // [3 nh d][H]: q | k | v rows, stacked at create
    float* wgu;   // [2 I][H]: gate | up rows
  };
  std::vector<Layer> layers;
  std::vector<double> inv_freq;
  int64_t cap = 0, len = 0;
  float* kv = nullptr;
  cudaStream_t st = nullptr;
  int32_t* d_err = nullptr;
  DevBuf x, y, qkv, Q, O, tmp, gu, a, part, tables;
};

namespace {

int tfail(int code, const char* msg) { return dflash__set_error(code, msg); }

int tcheck(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return DFLASH_OK;
  char buf[256];
  snprintf(buf, sizeof buf, "%s: %s", what, cudaGetErrorString(e));
  return tfail(DFLASH_ERR_CUDA, buf);
}

constexpr int kTargetMaxRows = 64;  // rows per internal chunk of a forward

}  // namespace

extern "C" {

DFLASH_API int dflash_target_create(const dflash_target_config* cfg, const dflash_target_weights* w, int64_t max_ctx,
                                    void* stream, dflash_target** out) {
  if (!cfg || !w || !out || !w->embed || !w->unembed || !w->final_norm || !w->layers)
    return tfail(DFLASH_ERR_INVALID_ARG, "dflash_target_create: null argument");
  const dflash_target_config& c = *cfg;
  if (c.hidden <= 0 || c.n_heads <= 0 || c.head_dim <= 0 || c.head_dim % 4 || c.head_dim > 128 || c.intermediate <= 0 || c.hidden % 4 || c.intermediate % 4 || c.vocab <= 0 ||
      c.n_layers <= 0 || c.n_layers > 64 || c.hidden > 4096 || c.n_heads * c.head_dim > 4096 || max_ctx <= 0)
    return tfail(DFLASH_ERR_SHAPE, "dflash_target_create: unsupported shape");
  if ((uintptr_t)w->unembed % 16) return tfail(DFLASH_ERR_INVALID_ARG, "dflash_target_create: unembed not 16-byte aligned");
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_target_layer& L = w->layers[l];
    if (!L.n1 || !L.wq || !L.wk || !L.wv || !L.wo || !L.n2 || !L.wg || !L.wu || !L.wd)
      return tfail(DFLASH_ERR_INVALID_ARG, "dflash_target_create: null layer weight");
    if (((uintptr_t)L.wo | (uintptr_t)L.wd) % 16)
      return tfail(DFLASH_ERR_INVALID_ARG, "dflash_target_create: wo or wd not 16-byte aligned");
  }
  dflash_target* t = new dflash_target();
  t->cfg = c;
  t->E = (const float*)w->embed;
  t->U = (const float*)w->unembed;
  t->nf = (const float*)w->final_norm;
  t->st = (cudaStream_t)stream;
  t->cap = max_ctx;
  const int H = c.hidden, qd = c.n_heads * c.head_dim, I = c.intermediate;
  for (int j = 0; j < c.head_dim / 2; ++j) t->inv_freq.push_back(std::pow((double)c.rope_theta, -2.0 * j / c.head_dim));
  cudaError_t e = cudaMalloc(&t->d_err, 16);
  if (e == cudaSuccess) e = cudaMemset(t->d_err, 0, 16);
  if (e == cudaSuccess) e = cudaMalloc(&t->kv, (size_t)2 * c.n_layers * c.n_heads * max_ctx * c.head_dim * 4);
  for (int l = 0; l < c.n_layers && e == cudaSuccess; ++l) {
    const dflash_target_layer& L = w->layers[l];
    dflash_target::Layer Lw{(const float*)L.n1, (const float*)L.wo, (const float*)L.n2, (const float*)L.wd, nullptr,
                            nullptr};
    const size_t qb = (size_t)qd * H * 4, gb = (size_t)I * H * 4;
    e = cudaMalloc(&Lw.wqkv, 3 * qb);
    if (e == cudaSuccess) e = cudaMemcpy(Lw.wqkv, L.wq, qb, cudaMemcpyDeviceToDevice);
    if (e == cudaSuccess) e = cudaMemcpy((char*)Lw.wqkv + qb, L.wk, qb, cudaMemcpyDeviceToDevice);
    if (e == cudaSuccess) e = cudaMemcpy((char*)Lw.wqkv + 2 * qb, L.wv, qb, cudaMemcpyDeviceToDevice);
    if (e == cudaSuccess) e = cudaMalloc(&Lw.wgu, 2 * gb);
    if (e == cudaSuccess) e = cudaMemcpy(Lw.wgu, L.wg, gb, cudaMemcpyDeviceToDevice);
    if (e == cudaSuccess) e = cudaMemcpy((char*)Lw.wgu + gb, L.wu, gb, cudaMemcpyDeviceToDevice);
    t->layers.push_back(Lw);
  }
  if (e != cudaSuccess) {
    const int rc = tcheck(e, "dflash_target_create");
    dflash_target_destroy(t);
    return rc;
  }
  *out = t;
  return DFLASH_OK;
}

DFLASH_API int dflash_target_destroy(dflash_target* t) {
  if (!t) return DFLASH_OK;
  cudaDeviceSynchronize();
  for (auto& L : t->layers) {
    cudaFree(L.wqkv);
    cudaFree(L.wgu);
  }
  for (DevBuf* b : {&t->x, &t->y, &t->qkv, &t->Q, &t->O, &t->tmp, &t->gu, &t->a, &t->part, &t->tables}) cudaFree(b->p);
  cudaFree(t->kv);
  cudaFree(t->d_err);
  delete t;
  return DFLASH_OK;
}

DFLASH_API int dflash_target_length(const dflash_target* t, int64_t* length) {
  if (!t || !length) return tfail(DFLASH_ERR_INVALID_ARG, "dflash_target_length: null argument");
  *length = t->len;
  return DFLASH_OK;
}

DFLASH_API int dflash_target_trim(dflash_target* t, int64_t length) {
  if (!t) return tfail(DFLASH_ERR_INVALID_ARG, "dflash_target_trim: null target");
  if (length < 0 || length > t->len) return tfail(DFLASH_ERR_STATE, "dflash_target_trim: length outside [0, cached]");
  t->len = length;  // rows past it are overwritten by the next forward
  return DFLASH_OK;
}

DFLASH_API int dflash_target_argmax(dflash_target* t, const float* logits, int32_t rows, int32_t* out) {
  if (!t || !logits || !out || rows <= 0) return tfail(DFLASH_ERR_INVALID_ARG, "dflash_target_argmax: bad argument");
  launch_k(k_row_argmax, rows, 128, 0, t->st, logits, t->cfg.vocab, out);
  return tcheck(cudaGetLastError(), "dflash_target_argmax");
}

DFLASH_API int dflash_target_forward(dflash_target* t, const int32_t* tokens, int32_t rows, int64_t start,
                                     float* logits, float* taps) {
  if (!t || !tokens || !logits || rows <= 0) return tfail(DFLASH_ERR_INVALID_ARG, "dflash_target_forward: bad argument");
  if (start != t->len) return tfail(DFLASH_ERR_CONTEXT_GAP, "dflash_target_forward: start is not the cached length");
  if (start + rows > t->cap) return tfail(DFLASH_ERR_CAPACITY, "dflash_target_forward: beyond max_ctx");
  const dflash_target_config& c = t->cfg;
  const int H = c.hidden, nh = c.n_heads, d = c.head_dim, qd = nh * d, I = c.intermediate, V = c.vocab;
  const int NT = 2 * c.n_layers + 1;
  cudaStream_t st = t->st;
  for (int r0 = 0; r0 < rows; r0 += kTargetMaxRows) {
    const int R = std::min(kTargetMaxRows, rows - r0);
    const int64_t F = start + r0;
    // per-call tables: the session view of the cache, attention items, RoPE rows
    std::vector<char> host;
    auto add = [&](const void* src, size_t n) {
      const size_t off = (host.size() + 15) & ~(size_t)15;
      host.resize(off + n);
      memcpy(host.data() + off, src, n);
      return off;
    };
    void* kvp = t->kv;
    const int64_t capv = t->cap, fr = F;
    const int32_t seq = 0, zero = 0;
    const CUtensorMap* nomap = nullptr;
    std::vector<AttnItem> items;
    const int64_t kend = F + R, chunk = 256;
    const int S = (int)cdivu(kend, chunk);
    for (int h = 0; h < nh; ++h)
      for (int s = 0; s < S; ++s) items.push_back(AttnItem{0, h, s * chunk, std::min<int64_t>(kend, (s + 1) * chunk)});
    std::vector<float2> rope((size_t)R * (d / 2));
    for (int r = 0; r < R; ++r)
      for (int j = 0; j < d / 2; ++j) {
        const double ang = (double)(F + r) * t->inv_freq[j];
        rope[(size_t)r * (d / 2) + j] = make_float2((float)std::cos(ang), (float)std::sin(ang));
      }
    const size_t o_kv = add(&kvp, sizeof kvp), o_cap = add(&capv, 8), o_fr = add(&fr, 8), o_seq = add(&seq, 4),
                 o_map = add(&nomap, sizeof nomap), o_items = add(items.data(), items.size() * sizeof(AttnItem)),
                 o_first = add(&zero, 4), o_cnt = add(&S, 4), o_rope = add(rope.data(), rope.size() * sizeof(float2));
    int rc = tcheck(t->tables.ensure(host.size() + 16, st), "target tables");
    if (rc == DFLASH_OK && host.size() <= (size_t)kTableParamMax) {
      if (launch_table_write(t->tables.p, host.data(), host.size(), st)) rc = tfail(DFLASH_ERR_CUDA, "table write");
    } else if (rc == DFLASH_OK) {
      rc = tcheck(cudaMemcpyAsync(t->tables.p, host.data(), host.size(), cudaMemcpyHostToDevice, st), "tables");
      if (rc == DFLASH_OK) rc = tcheck(cudaStreamSynchronize(st), "tables");  // host block is a local
    }
    if (rc != DFLASH_OK) return rc;
    char* tb = t->tables.as<char>();
    SessTables tabs{(void* const*)(tb + o_kv), (const int64_t*)(tb + o_cap), (const int64_t*)(tb + o_fr),
                    (const int32_t*)(tb + o_seq), (const CUtensorMap* const*)(tb + o_map), nullptr};
    // buffers
    const size_t f4 = 4;
    cudaError_t e = t->x.ensure((size_t)R * H * f4, st);
    if (e == cudaSuccess) e = t->y.ensure((size_t)R * H * f4, st);
    if (e == cudaSuccess) e = t->qkv.ensure((size_t)R * 3 * qd * f4, st);
    if (e == cudaSuccess) e = t->Q.ensure((size_t)R * qd * f4, st);
    if (e == cudaSuccess) e = t->O.ensure((size_t)R * qd * f4, st);
    if (e == cudaSuccess) e = t->tmp.ensure((size_t)R * std::max(H, V) * f4, st);
    if (e == cudaSuccess) e = t->gu.ensure((size_t)R * 2 * I * f4, st);
    if (e == cudaSuccess) e = t->a.ensure((size_t)R * I * f4, st);
    if (e == cudaSuccess) e = t->part.ensure(items.size() * (size_t)R * (d + 4) * f4, st);
    if ((rc = tcheck(e, "target buffers")) != DFLASH_OK) return rc;
    float* X = t->x.as<float>();
    float* Y = t->y.as<float>();
    float* tp = taps ? taps + (size_t)r0 * NT * H : nullptr;
    const int64_t tap_ld = (int64_t)NT * H * 4;
    auto tap = [&](int k) {
      if (tp) launch_copy_rows(tp + (size_t)k * H, tap_ld, X, (int64_t)H * 4, (int64_t)H * 4, R, st);
    };
    launch_k(k_gather_rows, R, 128, 0, st, t->E, tokens + r0, V, H, X, t->d_err);
    tap(0);
    AttnParams ap{nh, nh, d, R, 0, 1, c.n_layers, 0, 1.f / std::sqrt((float)d), 1, nullptr, nullptr};
    for (int l = 0; l < c.n_layers; ++l) {
      const dflash_target::Layer& L = t->layers[l];
      launch_rmsnorm(DT::F32, true, X, R, nullptr, H, L.n1, Y, H, R, H, R, 0, 0, c.rms_eps, st);
      launch_gemm_rows(Y, H, L.wqkv, H, t->qkv.as<float>(), 3 * qd, R, 3 * qd, H, st);
      launch_k(k_target_qkv, dim3(R, nh), 64, 0, st, (const float*)t->qkv.as<float>(),
               (const float2*)(tb + o_rope), nh, d, F, t->cap, l, t->Q.as<float>(), t->kv);
      ap.layer = l;
      launch_attention_simt(DT::F32, t->Q.p, (const AttnItem*)(tb + o_items), (int)items.size(), tabs, ap,
                            t->part.as<float>(), st);
      launch_attention_combine(DT::F32, t->part.as<float>(), (const int32_t*)(tb + o_first),
                               (const int32_t*)(tb + o_cnt), 1, ap, nullptr, t->O.p, st);
      launch_gemm_rows(t->O.as<float>(), qd, L.wo, qd, t->tmp.as<float>(), H, R, H, qd, st);
      launch_residual(DT::F32, X, t->tmp.as<float>(), H, R, H, st);
      tap(1 + 2 * l);
      launch_rmsnorm(DT::F32, true, X, R, nullptr, H, L.n2, Y, H, R, H, R, 0, 0, c.rms_eps, st);
      launch_gemm_rows(Y, H, L.wgu, H, t->gu.as<float>(), 2 * I, R, 2 * I, H, st);
      launch_swiglu(DT::F32, t->gu.as<float>(), 2 * I, R, I, I, t->a.p, st);
      launch_gemm_rows(t->a.as<float>(), I, L.wd, I, t->tmp.as<float>(), H, R, H, I, st);
      launch_residual(DT::F32, X, t->tmp.as<float>(), H, R, H, st);
      tap(2 + 2 * l);
    }
    launch_rmsnorm(DT::F32, true, X, R, nullptr, H, t->nf, Y, H, R, H, R, 0, 0, c.rms_eps, st);
    launch_gemm_rows(Y, H, t->U, H, logits + (size_t)r0 * V, V, R, V, H, st);
    if ((rc = tcheck(cudaGetLastError(), "target forward")) != DFLASH_OK) return rc;
    t->len = F + R;
  }
  return DFLASH_OK;
}

DFLASH_API int dflash_logits_compare(const float* block, const float* chain, int32_t rows, int32_t vocab,
                                     dflash_exactness_row* out, void* stream) {
  if (!block || !chain || !out || rows <= 0 || vocab <= 0)
    return tfail(DFLASH_ERR_INVALID_ARG, "dflash_logits_compare: bad argument");
  launch_k(k_logits_compare, rows, 256, 0, (cudaStream_t)stream, block, chain, (int)vocab, out);
  return tcheck(cudaGetLastError(), "dflash_logits_compare");
}

DFLASH_API int dflash_exactness_summarize(const dflash_exactness_row* rows_host, int32_t rows,
                                          dflash_exactness_summary* out) {
  if (!rows_host || !out || rows <= 0) return tfail(DFLASH_ERR_INVALID_ARG, "dflash_exactness_summarize: bad argument");
  dflash_exactness_summary s{};
  s.rows = rows;
  for (int r = 0; r < rows; ++r) {
    s.differing_bytes += rows_host[r].differing_bytes;
    s.disagreements += rows_host[r].block_top[0] != rows_host[r].chain_top[0];
  }
  s.first_row_differing_bytes = rows_host[0].differing_bytes;
  s.allows = s.first_row_differing_bytes == 0;
  *out = s;
  return DFLASH_OK;
}

DFLASH_API int dflash_target_exactness_probe(dflash_target* t, const int32_t* tokens, int32_t rows, int64_t start,
                                             float* block_logits, float* chain_logits,
                                             dflash_exactness_row* out_rows, dflash_exactness_summary* summary) {
  if (!t || !tokens || !block_logits || !chain_logits || !out_rows || rows <= 0)
    return tfail(DFLASH_ERR_INVALID_ARG, "dflash_target_exactness_probe: bad argument");
  if (start != t->len) return tfail(DFLASH_ERR_CONTEXT_GAP, "dflash_target_exactness_probe: start is not the cached length");
  const int64_t V = t->cfg.vocab;
  int rc = dflash_target_forward(t, tokens, rows, start, block_logits, nullptr);
  if (rc == DFLASH_OK) t->len = start;
  for (int i = 0; i < rows && rc == DFLASH_OK; ++i)
    rc = dflash_target_forward(t, tokens + i, 1, start + i, chain_logits + i * V, nullptr);
  t->len = std::min(t->len, start);
  if (rc != DFLASH_OK) return rc;
  if ((rc = dflash_logits_compare(block_logits, chain_logits, rows, (int32_t)V, out_rows, t->st)) != DFLASH_OK) return rc;
  if (!summary) return DFLASH_OK;
  std::vector<dflash_exactness_row> h(rows);
  rc = tcheck(cudaMemcpyAsync(h.data(), out_rows, rows * sizeof(dflash_exactness_row), cudaMemcpyDeviceToHost, t->st),
              "exactness rows");
  if (rc == DFLASH_OK) rc = tcheck(cudaStreamSynchronize(t->st), "exactness rows");
  if (rc != DFLASH_OK) return rc;
  return dflash_exactness_summarize(h.data(), rows, summary);
}

DFLASH_API int dflash_target_device_status(dflash_target* t) {
  if (!t) return tfail(DFLASH_ERR_INVALID_ARG, "dflash_target_device_status: null target");
  int rc = tcheck(cudaStreamSynchronize(t->st), "target status");
  if (rc != DFLASH_OK) return rc;
  int32_t e = 0;
  if ((rc = tcheck(cudaMemcpy(&e, t->d_err, 4, cudaMemcpyDeviceToHost), "target status")) != DFLASH_OK) return rc;
  if (e) return tfail(DFLASH_ERR_DEVICE, "target: a token id outside [0, vocab)");
  return DFLASH_OK;
}

}  // extern "C"
