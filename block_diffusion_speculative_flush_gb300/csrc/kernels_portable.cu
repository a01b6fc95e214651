// Portable kernels of the DFlash draft round: every step that is not a
// weight-streaming matrix product.  Each is templated on the storage type
// (fp32 for the tiny config, bf16 otherwise) and accumulates in fp32.
//
// Steps and the passages they follow:
//   tap_norm       aux_hidden_norms: one RMSNorm per target tap (Laguna PR #1771)
//   rmsnorm        hidden_norm / input_layernorm / post-attention / final norms
//   embed          the block [anchor, mask x n] (dflash.go propose)
//   rope_table     rotary angles per row, computed in double
//   qkv_post       per-head q/k norm + RoPE, cache write of context and block
//                  K/V at their own slots (dflash.go: a context entry at slot S
//                  derives only from the features at S)
//   attention      block queries against [context | block] keys, GQA, window,
//                  causal or bidirectional block mask, split over keys
//   sample         one batched distribution over rows 1..n (dflash.go selectBlock)
//   verify_accept  accepted prefix + bonus token from the target logits and
//                  the proposal probabilities (DFlash2 commit note)
#include <float.h>
#include <math.h>

#include <cstring>
#include <type_traits>

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "launch.h"

namespace dfl {

namespace {

// 8 bf16 of a 16-byte word as floats, and back.
__device__ __forceinline__ void unpack8(const uint4& w, float* v) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float* v) {
  uint32_t u[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    u[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return make_uint4(u[0], u[1], u[2], u[3]);
}

// bf16 rows held in registers as 16-byte words (up to kNormVec per thread):
// one load of each input word, one store of each output word.
constexpr int kNormVec = 4;
__device__ __forceinline__ bool norm_vec_ok(const void* x, const void* g, const void* o, int H) {
  return H % 8 == 0 && H / 8 <= kNormVec * (int)blockDim.x && (((uintptr_t)x | (uintptr_t)g | (uintptr_t)o) & 15) == 0;
}
// The gain words of this thread (loaded ahead: the gain is a weight).
__device__ __forceinline__ void norm_gain_vec(const bf16* g, int H, uint4 (&gw)[kNormVec]) {
  const int nv = H / 8;
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) {
    const int c = threadIdx.x + i * blockDim.x;
    gw[i] = c < nv ? __ldg(reinterpret_cast<const uint4*>(g) + c) : make_uint4(0, 0, 0, 0);
  }
}
__device__ __forceinline__ void norm_row_vec(const bf16* x, const uint4 (&gw)[kNormVec], bf16* o, int H, float eps,
                                             float* red) {
  const int nv = H / 8;
  uint4 w[kNormVec];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) {
    const int c = threadIdx.x + i * blockDim.x;
    w[i] = c < nv ? reinterpret_cast<const uint4*>(x)[c] : make_uint4(0, 0, 0, 0);
    float v[8];
    unpack8(w[i], v);
#pragma unroll
    for (int e = 0; e < 8; ++e) ss += v[e] * v[e];
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / (float)H + eps);
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) {
    const int c = threadIdx.x + i * blockDim.x;
    if (c >= nv) continue;
    float v[8], gv[8];
    unpack8(w[i], v);
    unpack8(gw[i], gv);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = v[e] * inv * gv[e];
    reinterpret_cast<uint4*>(o)[c] = pack8(v);
  }
}
__device__ __forceinline__ void norm_row_vec(const bf16* x, const bf16* g, bf16* o, int H, float eps, float* red) {
  uint4 gw[kNormVec];
  norm_gain_vec(g, H, gw);
  norm_row_vec(x, gw, o, H, eps, red);
}

// fp32 rows of up to 4096 into bf16 (the fc output's hidden_norm): 128
// threads, each holding its eight float4 words in registers; one load of each
// input word and of each gain word, one 8-byte store per output word.
constexpr int kNormF32Vec = 8;
__global__ void __launch_bounds__(128) k_rmsnorm_f32v(const float* __restrict__ in, int64_t ld_in,
                                                      const bf16* __restrict__ g, bf16* __restrict__ out,
                                                      int64_t ld_out, int H, float eps) {
  pdl_trigger();
  const int j = blockIdx.x, nv = H / 4;
  uint2 gw[kNormF32Vec];  // the gain is a weight: read before the wait
#pragma unroll
  for (int i = 0; i < kNormF32Vec; ++i) {
    const int c = threadIdx.x + i * blockDim.x;
    gw[i] = c < nv ? __ldg(reinterpret_cast<const uint2*>(g) + c) : make_uint2(0u, 0u);
  }
  pdl_wait();
  __shared__ float red[32];
  const float4* x = after_wait(reinterpret_cast<const float4*>(in + (int64_t)j * ld_in));
  float4 w[kNormF32Vec];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kNormF32Vec; ++i) {
    const int c = threadIdx.x + i * blockDim.x;
    w[i] = c < nv ? x[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    ss += w[i].x * w[i].x;
    ss += w[i].y * w[i].y;
    ss += w[i].z * w[i].z;
    ss += w[i].w * w[i].w;
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / (float)H + eps);
  bf16* o = out + (int64_t)j * ld_out;
#pragma unroll
  for (int i = 0; i < kNormF32Vec; ++i) {
    const int c = threadIdx.x + i * blockDim.x;
    if (c >= nv) continue;
    const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[i].x));
    const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[i].y));
    const __nv_bfloat162 a = __floats2bfloat162_rn(w[i].x * inv * g01.x, w[i].y * inv * g01.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(w[i].z * inv * g23.x, w[i].w * inv * g23.y);
    uint2 raw;
    raw.x = *reinterpret_cast<const uint32_t*>(&a);
    raw.y = *reinterpret_cast<const uint32_t*>(&b);
    reinterpret_cast<uint2*>(o)[c] = raw;
  }
}

template <typename T>
__global__ void k_tap_norm(const T* const* __restrict__ src, const T* __restrict__ aux, T* __restrict__ u,
                           int K, int Ht, float eps) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int r = blockIdx.x, k = blockIdx.y;
  const T* f = src[(size_t)r * K + k];  // tap k of row r
  if constexpr (std::is_same<T, bf16>::value) {
    T* o = u + (size_t)r * K * Ht + (size_t)k * Ht;
    if (norm_vec_ok(f, aux + (size_t)k * Ht, o, Ht)) {
      norm_row_vec(f, aux + (size_t)k * Ht, o, Ht, eps, red);
      return;
    }
  }
  float ss = 0.f;
  for (int j = threadIdx.x; j < Ht; j += blockDim.x) {
    const float x = to_f(f[j]);
    ss += x * x;
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / (float)Ht + eps);
  const T* g = aux + (size_t)k * Ht;
  T* o = u + (size_t)r * K * Ht + (size_t)k * Ht;
  for (int j = threadIdx.x; j < Ht; j += blockDim.x) o[j] = from_f<T>(to_f(f[j]) * inv * to_f(g[j]));
}

// One row of RMSNorm by the whole CTA; the row stays in registers between
// the sum of squares and the scaled write (up to 8 x blockDim.x elements).
template <typename TIn, typename T>
__device__ __forceinline__ void rmsnorm_row(const TIn* __restrict__ x, const T* __restrict__ g, T* __restrict__ o,
                                            int H, float eps, float* red) {
  if constexpr (std::is_same<TIn, bf16>::value && std::is_same<T, bf16>::value) {
    if (norm_vec_ok(x, g, o, H)) {
      norm_row_vec(x, g, o, H, eps, red);
      return;
    }
  }
  constexpr int MAXV = 8;
  float v[MAXV];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < MAXV; ++k) {
    const int t = threadIdx.x + k * blockDim.x;
    v[k] = t < H ? to_f(x[t]) : 0.f;
    ss += v[k] * v[k];
  }
  for (int t = threadIdx.x + MAXV * blockDim.x; t < H; t += blockDim.x) {  // rows wider than the registers
    const float y = to_f(x[t]);
    ss += y * y;
  }
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / (float)H + eps);
#pragma unroll
  for (int k = 0; k < MAXV; ++k) {
    const int t = threadIdx.x + k * blockDim.x;
    if (t < H) o[t] = from_f<T>(v[k] * inv * to_f(g[t]));
  }
  for (int t = threadIdx.x + MAXV * blockDim.x; t < H; t += blockDim.x) o[t] = from_f<T>(to_f(x[t]) * inv * to_f(g[t]));
}

// One CTA per output row.
template <typename TIn, typename T>
__global__ void __launch_bounds__(512) k_rmsnorm(const TIn* __restrict__ in0, int rows0, const TIn* __restrict__ in1,
                                                 int64_t ld_in, const T* __restrict__ g, T* __restrict__ out,
                                                 int64_t ld_out, int H, int a, int b, int c, float eps) {
  pdl_trigger();
  __shared__ float red[32];
  const int j = blockIdx.x;
  const int src = (j / a) * b + (j % a) + c;
  const TIn* x = src < rows0 ? in0 + (int64_t)src * ld_in : in1 + (int64_t)(src - rows0) * ld_in;
  T* o = out + (int64_t)j * ld_out;
  if constexpr (std::is_same<TIn, bf16>::value && std::is_same<T, bf16>::value) {
    if (norm_vec_ok(x, g, o, H)) {
      // the gain is a weight: its words are read before the wait, the row after
      uint4 gw[kNormVec];
      norm_gain_vec(g, H, gw);
      pdl_wait();
      norm_row_vec(after_wait(x), gw, o, H, eps, red);
      return;
    }
  }
  pdl_wait();
  rmsnorm_row(after_wait(x), g, o, H, eps, red);
}

// Every layer's input norm of the same rows at once (a context-only
// forward): CTA (j, l) writes row j of out + l * out_layer with the gain of
// layer l, by the arithmetic of k_rmsnorm.
template <typename T>
__global__ void __launch_bounds__(512) k_rmsnorm_layers(const T* __restrict__ in, int64_t ld_in,
                                                        const T* const* __restrict__ gains, T* __restrict__ out,
                                                        int64_t ld_out, int64_t out_layer, int H, float eps) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int j = blockIdx.x, l = blockIdx.y;
  rmsnorm_row(in + (int64_t)j * ld_in, gains[l], out + l * out_layer + (int64_t)j * ld_out, H, eps, red);
}

// Block rows [anchor, mask x n]: rows of E copied 16 bytes at a time.
template <typename T>
__global__ void k_embed(const T* __restrict__ E, const int32_t* __restrict__ current,
                        const int32_t* __restrict__ sess_map, int mask_token, int V, int nrows, int H,
                        T* __restrict__ h, int32_t* __restrict__ err) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const int b = r / nrows, i = r % nrows;
  int tok = i == 0 ? current[sess_map ? sess_map[b] : b] : mask_token;
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) atomicOr(err, 1);
    tok = 0;
  }
  const uint4* e = reinterpret_cast<const uint4*>(E + (int64_t)tok * H);
  uint4* o = reinterpret_cast<uint4*>(h + (int64_t)r * H);
  const int nv = (int)(H * sizeof(T) / 16);
  for (int t = threadIdx.x; t < nv; t += blockDim.x) o[t] = e[t];
}

// cos / sin of pos * theta^(-2j/d), the angle formed and reduced in double so
// that large positions keep full fp32 accuracy; row m of the table is position
// meta[m].pos, or first + m without a row table.
__global__ void k_rope_table(const RowMeta* __restrict__ meta, int64_t first, int d, float theta,
                             float2* __restrict__ table) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x, j = threadIdx.x;
  if (j >= d / 2) return;
  const double inv = pow((double)theta, -2.0 * (double)j / (double)d);
  const double ang = (double)(meta ? meta[m].pos : first + m) * inv;
  double s, c;
  sincos(ang, &s, &c);
  table[(int64_t)m * (d / 2) + j] = make_float2((float)c, (float)s);
}

// One warp per head of one row.  Lane l holds elements l + 32u of the head,
// so RoPE partners (j, j + d/2) sit in the same lane.
template <typename T, int DU>  // DU = d / 32
__global__ void k_qkv_post(const float* __restrict__ qkv, int64_t ldq, const RowMeta* __restrict__ meta,
                           const float2* __restrict__ rope, const T* __restrict__ q_norm,
                           const T* __restrict__ k_norm, int Hq, int Hkv, int gated, float eps, SessTables tabs,
                           int layer, T* __restrict__ Q, float* __restrict__ G, int v_apart, int early) {
  constexpr int d = DU * 32;
  const int m = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int hh = blockIdx.y * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const bool is_q = hh < Hq, head = hh < Hq + Hkv;
  const int kh = hh - Hq;
  // the head-norm gain is a weight: read before the wait
  float gv[DU];
  const T* gn = is_q ? q_norm : k_norm;
#pragma unroll
  for (int u = 0; u < DU; ++u) gv[u] = head ? to_f(gn[lane + 32 * u]) : 0.f;
  // The row's table entry, its RoPE pair and the session's cache: written at
  // the start of the call.  With `early` the product before this kernel let
  // it start only once everything before that product had finished, so they
  // are read before the wait.
  RowMeta rm;
  float2 cs[DU / 2];
  int64_t cap = 1;
  T* base = nullptr;
  auto tables = [&] {
    rm = meta[m];
    if (!head) return;
    const float2* rt = rope + rm.pos * (d / 2);  // the table is indexed by position
#pragma unroll
    for (int u = 0; u < DU / 2; ++u) cs[u] = rt[lane + 32 * u];
    if (!is_q) {
      cap = tabs.cap[rm.sess];
      base = (T*)tabs.kv[rm.sess];
    }
  };
  if (early) tables();
  // The attention kernel that follows reads the session tables and the
  // cache rows older than this forward before its own wait: it may start
  // only once every kernel before this one has finished, so the trigger
  // comes after the wait.
  pdl_wait();
  pdl_trigger();
  const float* row = after_wait(qkv + (int64_t)m * ldq);  // the product just before
  // the head's values (and a K head's V values) in one round trip
  float y[DU], xv[DU];
#pragma unroll
  for (int u = 0; u < DU; ++u) {
    y[u] = head ? row[(int64_t)hh * d + lane + 32 * u] : 0.f;
    xv[u] = (head && !is_q && !v_apart) ? row[(int64_t)(Hq + Hkv + kh) * d + lane + 32 * u] : 0.f;
  }
  if (!early) tables();
  if (gated && rm.blk >= 0 && blockIdx.y == 0) {
    for (int hq = threadIdx.x; hq < Hq; hq += blockDim.x) {
      const float x = row[(Hq + 2 * Hkv) * d + hq];
      G[(int64_t)rm.blk * Hq + hq] = 1.f / (1.f + expf(-x));
    }
  }
  if (!head) return;
  if (is_q && rm.blk < 0) return;  // context rows need only K and V
  float ss = 0.f;
#pragma unroll
  for (int u = 0; u < DU; ++u) ss += y[u] * y[u];
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)d + eps);
#pragma unroll
  for (int u = 0; u < DU; ++u) y[u] = y[u] * inv * gv[u];
#pragma unroll
  for (int u = 0; u < DU / 2; ++u) {
    const float a = y[u], b = y[u + DU / 2];
    y[u] = a * cs[u].x - b * cs[u].y;
    y[u + DU / 2] = b * cs[u].x + a * cs[u].y;
  }
  if (is_q) {
    T* q = Q + ((int64_t)rm.blk * Hq + hh) * d;
#pragma unroll
    for (int u = 0; u < DU; ++u) q[lane + 32 * u] = from_f<T>(y[u]);
    return;
  }
  const int64_t slot = rm.pos % cap;
  T* kd = base + (((int64_t)(2 * layer) * Hkv + kh) * cap + slot) * d;
  T* vd = base + ((int64_t)(2 * layer + 1) * Hkv + kh) * cap * d + slot;  // V^T plane: [d][cap]
#pragma unroll
  for (int u = 0; u < DU; ++u) {
    kd[lane + 32 * u] = from_f<T>(y[u]);
    if (!v_apart) vd[(int64_t)(lane + 32 * u) * cap] = from_f<T>(xv[u]);
  }
}

// V of one KV head for 32 consecutive rows into the transposed V planes
// ([d][cap]): the rows go through shared memory, and lane r writes row r's
// entry of each plane row, so 32 consecutive slots of one session land as one
// contiguous run (k_qkv_post writes them one plane row per lane otherwise).
template <typename T, int D>
__global__ void __launch_bounds__(256) k_v_cache_t(const float* __restrict__ qkv, int64_t ldq,
                                                   const RowMeta* __restrict__ meta, int M, int Hq, int Hkv,
                                                   SessTables tabs, int layer) {
  pdl_wait();  // as in k_qkv_post: the attention that follows relies on it
  pdl_trigger();
  __shared__ float tile[32][D + 1];
  const int kh = blockIdx.y, m0 = blockIdx.x * 32;
  const int64_t col = (int64_t)(Hq + Hkv + kh) * D;
  for (int e = threadIdx.x; e < 32 * D; e += blockDim.x) {
    const int r = e / D, j = e % D;
    tile[r][j] = m0 + r < M ? qkv[(int64_t)(m0 + r) * ldq + col + j] : 0.f;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int m = m0 + lane;
  if (m >= M) return;
  const RowMeta rm = meta[m];
  const int64_t cap = tabs.cap[rm.sess];
  const int64_t slot = rm.pos % cap;
  T* vd = (T*)tabs.kv[rm.sess] + ((int64_t)(2 * layer + 1) * Hkv + kh) * cap * D + slot;
  for (int j = w; j < D; j += nw) vd[(int64_t)j * cap] = from_f<T>(tile[lane][j]);
}

// Context-only forward: K and V of 32 consecutive rows of one KV head into
// the cache.  Each warp takes four rows of K with the arithmetic of
// k_qkv_post (lane l holds elements l + 32u; the same sum order, norm, gain
// and rotation), so a context row's cache entry is the same bits whichever
// kernel wrote it; V goes through shared memory into the transposed planes as
// in k_v_cache_t.  One CTA replaces a grid of M x (Hq + Hkv) / 4 head warps.
template <typename T, int D>
__global__ void __launch_bounds__(256) k_kv_ctx(const float* __restrict__ qkv_all, int64_t ldq, int64_t kcol0,
                                                int64_t vcol0, int64_t layer_stride, const RowMeta* __restrict__ meta,
                                                int M, const float2* __restrict__ rope,
                                                const T* const* __restrict__ k_norms, int Hkv, float eps,
                                                SessTables tabs, int layer0) {
  pdl_trigger();
  pdl_wait();
  constexpr int DU = D / 32;
  __shared__ float tile[32][D + 1];
  const int kh = blockIdx.y, m0 = blockIdx.x * 32, layer = layer0 + (int)blockIdx.z;
  const float* qkv = qkv_all + (int64_t)blockIdx.z * layer_stride;
  const T* k_norm = k_norms[blockIdx.z];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int64_t vcol = vcol0 + (int64_t)kh * D;
  for (int e = threadIdx.x; e < 32 * D; e += blockDim.x) {
    const int r = e / D, j = e % D;
    tile[r][j] = m0 + r < M ? qkv[(int64_t)(m0 + r) * ldq + vcol + j] : 0.f;
  }
  // K: warp w takes rows w, w + 8, w + 16, w + 24; every load of its four
  // rows (meta, K, gains, then the rotation of each row's position) is issued
  // before the arithmetic that needs it
  constexpr int RPW = 4;
  float y[RPW][DU], gn[DU];
  int64_t pos[RPW];
  int sess[RPW];
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    const int r = w + k * 8;
    pos[k] = -1;
    sess[k] = 0;
    if (m0 + r < M) {
      const RowMeta rm = meta[m0 + r];
      pos[k] = rm.pos;
      sess[k] = rm.sess;
      const float* x = qkv + (int64_t)(m0 + r) * ldq + kcol0 + (int64_t)kh * D;
#pragma unroll
      for (int u = 0; u < DU; ++u) y[k][u] = x[lane + 32 * u];
    }
  }
#pragma unroll
  for (int u = 0; u < DU; ++u) gn[u] = to_f(k_norm[lane + 32 * u]);
  float2 cs[RPW][DU / 2];
#pragma unroll
  for (int k = 0; k < RPW; ++k)
    if (pos[k] >= 0) {
      const float2* rt = rope + pos[k] * (D / 2);
#pragma unroll
      for (int u = 0; u < DU / 2; ++u) cs[k][u] = rt[lane + 32 * u];
    }
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    if (pos[k] < 0) continue;  // the same for the whole warp
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < DU; ++u) ss += y[k][u] * y[k][u];
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / (float)D + eps);
#pragma unroll
    for (int u = 0; u < DU; ++u) y[k][u] = y[k][u] * inv * gn[u];
#pragma unroll
    for (int u = 0; u < DU / 2; ++u) {
      const float a = y[k][u], b = y[k][u + DU / 2];
      y[k][u] = a * cs[k][u].x - b * cs[k][u].y;
      y[k][u + DU / 2] = b * cs[k][u].x + a * cs[k][u].y;
    }
    const int64_t cap = tabs.cap[sess[k]];
    T* kd = (T*)tabs.kv[sess[k]] + (((int64_t)(2 * layer) * Hkv + kh) * cap + pos[k] % cap) * D;
#pragma unroll
    for (int u = 0; u < DU; ++u) kd[lane + 32 * u] = from_f<T>(y[k][u]);
  }
  __syncthreads();
  const int m = m0 + lane;
  if (m >= M) return;
  const RowMeta rm = meta[m];
  const int64_t cap = tabs.cap[rm.sess];
  T* vd = (T*)tabs.kv[rm.sess] + ((int64_t)(2 * layer + 1) * Hkv + kh) * cap * D + rm.pos % cap;
  for (int j = w; j < D; j += nw) vd[(int64_t)j * cap] = from_f<T>(tile[lane][j]);
}

// Key visibility for block row i (position F + i) and key position r.
__device__ __forceinline__ bool key_visible(int64_t F, int i, int64_t r, int window, int causal) {
  if (window && (F + i) - r >= window) return false;
  if (causal && r >= F && (r - F) > i) return false;
  return true;
}

// Split-key attention on CUDA cores: one CTA per work item (session, KV head,
// key range); all n+1 rows x group query heads of that KV head at once.
// Partial (max, sum, acc[d]) per query row; merged by k_attn_combine.
template <typename T>
__global__ void k_attn_simt(const T* __restrict__ Q, const AttnItem* __restrict__ items, SessTables tabs,
                            AttnParams p, float* __restrict__ part) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float sm[];
  const int d = p.d, G = p.Hq / p.Hkv, R = p.nrows * G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float* qs = sm;                      // [R][d]
  float* ks = qs + R * d;              // [32][d+1]
  float* vs = ks + 32 * (d + 1);       // [32][d]
  float* ms = vs + 32 * d;             // [R]
  float* ls = ms + R;                  // [R]
  float* acc = ls + R;                 // [R][d]
  const AttnItem it = items[blockIdx.x];
  const int64_t F = tabs.frontier[it.sess], cap = tabs.cap[it.sess];
  const T* Kb = (const T*)tabs.kv[it.sess] + ((int64_t)(2 * p.layer) * p.Hkv + it.kvh) * cap * d;
  const T* Vb = (const T*)tabs.kv[it.sess] + ((int64_t)(2 * p.layer + 1) * p.Hkv + it.kvh) * cap * d;
  for (int e = threadIdx.x; e < R * d; e += blockDim.x) {
    const int rr = e / d, t = e % d;
    const int i = rr / G, g = rr % G;
    qs[e] = to_f(Q[(((int64_t)it.sess * p.nrows + i) * p.Hq + it.kvh * G + g) * d + t]) * p.scale;
    acc[e] = 0.f;
  }
  for (int rr = threadIdx.x; rr < R; rr += blockDim.x) {
    ms[rr] = -INFINITY;
    ls[rr] = 0.f;
  }
  __syncthreads();
  for (int64_t kt = it.k0; kt < it.k1; kt += 32) {
    for (int e = threadIdx.x; e < 32 * d; e += blockDim.x) {
      const int j = e / d, t = e % d;
      const int64_t r = kt + j;
      float kv = 0.f, vv = 0.f;
      if (r < it.k1) {
        const int64_t slot = r % cap;
        kv = to_f(Kb[slot * d + t]);
        vv = to_f(Vb[(int64_t)t * cap + slot]);
      }
      ks[j * (d + 1) + t] = kv;
      vs[j * d + t] = vv;
    }
    __syncthreads();
    for (int rr = warp; rr < R; rr += nw) {
      const int i = rr / G;
      const int64_t r = kt + lane;
      const bool vis = r < it.k1 && key_visible(F, i, r, p.window, p.causal);
      float s = -INFINITY;
      if (vis) {
        float a = 0.f;
        for (int t = 0; t < d; ++t) a += qs[rr * d + t] * ks[lane * (d + 1) + t];
        s = a;
      }
      const float mt = warp_max(s);
      if (mt == -INFINITY) continue;
      const float m_old = ms[rr];
      const float m_new = fmaxf(m_old, mt);
      const float pj = vis ? expf(s - m_new) : 0.f;
      const float corr = m_old == -INFINITY ? 0.f : expf(m_old - m_new);
      const float psum = warp_sum(pj);
      for (int t = lane; t < d; t += 32) {
        float a = acc[rr * d + t] * corr;
        for (int j = 0; j < 32; ++j) a += __shfl_sync(0xffffffffu, pj, j) * vs[j * d + t];
        acc[rr * d + t] = a;
      }
      __syncwarp();
      if (lane == 0) {
        ms[rr] = m_new;
        ls[rr] = ls[rr] * corr + psum;
      }
      __syncwarp();
    }
    __syncthreads();
  }
  float* out = part + (int64_t)blockIdx.x * R * (d + 4);
  for (int e = threadIdx.x; e < R * (d + 4); e += blockDim.x) {
    const int rr = e / (d + 4), t = e % (d + 4);
    out[e] = t == 0 ? ms[rr] : (t == 1 ? ls[rr] : (t < 4 ? 0.f : acc[rr * d + t - 4]));
  }
}

// The merge below for d = 128 and at most NS splits: every lane loads every
// split's (m, l) and its four output columns of every split at once (one
// round trip to memory), then merges them in split order.  Splits past S
// weigh zero and add exact zeros, so NS does not change the result.
template <int NS, typename T>
__device__ __forceinline__ void combine_d128(const float* __restrict__ base, int64_t sstride, int S, int lane,
                                             float gate, T* __restrict__ out) {
  float2 ml[NS];
  float4 v[NS];
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    if (k < S) {
      ml[k] = *reinterpret_cast<const float2*>(base + k * sstride);
      v[k] = *reinterpret_cast<const float4*>(base + k * sstride + 4 + lane * 4);
    } else {
      ml[k] = make_float2(-INFINITY, 0.f);
      v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < NS; ++k) M = fmaxf(M, ml[k].x);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const float w = ml[k].x == -INFINITY ? 0.f : expf(ml[k].x - M);
    L += ml[k].y * w;
    acc.x += w * v[k].x;
    acc.y += w * v[k].y;
    acc.z += w * v[k].z;
    acc.w += w * v[k].w;
  }
  const float scale = gate / L;
  out += lane * 4;
  out[0] = from_f<T>(acc.x * scale);
  out[1] = from_f<T>(acc.y * scale);
  out[2] = from_f<T>(acc.z * scale);
  out[3] = from_f<T>(acc.w * scale);
}

// Merge of the key splits of one (block row, query head) per warp:
// M = max m_s, L = sum l_s e^(m_s - M), o = sum O_s e^(m_s - M) / L, then
// the per-head gate.  Partial rows are [m, l, -, -, O[d]] (16-byte aligned O).
// NSMAX (16 or 32): the most splits merged in one pass; the wider variant
// holds twice the registers, so it is launched only when a session needs it.
template <int NSMAX, typename T>
__global__ void __launch_bounds__(128) k_attn_combine(const float* __restrict__ part,
                                                      const int32_t* __restrict__ item_first,
                                                      const int32_t* __restrict__ item_count, AttnParams p, int total,
                                                      const float* __restrict__ Gt, T* __restrict__ O, int early) {
  pdl_trigger();
  // early: the attention kernel before this one let it start only after its
  // own wait, so the item tables and the gates (written earlier in the call)
  // are read before this kernel's wait, the partials after it
  if (!early) pdl_wait();
  __shared__ float wsm[4][64];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int gw = blockIdx.x * 4 + wl;  // (b, i, hq) flattened
  if (gw >= total) return;
  const int d = p.d, G = p.Hq / p.Hkv, R = p.nrows * G, PD = d + 4;
  const int hq = gw % p.Hq, bi = gw / p.Hq;
  const int b = bi / p.nrows, i = bi % p.nrows;
  const int kvh = hq / G, rr = i * G + hq % G;
  const int S = item_count[b];
  const float* base = part + ((int64_t)(item_first[b] + kvh * S) * R + rr) * PD;
  const int64_t sstride = (int64_t)R * PD;
  const float gate = Gt ? Gt[(int64_t)bi * p.Hq + hq] : 1.f;
  if (early) pdl_wait();
  base = after_wait(base);  // the partials: written by the kernel just before
  if (S <= NSMAX && d == 128) {
    T* out = O + ((int64_t)bi * p.Hq + hq) * d;
    if (NSMAX == 16 || S <= 16)
      combine_d128<16>(base, sstride, S, lane, gate, out);
    else
      combine_d128<NSMAX>(base, sstride, S, lane, gate, out);
    return;
  }
  // (m, l) of up to 32 splits in one pass, one split per lane
  float M = -INFINITY, mv = -INFINITY, lv = 0.f;
  if (lane < S) {
    const float2 ml = *reinterpret_cast<const float2*>(base + lane * sstride);
    mv = ml.x;
    lv = ml.y;
  }
  for (int s = lane + 32; s < S; s += 32) M = fmaxf(M, base[s * sstride]);
  M = warp_max(fmaxf(M, mv));
  float L = 0.f;
  if (lane < S) {
    const float w = mv == -INFINITY ? 0.f : expf(mv - M);
    L = lv * w;
    wsm[wl][lane] = w;
  }
  for (int s = lane + 32; s < S; s += 32) {
    const float m = base[s * sstride];
    const float w = m == -INFINITY ? 0.f : expf(m - M);
    L += base[s * sstride + 1] * w;
    if (s < 64) wsm[wl][s] = w;
  }
  L = warp_sum(L);
  __syncwarp();
  const float scale = gate / L;
  T* out = O + ((int64_t)bi * p.Hq + hq) * d;
  for (int t4 = lane * 4; t4 < d; t4 += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // sixteen splits' loads in flight at a time; the sum keeps split order
    for (int s0 = 0; s0 < S; s0 += 16) {
      float4 v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k)
        v[k] = s0 + k < S ? *reinterpret_cast<const float4*>(base + (s0 + k) * sstride + 4 + t4)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int s = s0 + k;
        if (s >= S) break;
        float w;
        if (s < 64) {
          w = wsm[wl][s];
        } else {
          const float m = base[s * sstride];
          w = m == -INFINITY ? 0.f : expf(m - M);
        }
        acc.x += w * v[k].x;
        acc.y += w * v[k].y;
        acc.z += w * v[k].z;
        acc.w += w * v[k].w;
      }
    }
    out[t4] = from_f<T>(acc.x * scale);
    out[t4 + 1] = from_f<T>(acc.y * scale);
    out[t4 + 2] = from_f<T>(acc.z * scale);
    out[t4 + 3] = from_f<T>(acc.w * scale);
  }
}

template <typename T>
__global__ void k_residual(T* __restrict__ h, const float* __restrict__ delta, int64_t ld, int H) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  for (int t = threadIdx.x; t < H; t += blockDim.x) {
    T* p = h + (int64_t)r * H + t;
    *p = from_f<T>(to_f(*p) + delta[(int64_t)r * ld + t]);
  }
}

template <typename T>
__global__ void k_swiglu(const float* __restrict__ gu, int64_t ld, int I, int up_off, T* __restrict__ a) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  for (int t = threadIdx.x; t < I; t += blockDim.x) {
    const float g = gu[(int64_t)r * ld + t], u = gu[(int64_t)r * ld + up_off + t];
    a[(int64_t)r * I + t] = from_f<T>(g / (1.f + expf(-g)) * u);
  }
}

// Y[M][N] = X[M][K] . W[N][K]^T on CUDA cores, fp32 accumulation with a
// fixed k order (independent of M).  64x64 tiles, 4x4 outputs per thread.
template <typename T>
__global__ void __launch_bounds__(256) k_gemm_simt(const T* __restrict__ X, int64_t ldx, const T* __restrict__ W,
                                                   int64_t ldw, float* __restrict__ Y, int64_t ldy, int M, int N,
                                                   int K) {
  pdl_trigger();
  pdl_wait();
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float c[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int e = threadIdx.x; e < 64 * 16; e += 256) {
      const int r = e / 16, kk = e % 16;
      const int gm = m0 + r, gn = n0 + r, gk = k0 + kk;
      As[kk][r] = (gm < M && gk < K) ? to_f(X[(int64_t)gm * ldx + gk]) : 0.f;
      Bs[kk][r] = (gn < N && gk < K) ? to_f(W[(int64_t)gn * ldw + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty + 16 * i];
        b[i] = Bs[kk][tx + 16 * i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) c[i][j] = fmaf(a[i], b[j], c[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gm = m0 + ty + 16 * i, gn = n0 + tx + 16 * j;
      if (gm < M && gn < N) Y[(int64_t)gm * ldy + gn] = c[i][j];
    }
}

template <typename T>
__global__ void k_kv_copy(T* __restrict__ cache, int64_t cap, int64_t first, T* __restrict__ flat, int n, int d,
                          int to_cache, int transposed) {
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.y, r = blockIdx.x;
  const int64_t slot = (first + r) % cap;
  T* plane = cache + (int64_t)h * cap * d;
  T* f = flat + ((int64_t)h * n + r) * d;
  for (int t = threadIdx.x; t < d; t += blockDim.x) {
    T* c = transposed ? plane + (int64_t)t * cap + slot : plane + slot * d + t;
    if (to_cache)
      *c = f[t];
    else
      f[t] = *c;
  }
}

// ---------------------------------------------------------------------------
// sampling
// ---------------------------------------------------------------------------
__device__ __forceinline__ float load_logit(const void* p, int in_bf16, int64_t idx) {
  return in_bf16 ? __bfloat162float(((const bf16*)p)[idx]) : ((const float*)p)[idx];
}

// One row of logits, read four entries at a time (one 16-byte fp32 or
// 8-byte bf16 load when the row is aligned and V % 4 == 0).
struct RowRef {
  const void* p;
  int bf;
  bool vec;
};
__device__ __forceinline__ RowRef row_ref(const SampleArgs& a, int row) {
  RowRef r{nullptr, 0, false};
  if (a.seq_logits) {
    r.p = a.seq_logits[row / a.rows_per_seq] + (int64_t)(row % a.rows_per_seq) * a.ld;
  } else {
    r.bf = a.in_bf16;
    r.p = r.bf ? (const void*)((const bf16*)a.logits + (int64_t)row * a.ld)
               : (const void*)((const float*)a.logits + (int64_t)row * a.ld);
  }
  r.vec = (a.V & 3) == 0 && ((uintptr_t)r.p & (r.bf ? 7u : 15u)) == 0;
  r.p = after_wait(r.p);  // callers resolve rows after their wait
  return r;
}
// Entries 4g..4g+3 scaled by invT (the same product as the draw's); entries
// at or past V read as NaN, which is never comparable.
__device__ __forceinline__ void load_quad(const RowRef& r, int g, int V, float invT, float x[4]) {
  const int v = 4 * g;
  if (r.vec && v < V) {
    if (r.bf) {
      const uint2 w = reinterpret_cast<const uint2*>(r.p)[g];
      x[0] = __uint_as_float(w.x << 16) * invT;
      x[1] = __uint_as_float(w.x & 0xffff0000u) * invT;
      x[2] = __uint_as_float(w.y << 16) * invT;
      x[3] = __uint_as_float(w.y & 0xffff0000u) * invT;
    } else {
      const float4 f = reinterpret_cast<const float4*>(r.p)[g];
      x[0] = f.x * invT;
      x[1] = f.y * invT;
      x[2] = f.z * invT;
      x[3] = f.w * invT;
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k)
    x[k] = v + k < V ? (r.bf ? __bfloat162float(((const bf16*)r.p)[v + k]) : ((const float*)r.p)[v + k]) * invT
                     : __int_as_float(0x7fc00000);
}

// Exclusive prefix sum over the CTA's threads in thread order; total gets the
// sum.  sm holds 33 entries; every thread of the CTA must call it.
template <typename T>
__device__ __forceinline__ T block_scan_excl(T x, T* sm, T& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  T incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm[w] = incl;
  __syncthreads();
  if (w == 0) {
    const T t = lane < nw ? sm[lane] : T(0);
    T ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += y;
    }
    if (lane < nw) sm[lane] = ti - t;
    if (lane == 31) sm[32] = ti;
  }
  __syncthreads();
  const T r = sm[w] + (incl - x);
  total = sm[32];
  __syncthreads();
  return r;
}

// part[row][chunk] = (max of l/T, sum exp(l/T - max), best score, best index)
// where the score is l/T + Gumbel (draft draw) or l/T (argmax / row stats).
// Logit v of sampled row `row`, from the session's own rows when given.
__device__ __forceinline__ float sample_logit(const SampleArgs& a, int row, int v) {
  if (a.seq_logits)
    return a.seq_logits[row / a.rows_per_seq][(int64_t)(row % a.rows_per_seq) * a.ld + v];
  return load_logit(a.logits, a.in_bf16, (int64_t)row * a.ld + v);
}

constexpr int kSampleSteps = 4;
constexpr int kSampleThreads = 256;

__global__ void __launch_bounds__(256, 4) k_sample_partials(SampleArgs a, int chunk, float4* __restrict__ part) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sm_m[32], sm_l[32], sm_s[32];
  __shared__ int32_t sm_i[32];
  const int row = blockIdx.x, c = blockIdx.y, nch = gridDim.y;
  const int v0 = c * chunk, v1 = min(a.V, v0 + chunk);
  const float invT = a.temperature > 0.f ? 1.f / a.temperature : 1.f;
  const int b = row / a.rows_per_seq;
  const uint32_t prow = (uint32_t)(row % a.rows_per_seq + a.row_offset);
  const uint32_t seq = a.seq_ids ? (uint32_t)a.seq_ids[b] : (uint32_t)b;
  const uint64_t cutv = a.cut ? a.cut[row] : 0ull;
  float m = -INFINITY, l = 0.f;
  ArgMax best{-INFINITY, INT32_MAX};
  const RowRef rr = row_ref(a, row);
  // four consecutive entries per thread and step: one Philox evaluation gives
  // their four random words (chunks start on multiples of 4); kSampleSteps
  // steps' loads are issued before any is used.
  // The common case (fp32 rows on 16-byte boundaries, no truncation) first:
  // the same steps and the same arithmetic in the same order, with the
  // per-entry range tests only on a quad that crosses the chunk's end.
  if (!cutv && rr.vec && !rr.bf && blockDim.x == kSampleThreads) {
    const float* rowp = static_cast<const float*>(rr.p);
    float bv = -INFINITY;  // this thread's best score; entries come in index order
    int bi = INT32_MAX;
    for (int base = v0 + 4 * threadIdx.x; base < v1; base += 4 * kSampleThreads * kSampleSteps) {
      float x[kSampleSteps][4];
#pragma unroll
      for (int it = 0; it < kSampleSteps; ++it) {
        const int v4 = base + it * 4 * kSampleThreads;
        if (v4 + 3 < v1) {
          const float4 f = *reinterpret_cast<const float4*>(rowp + v4);
          x[it][0] = f.x * invT;
          x[it][1] = f.y * invT;
          x[it][2] = f.z * invT;
          x[it][3] = f.w * invT;
        } else {
#pragma unroll
          for (int w = 0; w < 4; ++w) x[it][w] = v4 + w < v1 ? rowp[v4 + w] * invT : -INFINITY;
        }
      }
      float ms = -INFINITY;
#pragma unroll
      for (int it = 0; it < kSampleSteps; ++it)
#pragma unroll
        for (int w = 0; w < 4; ++w) ms = fmaxf(ms, x[it][w]);
      if (ms != -INFINITY) {
        float ls = 0.f;
#pragma unroll
        for (int it = 0; it < kSampleSteps; ++it)
#pragma unroll
          for (int w = 0; w < 4; ++w) ls += __expf(x[it][w] - ms);
        if (ms > m) {
          l = (m == -INFINITY ? 0.f : l * __expf(m - ms)) + ls;
          m = ms;
        } else {
          l += ls * __expf(ms - m);
        }
      }
#pragma unroll
      for (int it = 0; it < kSampleSteps; ++it) {
        const int v4 = base + it * 4 * kSampleThreads;
        uint4 r = make_uint4(0, 0, 0, 0);
        if (a.gumbel && v4 < v1) r = rand_block(a.seed, a.rnd, kStreamDraft, seq, prow, (uint32_t)v4 >> 2);
        const uint32_t wd[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          // an entry past the chunk is -inf and never beats a score
          const float sc = a.gumbel ? x[it][w] + gumbel_of(wd[w]) : x[it][w];
          if (sc > bv) {
            bv = sc;
            bi = v4 + w;
          }
        }
      }
    }
    best = ArgMax{bv, bi};
  } else
  for (int base = v0 + 4 * threadIdx.x; base < v1; base += 4 * blockDim.x * kSampleSteps) {
    float x[kSampleSteps][4];
#pragma unroll
    for (int it = 0; it < kSampleSteps; ++it) {
      const int v4 = base + it * 4 * blockDim.x;
      if (v4 < v1) {
        load_quad(rr, v4 >> 2, a.V, invT, x[it]);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) x[it][k] = 0.f;
      }
    }
    // entries outside the chunk or the truncated support become -inf: they
    // add nothing to the sum and never win the draw
#pragma unroll
    for (int it = 0; it < kSampleSteps; ++it) {
      const int v4 = base + it * 4 * blockDim.x;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int v = v4 + w;
        if (v >= v1 || (cutv && order_key(x[it][w], v) < cutv)) x[it][w] = -INFINITY;
      }
    }
    // the step's max, then one exponential per entry
    float ms = -INFINITY;
#pragma unroll
    for (int it = 0; it < kSampleSteps; ++it)
#pragma unroll
      for (int w = 0; w < 4; ++w) ms = fmaxf(ms, x[it][w]);
    if (ms != -INFINITY) {
      float ls = 0.f;
#pragma unroll
      for (int it = 0; it < kSampleSteps; ++it)
#pragma unroll
        for (int w = 0; w < 4; ++w) ls += __expf(x[it][w] - ms);
      if (ms > m) {
        l = (m == -INFINITY ? 0.f : l * __expf(m - ms)) + ls;
        m = ms;
      } else {
        l += ls * __expf(ms - m);
      }
    }
#pragma unroll
    for (int it = 0; it < kSampleSteps; ++it) {
      const int v4 = base + it * 4 * blockDim.x;
      if (v4 >= v1) break;
      uint4 r = make_uint4(0, 0, 0, 0);
      if (a.gumbel) r = rand_block(a.seed, a.rnd, kStreamDraft, seq, prow, (uint32_t)v4 >> 2);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int v = v4 + w;
        if (v >= v1) break;
        const float s = x[it][w];
        if (s == -INFINITY && cutv) continue;  // outside the truncated support
        float score = s;
        if (a.gumbel) score += gumbel_of(word_of(r, w));
        best = better(best, ArgMax{score, v});
      }
    }
  }
  // warp merge
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), l2 = __shfl_xor_sync(0xffffffffu, l, o);
    const float M = fmaxf(m, m2);
    l = (m == -INFINITY ? 0.f : l * __expf(m - M)) + (m2 == -INFINITY ? 0.f : l2 * __expf(m2 - M));
    m = M;
  }
  best = warp_argmax(best);
  if (lane == 0) {
    sm_m[w] = m;
    sm_l[w] = l;
    sm_s[w] = best.v;
    sm_i[w] = best.i;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int i = 0; i < nw; ++i) M = fmaxf(M, sm_m[i]);
    float L = 0.f;
    ArgMax bb{-INFINITY, INT32_MAX};
    for (int i = 0; i < nw; ++i) {
      if (sm_m[i] != -INFINITY) L += sm_l[i] * __expf(sm_m[i] - M);
      bb = better(bb, ArgMax{sm_s[i], sm_i[i]});
    }
    part[(int64_t)row * nch + c] = make_float4(M, L, bb.v, __int_as_float(bb.i));
  }
}

__global__ void k_sample_combine(SampleArgs a, int chunks, const float4* __restrict__ part, int32_t* __restrict__ tok,
                                 float* __restrict__ qtok, float* __restrict__ lse) {
  pdl_trigger();
  pdl_wait();
  // one warp per row, lane c over chunks c, c + 32, ...
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= a.rows) return;
  float M = -INFINITY;
  for (int c = lane; c < chunks; c += 32) M = fmaxf(M, part[(int64_t)row * chunks + c].x);
  M = warp_max(M);
  float L = 0.f;
  ArgMax bb{-INFINITY, INT32_MAX};
  for (int c = lane; c < chunks; c += 32) {
    const float4 pc = part[(int64_t)row * chunks + c];
    if (pc.x != -INFINITY) L += pc.y * expf(pc.x - M);
    bb = better(bb, ArgMax{pc.z, __float_as_int(pc.w)});
  }
  L = warp_sum(L);
  bb = warp_argmax(bb);
  if (lane != 0) return;
  // a row whose scores were all NaN has no argmax: record it and answer 0
  // rather than reading a logit at an undefined index
  if (bb.i < 0 || bb.i >= a.V) {
    if (a.err) atomicOr(a.err, 16);
    bb.i = 0;
  }
  const float ls = M + logf(L);
  int orow = row;
  if (a.out_map) orow = a.out_map[row / a.rows_per_seq] * a.rows_per_seq + row % a.rows_per_seq;
  if (tok) tok[orow] = bb.i;
  if (lse) lse[orow] = ls;
  if (a.sess_tok) a.sess_tok[row / a.rows_per_seq][row % a.rows_per_seq] = bb.i;
  if (a.sess_lse) a.sess_lse[row / a.rows_per_seq][row % a.rows_per_seq] = ls;
  if (qtok) {
    if (a.temperature > 0.f) {
      const float x = sample_logit(a, row, bb.i) / a.temperature;
      qtok[orow] = expf(x - ls);
    } else {
      qtok[orow] = 1.f;
    }
  }
}

// ---------------------------------------------------------------------------
// truncated distributions: the cut of each row
// ---------------------------------------------------------------------------
// The cut kernel runs a cluster of CTAs per row.  Rows up to
// kCutRegQuads * 4 * kCutThreads * kCutMaxCluster entries are read once into
// registers (kCutRegQuads quads per thread) and every pass runs on them; longer
// rows are streamed from memory in every pass by a cluster of kCutCluster CTAs.
constexpr int kCutThreads = 1024;
constexpr int kCutRegQuads = 5;
constexpr int kCutMaxCluster = 8;
constexpr int kCutStreamThreads = 512;
constexpr int kCutQuads = 4;    // quads in flight per thread in each streamed pass
constexpr int kCutCluster = 8;  // CTAs per row when streaming

// Histogram update of one entry's order word: digit (o >> shift) & 255 of
// the entries that match the prefix so far, equal digits of a warp
// aggregated into one atomic on the warp's private histogram.
__device__ __forceinline__ void hist_add(int (*hist)[256], int w, int lane, uint32_t o, uint32_t pmask,
                                         uint32_t prefix, int shift) {
  const bool act = o != 0u && (o & pmask) == prefix;
  const unsigned am = __ballot_sync(0xffffffffu, act);
  if (act) {
    const uint32_t dg = (o >> shift) & 255u;
    const unsigned peers = __match_any_sync(am, dg);
    if (lane == __ffs(peers) - 1) atomicAdd(&hist[w][dg], __popc(peers));
  }
}

__device__ __forceinline__ uint64_t key_of_order(uint32_t o, int v) {
  return ((uint64_t)o << 32) | (uint64_t)(0xffffffffu - (uint32_t)v);
}

// A cluster of CTAs per row, each over a contiguous slice of the row.  The
// k-th entry of the sampler's order (value descending, then id) is found by
// radix select over the 32-bit order words: four 8-bit digits, each CTA
// counting its slice in warp-private histograms, every CTA summing the
// cluster's counts through distributed shared memory (double-buffered by
// pass, one cluster barrier per pass) and taking the same digit.  The k
// candidates are gathered into the first CTA (ties at the k-th value by id,
// in id order across the slices), sorted by key (bitonic), and top-p (the
// mass strictly before an entry below top_p) and min-p (probability at least
// min_p times the largest) cut the sorted list.  The cut is the key of the
// last entry kept; rows of a session without truncation get 0, rows with no
// comparable entry ~0.  Every CTA of a cluster takes the same branches.
// RQ > 0: the slice is RQ quads per thread, read once into registers;
// RQ == 0: the slice is streamed from memory in every pass.
template <int THREADS, int RQ>
__global__ void __launch_bounds__(THREADS, 1) k_trunc_cut(SampleArgs a, const Trunc* __restrict__ tr,
                                                         uint64_t* __restrict__ cut,
                                                         uint64_t* const* __restrict__ sess_cut) {
  constexpr int NW = THREADS / 32;
  constexpr int PER = kTruncMaxK / THREADS;  // sorted candidates per thread in the top-p scan
  pdl_trigger();
  pdl_wait();
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  __shared__ int hist[NW][256];
  __shared__ int tot[2][256];  // this CTA's digit counts, double-buffered by pass
  __shared__ uint64_t cand[kTruncMaxK];
  __shared__ int scan_i[33];
  __shared__ float scan_f[33];
  __shared__ int s_bin, s_above, s_eq, s_ncand, s_eqbase;
  const int C = (int)cl.num_blocks(), cr = (int)cl.block_rank();
  const int row = blockIdx.x / C, b = row / a.rows_per_seq;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const Trunc t = tr[b];
  const int V = a.V;
  if (t.top_k <= 0) {
    if (cr == 0 && tid == 0) {
      cut[row] = 0ull;
      if (sess_cut) sess_cut[b][row % a.rows_per_seq] = 0ull;
    }
    return;
  }
  if (tid == 0) s_ncand = 0;
  const float invT = a.temperature > 0.f ? 1.f / a.temperature : 1.f;
  const RowRef rr = row_ref(a, row);
  const int G = (V + 3) >> 2;
  int glo, ghi;
  if constexpr (RQ > 0) {
    glo = cr * THREADS * RQ;
    ghi = min(G, glo + THREADS * RQ);
  } else {
    glo = (int)((int64_t)G * cr / C);
    ghi = (int)((int64_t)G * (cr + 1) / C);
  }
  uint32_t ro[RQ > 0 ? RQ : 1][4];
  if constexpr (RQ > 0) {
#pragma unroll
    for (int u = 0; u < RQ; ++u) {
      const int g = glo + u * THREADS + tid;
      float x[4];
      if (g < ghi) {
        load_quad(rr, g, V, invT, x);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = __int_as_float(0x7fc00000);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) ro[u][k] = float_order(x[k]);
    }
  }
  // the order words of streamed quads g0 + u * THREADS + tid, u < kCutQuads
  auto stream_in = [&](int g0, uint32_t (&o)[kCutQuads][4]) {
    float x[kCutQuads][4];
#pragma unroll
    for (int u = 0; u < kCutQuads; ++u) {
      const int g = g0 + u * THREADS + tid;
      if (g < ghi) {
        load_quad(rr, g, V, invT, x[u]);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) x[u][k] = __int_as_float(0x7fc00000);
      }
    }
#pragma unroll
    for (int u = 0; u < kCutQuads; ++u)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[u][k] = float_order(x[u][k]);
  };

  uint32_t prefix = 0u, pmask = 0u;
  int need = min(t.top_k, kTruncMaxK), kc = 0;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass, buf = pass & 1;
    for (int i = tid; i < NW * 256; i += THREADS) (&hist[0][0])[i] = 0;
    __syncthreads();
    if constexpr (RQ > 0) {
#pragma unroll
      for (int u = 0; u < RQ; ++u)
#pragma unroll
        for (int k = 0; k < 4; ++k) hist_add(hist, w, lane, ro[u][k], pmask, prefix, shift);
    } else {
      for (int g0 = glo; g0 < ghi; g0 += THREADS * kCutQuads) {
        uint32_t o[kCutQuads][4];
        stream_in(g0, o);
#pragma unroll
        for (int u = 0; u < kCutQuads; ++u)
#pragma unroll
          for (int k = 0; k < 4; ++k) hist_add(hist, w, lane, o[u][k], pmask, prefix, shift);
      }
    }
    __syncthreads();
    if (tid < 256) {
      int c = 0;
      for (int q = 0; q < NW; ++q) c += hist[q][tid];
      tot[buf][tid] = c;
    }
    cl.sync();  // every CTA's counts of this pass are visible
    // the cluster's counts in descending digit order: thread j < 256 holds digit 255 - j
    int c = 0;
    if (tid < 256)
      for (int r = 0; r < C; ++r) c += cl.map_shared_rank(&tot[buf][0], r)[255 - tid];
    int total = 0;
    const int before = block_scan_excl(c, scan_i, total);
    if (pass == 0) {
      need = min(need, total);  // fewer comparable entries than k
      kc = need;
    }
    if (need == 0) break;       // the same in every CTA: nothing comparable in the row
    if (tid < 256 && c > 0 && before < need && need <= before + c) {
      s_bin = 255 - tid;
      s_above = before;
      s_eq = c;
    }
    __syncthreads();
    need -= s_above;
    prefix |= (uint32_t)s_bin << shift;
    pmask |= 255u << shift;
    if (pass == 3 && tid == 0) {
      // entries equal to the k-th value in the slices before this one
      int eb = 0;
      for (int r = 0; r < cr; ++r) eb += cl.map_shared_rank(&tot[buf][0], r)[s_bin];
      s_eqbase = eb;
    }
    __syncthreads();
  }
  cl.sync();  // no CTA reads another's counts after this
  if (kc == 0) {
    if (cr == 0 && tid == 0) {
      cut[row] = ~0ull;
      if (sess_cut) sess_cut[b][row % a.rows_per_seq] = ~0ull;
    }
    return;
  }
  {
    // gather into the first CTA: every entry above the k-th value, and the
    // first `need` entries (by id) equal to it.  Each group of THREADS quads
    // holds 4 * THREADS consecutive ids, thread by thread.
    const uint32_t tau = prefix;
    const bool all_eq = need == s_eq;
    int* ncand0 = cl.map_shared_rank(&s_ncand, 0);
    uint64_t* cand0 = cl.map_shared_rank(&cand[0], 0);
    int eq_base = s_eqbase;
    auto take_quad = [&](const uint32_t (&o)[4], int g) {
      int rank = 0;
      if (!all_eq) {
        int neq = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) neq += o[k] == tau;
        int tot_eq = 0;
        rank = eq_base + block_scan_excl(neq, scan_i, tot_eq);
        eq_base += tot_eq;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        bool take = o[k] > tau;
        if (o[k] == tau) take = all_eq || rank++ < need;
        if (take) {
          const int at = atomicAdd(ncand0, 1);
          if (at < kTruncMaxK) cand0[at] = key_of_order(o[k], 4 * g + k);
        }
      }
    };
    if constexpr (RQ > 0) {
#pragma unroll
      for (int u = 0; u < RQ; ++u) take_quad(ro[u], glo + u * THREADS + tid);
    } else {
      for (int g0 = glo; g0 < ghi; g0 += THREADS * kCutQuads) {
        uint32_t o[kCutQuads][4];
        stream_in(g0, o);
#pragma unroll
        for (int u = 0; u < kCutQuads; ++u) take_quad(o[u], g0 + u * THREADS + tid);
      }
    }
  }
  cl.sync();  // the candidates are in the first CTA
  if (cr != 0) return;
  int P = 1;
  while (P < kc) P <<= 1;
  for (int i = kc + tid; i < P; i += THREADS) cand[i] = 0ull;
  __syncthreads();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P; i += THREADS) {
        const int j = i ^ stride;
        if (j > i) {
          const uint64_t x = cand[i], y = cand[j];
          const bool desc = (i & size) == 0;
          if (desc ? x < y : x > y) {
            cand[i] = y;
            cand[j] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  int J = kc;
  if (t.top_p < 1.f || t.min_p > 0.f) {
    // thread i holds sorted entries PER*i .. PER*i + PER-1
    const float m = float_of_order((uint32_t)(cand[0] >> 32));
    float e[PER];
    float local = 0.f;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int j = PER * tid + k;
      e[k] = j < kc ? expf(float_of_order((uint32_t)(cand[j] >> 32)) - m) : 0.f;
      local += e[k];
    }
    float Z = 0.f;
    float before = block_scan_excl(local, scan_f, Z);
    int kept = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int j = PER * tid + k;
      bool keep = j < kc;
      if (t.top_p < 1.f) keep = keep && before < t.top_p * Z;
      if (t.min_p > 0.f) keep = keep && e[k] >= t.min_p;
      kept += keep;
      before += e[k];
    }
    int total = 0;
    (void)block_scan_excl(kept, scan_i, total);
    J = total;
  }
  if (tid == 0) {
    const uint64_t result = cand[max(J, 1) - 1];
    cut[row] = result;
    if (sess_cut) sess_cut[b][row % a.rows_per_seq] = result;
  }
}

// q of a DFlash2 proposal at position i: the candidate distribution's
// probability of v, 0 for an id outside the candidates.
__device__ __forceinline__ float candidate_q(const int32_t* ids, const float* probs, int kc, int i, int v) {
  for (int c = 0; c < kc; ++c)
    if (ids[i * kc + c] == v) return probs[i * kc + c];
  return 0.f;
}

// Acceptance scan of one session (T > 0): the first i in 1..n whose draft
// token fails u_i * q_i(d_i) < p_i(d_i), or 0 if all n pass.  A warp tests
// 32 positions at once and every lane returns the answer; a draft id outside
// [0, V) at or before the first failure sets bit 2 of the error word.
__device__ int verify_scan(const VerifyArgs& a, int b) {
  const int lane = threadIdx.x & 31;
  const int n = a.n, V = a.V;
  const int64_t tbase = (int64_t)b * (n + 1) * V;
  const uint32_t seq = a.seq_ids ? (uint32_t)a.seq_ids[b] : (uint32_t)b;
  const float invT = 1.f / a.temperature;
  const float Tq = a.dtemp[b];
  const float* dl = a.dlogits[b];
  const float* dlse = a.dlse[b];
  const int32_t* dtok = a.dtok[b];
  const uint64_t* dc = a.dcut ? a.dcut[b] : nullptr;
  const int32_t* cid = a.cand_ids ? a.cand_ids[b] : nullptr;
  const float* cpr = a.cand_probs ? a.cand_probs[b] : nullptr;
  for (int i0 = 1; i0 <= n; i0 += 32) {
    const int i = i0 + lane;
    bool fail = false, bad = false;
    if (i <= n) {
      int dtk = a.draft[b * n + i - 1];
      if (dtk < 0 || dtk >= V) {
        bad = true;
        dtk = 0;
      }
      const float st = load_logit(a.target, a.in_bf16, tbase + (int64_t)(i - 1) * V + dtk) * invT;
      float p = expf(st - a.lse_t[b * (n + 1) + i - 1]);
      if (a.cut_t && order_key(st, dtk) < a.cut_t[b * (n + 1) + i - 1]) p = 0.f;
      float q;
      if (cid && Tq > 0.f) {
        q = candidate_q(cid, cpr, a.ncand, i - 1, dtk);
      } else {
        const float dv = dl[(int64_t)(i - 1) * V + dtk];
        q = Tq > 0.f ? expf(dv / Tq - dlse[i - 1]) : (dtk == dtok[i - 1] ? 1.f : 0.f);
        if (Tq > 0.f && dc && order_key(dv * (1.f / Tq), dtk) < dc[i - 1]) q = 0.f;
      }
      const float r = uniform_open(rand_u32(a.seed, a.rnd, kStreamAccept, seq, (uint32_t)i, 0u));
      fail = !(r * q < p);
    }
    const unsigned fm = __ballot_sync(0xffffffffu, fail);
    const int first = fm ? i0 + __ffs(fm) - 1 : 0;
    const unsigned bm = __ballot_sync(0xffffffffu, bad && (first == 0 || i <= first));
    if (bm && lane == 0) atomicOr(a.err, 2);
    if (first) return first;
  }
  return 0;
}

// Bonus draw partials (T > 0), grid (session, vocabulary chunk): over the
// chunk of the target row after the accepted prefix, the residual mass
// sum max(0, p - q), the best log(max(0, p - q)) + Gumbel and the best
// log p + Gumbel.
__global__ void k_verify_bonus(VerifyArgs a, int chunk, VerifyPart* __restrict__ part) {
  pdl_trigger();
  pdl_wait();
  __shared__ int s_rej;
  __shared__ float sm_sum[32], sm_rs[32], sm_ps[32];
  __shared__ int32_t sm_ri[32], sm_pi[32];
  const int b = blockIdx.x, c = blockIdx.y, nch = gridDim.y;
  const int n = a.n, V = a.V;
  if (threadIdx.x < 32) {
    const int rj = verify_scan(a, b);
    if (threadIdx.x == 0) {
      s_rej = rj;
      if (c == 0) a.rej[b] = rj;
    }
  }
  __syncthreads();
  const int rej = s_rej;
  const int64_t tbase = (int64_t)b * (n + 1) * V;
  const uint32_t seq = a.seq_ids ? (uint32_t)a.seq_ids[b] : (uint32_t)b;
  const float invT = 1.f / a.temperature;
  const float Tq = a.dtemp[b];
  const float* dl = a.dlogits[b];
  const float* dlse = a.dlse[b];
  const int32_t* dtok = a.dtok[b];
  const int trow = rej ? rej - 1 : n;                 // target row of the bonus draw
  const uint32_t prow = rej ? (uint32_t)rej : (uint32_t)(n + 1);
  const float lse = a.lse_t[b * (n + 1) + trow];
  const uint64_t cutt = a.cut_t ? a.cut_t[b * (n + 1) + trow] : 0ull;
  const uint64_t* dc = a.dcut ? a.dcut[b] : nullptr;
  const int32_t* cid = (a.cand_ids && Tq > 0.f) ? a.cand_ids[b] : nullptr;
  const float* cpr = a.cand_probs ? a.cand_probs[b] : nullptr;
  const float invTq = Tq > 0.f ? 1.f / Tq : 1.f;
  const int v0 = c * chunk, v1 = min(V, v0 + chunk);
  float rsum = 0.f;
  ArgMax bres{-INFINITY, INT32_MAX}, bp{-INFINITY, INT32_MAX};
  for (int v4 = v0 + 4 * threadIdx.x; v4 < v1; v4 += 4 * blockDim.x) {
    const uint4 rw = rand_block(a.seed, a.rnd, kStreamBonus, seq, prow, (uint32_t)v4 >> 2);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int v = v4 + w;
      if (v >= v1) break;
      const float st = load_logit(a.target, a.in_bf16, tbase + (int64_t)trow * V + v) * invT;
      const float lp = st - lse;
      const bool kept = !cutt || order_key(st, v) >= cutt;
      const float g = gumbel_of(word_of(rw, w));
      if (kept) bp = better(bp, ArgMax{lp + g, v});
      if (rej) {
        const float p = kept ? expf(lp) : 0.f;
        float q;
        if (cid) {
          q = candidate_q(cid, cpr, a.ncand, rej - 1, v);
        } else {
          const float dv = dl[(int64_t)(rej - 1) * V + v];
          q = Tq > 0.f ? expf(dv / Tq - dlse[rej - 1]) : (v == dtok[rej - 1] ? 1.f : 0.f);
          if (Tq > 0.f && dc && order_key(dv * invTq, v) < dc[rej - 1]) q = 0.f;
        }
        const float res = fmaxf(p - q, 0.f);
        rsum += res;
        if (res > 0.f) bres = better(bres, ArgMax{logf(res) + g, v});
      }
    }
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  rsum = warp_sum(rsum);
  bres = warp_argmax(bres);
  bp = warp_argmax(bp);
  if (lane == 0) {
    sm_sum[w] = rsum;
    sm_rs[w] = bres.v;
    sm_ri[w] = bres.i;
    sm_ps[w] = bp.v;
    sm_pi[w] = bp.i;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    VerifyPart o{0.f, -INFINITY, INT32_MAX, -INFINITY, INT32_MAX};
    for (int i = 0; i < nw; ++i) {
      o.rsum += sm_sum[i];
      const ArgMax r = better(ArgMax{o.rv, o.ri}, ArgMax{sm_rs[i], sm_ri[i]});
      const ArgMax q = better(ArgMax{o.pv, o.pi}, ArgMax{sm_ps[i], sm_pi[i]});
      o.rv = r.v;
      o.ri = r.i;
      o.pv = q.v;
      o.pi = q.i;
    }
    part[(int64_t)b * nch + c] = o;
  }
}

// Accept length and bonus per session.  T == 0: accept while the target's
// argmax equals the draft token; bonus = argmax of row a.  T > 0: merge the
// bonus partials in chunk order.
__global__ void k_verify_finish(VerifyArgs a, int chunks, const VerifyPart* __restrict__ part) {
  pdl_trigger();
  pdl_wait();
  // one warp per session, lane c over chunks c, c + 32, ...
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (b >= a.B) return;
  const int n = a.n;
  int accn, bonus;
  if (a.temperature <= 0.f) {
    if (lane != 0) return;
    accn = 0;
    while (accn < n && a.amax_t[b * (n + 1) + accn] == a.draft[b * n + accn]) ++accn;
    bonus = a.amax_t[b * (n + 1) + accn];      // in range: the row statistics clamp it
  } else {
    const int rej = a.rej[b];
    float S = 0.f;
    ArgMax R{-INFINITY, INT32_MAX}, P{-INFINITY, INT32_MAX};
    for (int c = lane; c < chunks; c += 32) {
      const VerifyPart o = part[(int64_t)b * chunks + c];
      S += o.rsum;
      R = better(R, ArgMax{o.rv, o.ri});
      P = better(P, ArgMax{o.pv, o.pi});
    }
    S = warp_sum(S);
    R = warp_argmax(R);
    P = warp_argmax(P);
    if (lane != 0) return;
    accn = rej ? rej - 1 : n;
    bonus = (rej && S > 0.f) ? R.i : P.i;
    if (bonus < 0 || bonus >= a.V) {  // no comparable score (non-finite logits)
      atomicOr(a.err, 16);
      bonus = 0;
    }
  }
  a.accept[b] = accn;
  a.bonus[b] = bonus;
  if (a.accepted_total) *a.accepted_total[b] += accn;
}

inline unsigned cdiv(int64_t a, int64_t b) { return (unsigned)((a + b - 1) / b); }


// Row copy inside the launch chain (a stream copy would stop programmatic
// launch): grid (rows, pieces of 4096 bytes); 16-byte moves when both sides
// allow them.
__global__ void k_copy_rows(char* __restrict__ dst, int64_t dst_ld, const char* __restrict__ src, int64_t src_ld,
                            int64_t row_bytes, int vec) {
  pdl_trigger();
  pdl_wait();
  const int64_t r = blockIdx.x;
  const int64_t b0 = (int64_t)blockIdx.y * 4096, b1 = min(row_bytes, b0 + 4096);
  char* d = dst + r * dst_ld;
  const char* s = src + r * src_ld;
  if (vec) {
    for (int64_t b = b0 + (int64_t)threadIdx.x * 16; b < b1; b += (int64_t)blockDim.x * 16)
      *reinterpret_cast<uint4*>(d + b) = *reinterpret_cast<const uint4*>(s + b);
  } else {
    for (int64_t b = b0 + threadIdx.x; b < b1; b += blockDim.x) d[b] = s[b];
  }
}

// Copy blockIdx.y of the table; its rows split over blockIdx.x, 16 bytes a
// thread when every address and length allows it.
__global__ void k_copy_rows_batch(RowCopies t, int vec) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.y;
  const int64_t total = (int64_t)t.rows[i] * t.row_bytes;
  char* d = t.dst[i];
  const char* s = t.src[i];
  const int64_t ld = t.src_ld[i];
  if (vec) {
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 16; b < total;
         b += (int64_t)gridDim.x * blockDim.x * 16) {
      const int64_t r = b / t.row_bytes, c = b - r * t.row_bytes;
      *reinterpret_cast<uint4*>(d + b) = *reinterpret_cast<const uint4*>(s + r * ld + c);
    }
  } else {
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < total; b += (int64_t)gridDim.x * blockDim.x) {
      const int64_t r = b / t.row_bytes, c = b - r * t.row_bytes;
      d[b] = s[r * ld + c];
    }
  }
}

// Row r of tap k (rows src_ld bytes apart from src.p[k]) to dst + r * dst_ld
// + k * tap_bytes: K separate tap buffers into concatenated feature rows.
__global__ void k_copy_taps(char* __restrict__ dst, int64_t dst_ld, TapSrc src, int64_t src_ld, int64_t tap_bytes,
                            int vec) {
  pdl_trigger();
  pdl_wait();
  const int64_t r = blockIdx.x;
  const int k = blockIdx.y;
  char* d = dst + r * dst_ld + (int64_t)k * tap_bytes;
  const char* s = src.p[k] + r * src_ld;
  if (vec) {
    for (int64_t b = (int64_t)threadIdx.x * 16; b < tap_bytes; b += (int64_t)blockDim.x * 16)
      *reinterpret_cast<uint4*>(d + b) = *reinterpret_cast<const uint4*>(s + b);
  } else {
    for (int64_t b = threadIdx.x; b < tap_bytes; b += blockDim.x) d[b] = s[b];
  }
}

// Per-call tables as a kernel parameter, written to device memory once the
// previous kernel has completed (every kernel completes only after its own
// predecessor, so no earlier launch still reads the buffer).  Keeps the
// launch chain programmatic, where a host-to-device copy in the stream would
// wait for the previous kernel to drain and start the next one cold.
template <int N>
struct TableBytes {
  uint4 d[N / 16];
};
template <int N>
__global__ void k_table_write(uint4* __restrict__ dst, int n16, const __grid_constant__ TableBytes<N> src) {
  pdl_trigger();
  pdl_wait();
  for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = src.d[i];
}

// ---------------------------------------------------------------------------
// penalties over a token history
// ---------------------------------------------------------------------------
constexpr int kPenThreads = 1024;

// Sorts ids[0..n) in shared memory (n <= kMaxPenaltyHistory + a block of
// draft tokens, padded with INT32_MAX to a power of two), then calls
// f(id, count) once per distinct id, from the thread holding its first copy.
template <typename F>
__device__ __forceinline__ void for_each_distinct(int32_t* ids, int n, F f) {
  int N = 1;
  while (N < n) N <<= 1;
  for (int i = n + (int)threadIdx.x; i < N; i += blockDim.x) ids[i] = INT32_MAX;
  __syncthreads();
  for (int k = 2; k <= N; k <<= 1) {        // bitonic sort, ascending
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < N; i += blockDim.x) {
        const int l = i ^ j;
        if (l > i) {
          const int32_t a = ids[i], b = ids[l];
          if ((a > b) == ((i & k) == 0)) {
            ids[i] = b;
            ids[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int32_t v = ids[i];
    if (i > 0 && ids[i - 1] == v) continue;
    int c = 1;
    while (i + c < n && ids[i + c] == v) ++c;
    f(v, c);
  }
}

__device__ __forceinline__ float penalize(float x, int c, const Penalty& p) {
  x = x > 0.f ? x / p.repeat : x * p.repeat;
  return x - p.presence - p.frequency * (float)c;
}

__global__ void __launch_bounds__(kPenThreads) k_penalize_rows(const Penalty* __restrict__ pens,
                                                              float* const* __restrict__ rows, int rows_per_seq,
                                                              int64_t ld, int V) {
  __shared__ int32_t ids[kMaxPenaltyHistory];
  pdl_trigger();
  pdl_wait();
  const Penalty p = pens[blockIdx.x];
  if (p.n_hist <= 0) return;
  const int n = min(p.n_hist, kMaxPenaltyHistory);
  for (int i = threadIdx.x; i < n; i += blockDim.x) ids[i] = p.hist[i];
  __syncthreads();
  float* base = rows[blockIdx.x];
  for_each_distinct(ids, n, [&](int32_t v, int c) {
    if (v < 0 || v >= V) return;
    for (int r = 0; r < rows_per_seq; ++r) base[r * ld + v] = penalize(base[r * ld + v], c, p);
  });
}

template <typename T>
__global__ void __launch_bounds__(kPenThreads) k_penalize_target(const Penalty* __restrict__ pens,
                                                                const T* __restrict__ target, float* __restrict__ out,
                                                                const int32_t* __restrict__ draft, int n, int V) {
  // the history plus at most 511 draft tokens, padded to a power of two
  __shared__ int32_t ids[2 * kMaxPenaltyHistory];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x / (n + 1), r = blockIdx.x % (n + 1);
  const T* src = target + (int64_t)blockIdx.x * V;
  float* dst = out + (int64_t)blockIdx.x * V;
  for (int v = threadIdx.x; v < V; v += blockDim.x) dst[v] = to_f(src[v]);
  const Penalty p = pens[b];
  if (!(p.repeat != 1.f || p.presence != 0.f || p.frequency != 0.f)) return;  // no penalties: a plain copy
  const int nh = min(p.n_hist, kMaxPenaltyHistory);
  for (int i = threadIdx.x; i < nh; i += blockDim.x) ids[i] = p.hist[i];
  for (int i = threadIdx.x; i < r; i += blockDim.x) ids[nh + i] = draft[(int64_t)b * n + i];
  __syncthreads();  // the copied row is visible to every thread of the block too
  for_each_distinct(ids, nh + r, [&](int32_t v, int c) {
    if (v >= 0 && v < V) dst[v] = penalize(dst[v], c, p);
  });
}

}  // namespace

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
#define DFL_DISPATCH(dt, ...)                 \
  do {                                        \
    if ((dt) == DT::F32) {                    \
      using T = float;                        \
      __VA_ARGS__;                            \
    } else {                                  \
      using T = bf16;                         \
      __VA_ARGS__;                            \
    }                                         \
  } while (0)

void launch_tap_norm(DT dt, const void* const* src, int rows, const void* aux, void* u, int K, int Ht, float eps,
                     cudaStream_t st) {
  if (rows <= 0) return;
  DFL_DISPATCH(dt, launch_k(k_tap_norm<T>, dim3(rows, K), 256, 0, st, (const T* const*)src, (const T*)aux, (T*)u, K,
                                                                   Ht, eps));
}

void launch_rmsnorm(DT dt, bool in_f32, const void* in0, int rows0, const void* in1, int64_t ld_in, const void* g,
                    void* out, int64_t ld_out, int rows, int H, int a, int b, int c, float eps, cudaStream_t st) {
  if (rows <= 0) return;
  if (in_f32) {
    // fp32 rows into bf16 (one input, the identity row map): the vector
    // kernel whenever the width allows it; the choice depends on H only, so a
    // row's sum order never depends on how many rows share a call
    // (row map j -> (j / a) * b + j % a + c is the identity when a >= rows and c == 0)
    const bool vec = dt == DT::BF16 && H % 4 == 0 && H <= 4 * kNormF32Vec * 128 && rows0 >= rows && a >= rows &&
                     c == 0 && ld_in % 4 == 0 && ld_out % 4 == 0 && (((uintptr_t)in0 | (uintptr_t)g |
                     (uintptr_t)out) & 15) == 0;
    if (vec) {
      launch_k(k_rmsnorm_f32v, rows, 128, 0, st, (const float*)in0, ld_in, (const bf16*)g, (bf16*)out, ld_out, H, eps);
      return;
    }
    DFL_DISPATCH(dt, launch_k(k_rmsnorm<float, T>, rows, 512, 0, st, (const float*)in0, rows0, (const float*)in1, ld_in,
                                                                (const T*)g, (T*)out, ld_out, H, a, b, c, eps));
  } else {
    // bf16 rows of up to 4096 fit 128 threads of four 16-byte words each, so
    // sixteen rows per SM are in flight at once; the block shape depends on H
    // only, so a row's sum order never depends on how many rows share a call
    const int threads = (dt == DT::BF16 && H % 8 == 0 && H <= 8 * kNormVec * 128) ? 128 : 512;
    DFL_DISPATCH(dt, launch_k(k_rmsnorm<T, T>, rows, threads, 0, st, (const T*)in0, rows0, (const T*)in1, ld_in,
                                                            (const T*)g, (T*)out, ld_out, H, a, b, c, eps));
  }
}

void launch_embed(DT dt, const void* E, const int32_t* current, const int32_t* sess_map, int mask_token, int V,
                  int B, int nrows, int H, void* h, int32_t* err, cudaStream_t st) {
  if (B <= 0) return;
  DFL_DISPATCH(dt, launch_k(k_embed<T>, B * nrows, 128, 0, st, (const T*)E, current, sess_map, mask_token, V, nrows, H,
                                                          (T*)h, err));
}

void launch_rope_table(const RowMeta* meta, int64_t first, int M, int d, float theta, float2* table,
                       cudaStream_t st) {
  if (M <= 0) return;
  launch_k(k_rope_table, M, 64, 0, st, meta, first, d, theta, table);
}

void launch_kv_ctx(DT dt, const float* qkv, int64_t ldq, int64_t kcol0, int64_t vcol0, int64_t layer_stride,
                   const RowMeta* meta, int M, const float2* rope, const void* const* k_norms, int Hkv, int d,
                   float eps, SessTables tabs, int layer0, int layers, cudaStream_t st) {
  if (M <= 0 || layers <= 0) return;
  const dim3 grid(cdiv(M, 32), Hkv, layers);
  if (d == 64) {
    DFL_DISPATCH(dt, launch_k(k_kv_ctx<T, 64>, grid, 256, 0, st, qkv, ldq, kcol0, vcol0, layer_stride, meta, M, rope,
                              (const T* const*)k_norms, Hkv, eps, tabs, layer0));
  } else {
    DFL_DISPATCH(dt, launch_k(k_kv_ctx<T, 128>, grid, 256, 0, st, qkv, ldq, kcol0, vcol0, layer_stride, meta, M, rope,
                              (const T* const*)k_norms, Hkv, eps, tabs, layer0));
  }
}

void launch_rmsnorm_layers(DT dt, const void* in, int64_t ld_in, const void* const* gains, void* out, int64_t ld_out,
                           int64_t out_layer, int rows, int layers, int H, float eps, cudaStream_t st) {
  if (rows <= 0 || layers <= 0) return;
  // the block shape of launch_rmsnorm's storage-type rows, so the sums agree
  const int threads = (dt == DT::BF16 && H % 8 == 0 && H <= 8 * kNormVec * 128) ? 128 : 512;
  DFL_DISPATCH(dt, launch_k(k_rmsnorm_layers<T>, dim3(rows, layers), threads, 0, st, (const T*)in, ld_in,
                            (const T* const*)gains, (T*)out, ld_out, out_layer, H, eps));
}

int launch_qkv_post(DT dt, const float* qkv, int64_t ldq, const RowMeta* meta, int M, const float2* rope,
                    const void* q_norm, const void* k_norm, int Hq, int Hkv, int d, int gated, float eps,
                    SessTables tabs, int L, int layer, void* Q, float* G, cudaStream_t st, int early) {
  (void)L;
  if (M <= 0) return 0;
  const int heads = Hq + Hkv;
  dim3 grid(M, cdiv(heads, 4));
  // many rows: V goes to the cache in a second kernel, 32 rows at a time
  const int v_apart = M >= kVApartRows;
  if (d == 64) {
    DFL_DISPATCH(dt, launch_k(k_qkv_post<T, 2>, grid, 128, 0, st, qkv, ldq, meta, rope, (const T*)q_norm,
                                                              (const T*)k_norm, Hq, Hkv, gated, eps, tabs, layer,
                                                              (T*)Q, G, v_apart, early));
    if (v_apart)
      DFL_DISPATCH(dt, launch_k(k_v_cache_t<T, 64>, dim3(cdiv(M, 32), Hkv), 256, 0, st, qkv, ldq, meta, M, Hq, Hkv,
                                tabs, layer));
  } else {
    DFL_DISPATCH(dt, launch_k(k_qkv_post<T, 4>, grid, 128, 0, st, qkv, ldq, meta, rope, (const T*)q_norm,
                                                              (const T*)k_norm, Hq, Hkv, gated, eps, tabs, layer,
                                                              (T*)Q, G, v_apart, early));
    if (v_apart)
      DFL_DISPATCH(dt, launch_k(k_v_cache_t<T, 128>, dim3(cdiv(M, 32), Hkv), 256, 0, st, qkv, ldq, meta, M, Hq, Hkv,
                                tabs, layer));
  }
  return 1 + v_apart;
}

void launch_attention_simt(DT dt, const void* Q, const AttnItem* items, int n_items, SessTables tabs, AttnParams p,
                           float* part, cudaStream_t st) {
  if (n_items <= 0) return;
  const int R = p.nrows * (p.Hq / p.Hkv);
  const size_t smem = sizeof(float) * ((size_t)R * p.d * 2 + 32 * (p.d + 1) + 32 * p.d + 2 * R);
  DFL_DISPATCH(dt, {
    cudaFuncSetAttribute(k_attn_simt<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch_k(k_attn_simt<T>, n_items, 256, smem, st, (const T*)Q, items, tabs, p, part);
  });
}

void launch_attention_combine(DT dt, const float* part, const int32_t* item_first, const int32_t* item_count, int B,
                              AttnParams p, const float* G, void* O, cudaStream_t st, int max_splits, int early) {
  const int total = B * p.nrows * p.Hq;
  if (max_splits > 16 && max_splits <= 32) {
    DFL_DISPATCH(dt, launch_k(k_attn_combine<32, T>, cdiv(total, 4), 128, 0, st, part, item_first, item_count, p,
                              total, G, (T*)O, early));
  } else {
    DFL_DISPATCH(dt, launch_k(k_attn_combine<16, T>, cdiv(total, 4), 128, 0, st, part, item_first, item_count, p,
                              total, G, (T*)O, early));
  }
}

void launch_trunc_cut(const SampleArgs& a, const Trunc* tr, uint64_t* cut, uint64_t* const* sess_cut,
                      cudaStream_t st) {
  if (a.rows <= 0) return;
  const int64_t G = (a.V + 3) / 4, per_cta = (int64_t)kCutThreads * kCutRegQuads;
  const int creg = (int)((G + per_cta - 1) / per_cta);
  if (creg <= kCutMaxCluster) {
    // the row in registers: creg CTAs per row; one CTA per row cannot hold
    // it, so a refused cluster launch is an error here
    if (creg == 1) {
      launch_k(k_trunc_cut<kCutThreads, kCutRegQuads>, a.rows, kCutThreads, 0, st, a, tr, cut, sess_cut);
    } else {
      launch_kc(k_trunc_cut<kCutThreads, kCutRegQuads>, dim3(a.rows * creg), dim3(kCutThreads), 0, st, creg, a,
                tr, cut, sess_cut);
    }
    return;
  }
  // long rows streamed: a cluster of kCutCluster CTAs per row; one CTA per row
  // if that launch is refused
  if (launch_kc(k_trunc_cut<kCutStreamThreads, 0>, dim3(a.rows * kCutCluster), dim3(kCutStreamThreads), 0, st,
                kCutCluster, a, tr, cut, sess_cut) != cudaSuccess) {
    (void)cudaGetLastError();
    launch_k(k_trunc_cut<kCutStreamThreads, 0>, a.rows, kCutStreamThreads, 0, st, a, tr, cut, sess_cut);
  }
}

void launch_residual(DT dt, void* h, const float* delta, int64_t ld, int rows, int H, cudaStream_t st) {
  if (rows <= 0) return;
  DFL_DISPATCH(dt, launch_k(k_residual<T>, rows, 256, 0, st, (T*)h, delta, ld, H));
}

void launch_swiglu(DT dt, const float* gu, int64_t ld, int rows, int I, int up_off, void* a, cudaStream_t st) {
  if (rows <= 0) return;
  DFL_DISPATCH(dt, launch_k(k_swiglu<T>, rows, 256, 0, st, gu, ld, I, up_off, (T*)a));
}

void launch_gemm_simt(DT dt, const void* X, int64_t ldx, const void* W, int64_t ldw, float* Y, int64_t ldy, int M,
                      int N, int K, cudaStream_t st) {
  if (M <= 0 || N <= 0) return;
  dim3 grid(cdiv(N, 64), cdiv(M, 64));
  DFL_DISPATCH(dt, launch_k(k_gemm_simt<T>, grid, 256, 0, st, (const T*)X, ldx, (const T*)W, ldw, Y, ldy, M, N, K));
}

void launch_kv_copy(DT dt, void* cache, int64_t cap, int64_t first, void* flat, int n, int Hkv, int d, bool to_cache,
                    bool transposed, cudaStream_t st) {
  if (n <= 0) return;
  DFL_DISPATCH(dt, launch_k(k_kv_copy<T>, dim3(n, Hkv), 128, 0, st, (T*)cache, cap, first, (T*)flat, n, d,
                            (int)to_cache, (int)transposed));
}

void launch_sample_partials(const SampleArgs& a, int chunk, float4* part, cudaStream_t st) {
  if (a.rows <= 0) return;
  launch_k(k_sample_partials, dim3(a.rows, cdiv(a.V, chunk)), kSampleThreads, 0, st, a, chunk, part);
}

void launch_sample_combine(const SampleArgs& a, int chunks, const float4* part, int32_t* tok, float* qtok, float* lse,
                           cudaStream_t st) {
  if (a.rows <= 0) return;
  launch_k(k_sample_combine, cdiv(a.rows, 4), 128, 0, st, a, chunks, part, tok, qtok, lse);
}

void launch_verify_accept(const VerifyArgs& a, VerifyPart* part, cudaStream_t st) {
  if (a.B <= 0) return;
  const int chunk = kVerifyBonusChunk, chunks = verify_bonus_chunks(a.V);
  if (a.temperature > 0.f) launch_k(k_verify_bonus, dim3(a.B, chunks), 256, 0, st, a, chunk, part);
  launch_k(k_verify_finish, cdiv(a.B, 4), 128, 0, st, a, chunks, part);
}

void launch_penalize_rows(const Penalty* pen, float* const* rows, int rows_per_seq, int64_t ld, int V, int B,
                          cudaStream_t st) {
  if (B <= 0 || rows_per_seq <= 0) return;
  launch_k(k_penalize_rows, B, kPenThreads, 0, st, pen, rows, rows_per_seq, ld, V);
}

void launch_penalize_target(const Penalty* pen, const void* target, int in_bf16, float* out, const int32_t* draft,
                            int B, int n, int V, cudaStream_t st) {
  if (B <= 0) return;
  if (in_bf16)
    launch_k(k_penalize_target<bf16>, B * (n + 1), kPenThreads, 0, st, pen, (const bf16*)target, out, draft, n, V);
  else
    launch_k(k_penalize_target<float>, B * (n + 1), kPenThreads, 0, st, pen, (const float*)target, out, draft, n, V);
}

int launch_table_write(void* dst, const void* src, size_t bytes, cudaStream_t st) {
  const int n16 = (int)((bytes + 15) / 16);
  auto go = [&](auto tag) -> int {
    constexpr int N = decltype(tag)::value;
    TableBytes<N> t;
    memcpy(t.d, src, bytes);
    return launch_k(k_table_write<N>, 1, 256, 0, st, (uint4*)dst, n16, t) == cudaSuccess ? 0 : -1;
  };
  if (bytes <= 4096) return go(std::integral_constant<int, 4096>());
  if (bytes <= 16384) return go(std::integral_constant<int, 16384>());
  if (bytes <= kTableParamMax) return go(std::integral_constant<int, kTableParamMax>());
  return -1;
}

void launch_copy_rows(void* dst, int64_t dst_ld, const void* src, int64_t src_ld, int64_t row_bytes, int rows,
                      cudaStream_t st) {
  if (rows <= 0 || row_bytes <= 0) return;
  const int vec = ((uintptr_t)dst | (uintptr_t)src | (uintptr_t)dst_ld | (uintptr_t)src_ld | (uintptr_t)row_bytes) % 16 == 0;
  launch_k(k_copy_rows, dim3(rows, (unsigned)cdiv(row_bytes, 4096)), 256, 0, st, (char*)dst, dst_ld, (const char*)src,
           src_ld, row_bytes, vec);
}

void launch_copy_rows_batch(const RowCopies& t, cudaStream_t st) {
  if (t.n <= 0) return;
  int vec = t.row_bytes % 16 == 0;
  int64_t most = 0;
  for (int i = 0; i < t.n; ++i) {
    vec = vec && ((uintptr_t)t.dst[i] | (uintptr_t)t.src[i] | (uint64_t)t.src_ld[i]) % 16 == 0;
    most = std::max<int64_t>(most, (int64_t)t.rows[i] * t.row_bytes);
  }
  const unsigned bx = (unsigned)std::max<int64_t>(1, std::min<int64_t>(64, cdiv(most, 256 * 16 * 4)));
  launch_k(k_copy_rows_batch, dim3(bx, (unsigned)t.n), 256, 0, st, t, vec);
}

void launch_copy_taps(void* dst, int64_t dst_ld, const TapSrc& src, int K, int64_t src_ld, int64_t tap_bytes, int rows,
                      cudaStream_t st) {
  if (rows <= 0 || K <= 0) return;
  int vec = ((uintptr_t)dst | (uint64_t)dst_ld | (uint64_t)src_ld | (uint64_t)tap_bytes) % 16 == 0;
  for (int k = 0; k < K; ++k) vec = vec && (uintptr_t)src.p[k] % 16 == 0;
  launch_k(k_copy_taps, dim3(rows, K), 256, 0, st, (char*)dst, dst_ld, src, src_ld, tap_bytes, vec);
}

}  // namespace dfl
