// Block attention on tensor cores for bf16 drafts: the n+1 block rows x the
// group's query heads of one KV head attend over a range of key positions
// (context followed by the block's own rows), with the window limit and the
// causal / bidirectional in-block mask computed on the fly (Laguna PR: the
// window is a per-query limit over [context | block]).
//
// One CTA per work item (session, KV head, key range), one warp per 16 query
// rows.  Key / value tiles of 64 positions are staged into shared memory with
// 16-byte cp.async copies (double buffered; each row's slot is the position
// modulo the cache ring, so ring wrap needs no special case), stored with an
// XOR swizzle so that ldmatrix reads are conflict-free.  S = Q K^T and
// O += P V run as mma.sync m16n8k16 bf16 with fp32 accumulators; the softmax
// is online in the exp2 domain.  The CTA writes (max, sum, O) partials that
// the split combine merges, exactly like the CUDA-core kernel.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace dfl {

namespace {

constexpr int KT = 64;      // key positions per tile
constexpr int STAGES = 3;  // K/V tiles in flight

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0: fill with zeros, read nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi), packed in pairs.
__device__ __forceinline__ void split_pack(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ bool visible(int64_t F, int i, int64_t r, int window, int causal) {
  if (window && (F + i) - r >= window) return false;
  if (causal && r >= F && (r - F) > i) return false;
  return true;
}

// Byte offset of 16-byte chunk c of row r in a swizzled tile of D-wide rows.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(256) k_attn_mma(const bf16* __restrict__ Q, const AttnItem* __restrict__ items,
                                                  SessTables tabs, AttnParams p, float* __restrict__ part) {
  constexpr int CH = D / 8;       // 16-byte chunks per row
  constexpr int NB = KT / 8;      // 8-key blocks per tile
  constexpr int DB = D / 8;       // 8-wide output blocks
  extern __shared__ __align__(128) uint8_t smem[];
  const int G = p.Hq / p.Hkv, R = p.nrows * G;
  const int Rp = (R + 15) & ~15;
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + Rp * D * 2;            // [STAGES][KT][D]
  uint8_t* sV = sK + STAGES * KT * D * 2;   // [STAGES][KT][D]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const AttnItem it = items[blockIdx.x];
  const int64_t F = tabs.frontier[it.sess], cap = tabs.cap[it.sess];
  const bf16* Kb = (const bf16*)tabs.kv[it.sess] + ((int64_t)(2 * p.layer) * p.Hkv + it.kvh) * cap * D;
  const bf16* Vb = (const bf16*)tabs.kv[it.sess] + ((int64_t)(2 * p.layer + 1) * p.Hkv + it.kvh) * cap * D;

  // ---- Q rows of this KV head into shared memory (rows past R are zero)
  for (int e = tid; e < Rp * CH; e += blockDim.x) {
    const int r = e / CH, c = e % CH;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < R) {
      const int i = r / G, g = r % G;
      v = *reinterpret_cast<const uint4*>(Q + (((int64_t)it.sess * p.nrows + i) * p.Hq + it.kvh * G + g) * D + c * 8);
    }
    *reinterpret_cast<uint4*>(sQ + swz<D>(r, c)) = v;
  }

  auto load_tile = [&](int buf, int64_t kt) {
    for (int e = tid; e < 2 * KT * CH; e += blockDim.x) {
      const int which = e / (KT * CH), r = (e / CH) % KT, c = e % CH;
      const int64_t pos = kt + r;
      const bool ok = pos < it.k1;
      const int64_t slot = ok ? pos % cap : 0;
      const bf16* src = (which ? Vb : Kb) + slot * D + c * 8;
      uint8_t* dst = (which ? sV : sK) + buf * KT * D * 2;
      cp_async16(smem_addr(dst + swz<D>(r, c)), src, ok);
    }
    cp_async_commit();
  };

  const int64_t ntiles = (it.k1 - it.k0 + KT - 1) / KT;
  // prologue: STAGES - 1 tiles in flight (an empty group keeps the count uniform)
  for (int t = 0; t < STAGES - 1; ++t) {
    if (t < ntiles) {
      load_tile(t, it.k0 + (int64_t)t * KT);
    } else {
      cp_async_commit();
    }
  }
  __syncthreads();

  const bool active = warp * 16 < R;
  // Q fragments: 16 rows x D of this warp
  uint32_t qf[D / 16][4];
  if (active) {
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int r = warp * 16 + (lane & 15), c = ks * 2 + (lane >> 4);
      ldsm_x4(smem_addr(sQ + swz<D>(r, c)), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }
  }
  float o[DB][4];
#pragma unroll
  for (int j = 0; j < DB; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const float sl2 = p.scale * 1.4426950408889634f;  // scores in the exp2 domain
  const int row0 = warp * 16 + (lane >> 2);          // this thread's rows: row0, row0 + 8
  const int i0 = row0 / G, i1 = (row0 + 8) / G;

  for (int64_t t = 0; t < ntiles; ++t) {
    const int buf = (int)(t % STAGES);
    const int64_t kt = it.k0 + t * KT;
    // tile t has landed once at most STAGES - 2 younger groups are pending
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    // refill the buffer freed by tile t - 1 with tile t + STAGES - 1
    if (t + STAGES - 1 < ntiles) {
      load_tile((int)((t + STAGES - 1) % STAGES), it.k0 + (t + STAGES - 1) * KT);
    } else {
      cp_async_commit();
    }
    if (active) {
      const uint8_t* tK = sK + buf * KT * D * 2;
      const uint8_t* tV = sV + buf * KT * D * 2;
      float s[NB][4];
#pragma unroll
      for (int j = 0; j < NB; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int jp = 0; jp < NB / 2; ++jp) {
          uint32_t b0, b1, b2, b3;
          const int r = jp * 16 + ((lane >> 4) << 3) + (lane & 7);
          const int c = ks * 2 + ((lane >> 3) & 1);
          ldsm_x4(smem_addr(tK + swz<D>(r, c)), b0, b1, b2, b3);
          mma_bf16(s[2 * jp], qf[ks], b0, b1);
          mma_bf16(s[2 * jp + 1], qf[ks], b2, b3);
        }
      }
      // mask, scale, row max
      float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < NB; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int hi = e >> 1;
          const int64_t key = kt + j * 8 + 2 * (lane & 3) + (e & 1);
          const int row = row0 + 8 * hi;
          const bool ok = row < R && key < it.k1 && visible(F, hi ? i1 : i0, key, p.window, p.causal);
          s[j][e] = ok ? s[j][e] * sl2 : -INFINITY;
          mt[hi] = fmaxf(mt[hi], s[j][e]);
        }
      }
      float corr[2], mnew[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 1));
        mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 2));
        mnew[h] = fmaxf(mrow[h], mt[h]);
        corr[h] = (mrow[h] == -INFINITY) ? 0.f : exp2f(mrow[h] - mnew[h]);
        if (mnew[h] == -INFINITY) corr[h] = 1.f;
      }
      float ls[2] = {0.f, 0.f};
#pragma unroll
      for (int j = 0; j < NB; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int hi = e >> 1;
          const float v = (s[j][e] == -INFINITY) ? 0.f : exp2f(s[j][e] - mnew[hi]);
          s[j][e] = v;
          ls[hi] += v;
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        ls[h] += __shfl_xor_sync(0xffffffffu, ls[h], 1);
        ls[h] += __shfl_xor_sync(0xffffffffu, ls[h], 2);
        lrow[h] = lrow[h] * corr[h] + ls[h];
        mrow[h] = mnew[h];
      }
#pragma unroll
      for (int j = 0; j < DB; ++j) {
        o[j][0] *= corr[0];
        o[j][1] *= corr[0];
        o[j][2] *= corr[1];
        o[j][3] *= corr[1];
      }
      // O += P V, with P split into two bf16 terms (hi + lo) so that the
      // probabilities keep ~16 significant bits: V is exact in bf16 and
      // both products accumulate in fp32.
#pragma unroll
      for (int ks = 0; ks < KT / 16; ++ks) {
        uint32_t ah[4], al[4];
        split_pack(s[2 * ks][0], s[2 * ks][1], ah[0], al[0]);
        split_pack(s[2 * ks][2], s[2 * ks][3], ah[1], al[1]);
        split_pack(s[2 * ks + 1][0], s[2 * ks + 1][1], ah[2], al[2]);
        split_pack(s[2 * ks + 1][2], s[2 * ks + 1][3], ah[3], al[3]);
#pragma unroll
        for (int jp = 0; jp < DB / 2; ++jp) {
          uint32_t b0, b1, b2, b3;
          const int r = ks * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
          const int c = jp * 2 + (lane >> 4);
          ldsm_x4_t(smem_addr(tV + swz<D>(r, c)), b0, b1, b2, b3);
          mma_bf16(o[2 * jp], ah, b0, b1);
          mma_bf16(o[2 * jp], al, b0, b1);
          mma_bf16(o[2 * jp + 1], ah, b2, b3);
          mma_bf16(o[2 * jp + 1], al, b2, b3);
        }
      }
    }
    __syncthreads();
  }

  // ---- partials: (max in natural-log units, sum, -, -, unnormalised O)
  cp_async_wait<0>();
  if (!active) return;
  float* out = part + (int64_t)blockIdx.x * R * (D + 4);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = row0 + 8 * h;
    if (row >= R) continue;
    float* pr = out + (int64_t)row * (D + 4);
    if ((lane & 3) == 0) {
      pr[0] = mrow[h] == -INFINITY ? -INFINITY : mrow[h] * 0.6931471805599453f;
      pr[1] = lrow[h];
    }
#pragma unroll
    for (int j = 0; j < DB; ++j) {
      const int col = j * 8 + 2 * (lane & 3);
      *reinterpret_cast<float2*>(pr + 4 + col) = make_float2(o[j][2 * h], o[j][2 * h + 1]);
    }
  }
}

}  // namespace

bool launch_attention_mma(const void* Q, const AttnItem* items, int n_items, SessTables tabs, AttnParams p,
                          float* part, cudaStream_t st) {
  const int R = p.nrows * (p.Hq / p.Hkv);
  if (R > 128 || (p.d != 64 && p.d != 128)) return false;
  if (n_items <= 0) return true;
  const int Rp = (R + 15) & ~15;
  const int threads = std::max(32 * (Rp / 16), 64);
  const size_t smem = (size_t)Rp * p.d * 2 + 2 * STAGES * KT * p.d * 2;
  if (p.d == 128) {
    cudaFuncSetAttribute(k_attn_mma<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_attn_mma<128><<<n_items, threads, smem, st>>>((const bf16*)Q, items, tabs, p, part);
  } else {
    cudaFuncSetAttribute(k_attn_mma<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_attn_mma<64><<<n_items, threads, smem, st>>>((const bf16*)Q, items, tabs, p, part);
  }
  return true;
}

}  // namespace dfl
