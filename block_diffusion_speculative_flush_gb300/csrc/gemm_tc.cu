// Weight-streaming GEMM for the DFlash draft on sm_103a: tcgen05.mma with the
// accumulator in tensor memory, both operands brought into shared memory by
// TMA (cp.async.bulk.tensor) with 128-byte swizzle.
//
// Shape of the work.  The draft's products are skinny: a few to a few
// thousand activation rows (16 block rows per sequence, plus the pending
// context rows) against weight matrices of 10^7..10^9 elements.  The MMA's
// 128-row side therefore takes 128 weight rows (output features) and its N
// side takes the activation rows ("swap AB"):
//     D[feature][row] = W[feature][:] . X[row][:].
//
// Summation order.  K is cut into S splits, S a function of N, K and the SM
// count only.  Each split is accumulated from zero in TMEM, and the splits
// are added in split order: y = ((0 + P_0) + P_1) + ... + P_{S-1}.  Because
// S never depends on M, a row's result is bit-identical whatever other rows
// share the call.  Two schedules produce exactly that sum:
//
//  * split clusters (up to a few hundred rows): the S split CTAs of one tile
//    form a thread-block cluster; each stages its partial tile in its own
//    shared memory, and after a cluster barrier CTA r sums slice r of the
//    tile over the S partials through distributed shared memory.  No
//    partial touches global memory.
//  * persistent tiles (many rows): one CTA per SM walks tiles and, within a
//    tile, the S splits in order, with two TMEM accumulators so that the
//    tensor core fills one while the epilogue warps drain the other into a
//    running sum kept in a third TMEM region.  Consecutive tiles share a
//    weight tile, so the CTAs running at one time read each weight tile from
//    HBM once and find it in L2 after that.  Products with an fp32 output
//    use tiles 256 activation rows wide instead (MMA N = 256): per FLOP a
//    stage then moves a quarter fewer bytes from L2 into shared memory, and
//    the two 256-column accumulators fill TMEM, so the running sum of the
//    splits lives in the fp32 output itself, added in the same order.
//
// Roles in a 192-thread CTA: warp 0 lane 0 issues TMA loads into a
// STAGES-deep ring, warp 1 lane 0 issues the MMAs (4 x K=16 per 64-wide
// stage) and owns the TMEM allocation, warps 2..5 drain TMEM (warp w reads
// lanes 32*(w%4)..+31).  Every wait is bounded: a wait that runs past its
// limit sets bit 4 of the error word, and the CTA drains its own copies and
// MMAs, frees its TMEM and exits through the same barriers as a good run.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <string>
#include <type_traits>

#include "common.cuh"
#include "gemm_tc.h"
#include "launch.h"
#include "tc_ptx.cuh"

namespace dfl {

namespace {

namespace cg = cooperative_groups;
using namespace tc;
using bf16 = __nv_bfloat16;

thread_local std::string g_tc_err;

constexpr int BM = 128;        // weight rows per tile (MMA M)
constexpr int BK = 64;         // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
// Splits are clusters of at most 4 CTAs: with 8, only about half of the
// clusters of a one-wave grid were resident at once on GB300 and the rest ran
// as a second wave.
constexpr int kMaxSplits = 4;
constexpr int kMaxStages = 16;
constexpr size_t kBarrierBytes = 512;
constexpr int kPersistBN = 128;
constexpr int kWideBN = 256;   // persistent tiles of fp32-output products
constexpr int kErrBit = 4;

struct TcParams {
  void* Y;         // fp32 output, bf16 residual stream, or bf16 SwiGLU product
  int64_t ldy;
  int M, N;        // activation rows; output features
  int mode;        // TcMode
  int m_tiles, n_tiles, splits, kb_total;
  int vec;         // rows of Y start on 16-byte boundaries (ldy % 4 == 0, Y aligned)
  int stages;      // depth of the TMA ring (2..kMaxStages), from the shared memory budget
  void* const* yseg;  // fp32 output only: rows [j*seg_rows, (j+1)*seg_rows) go to yseg[j] (NULL: Y)
  int seg_rows;
  int* err;
  float* ws;          // 256-wide persistent tiles of the residual mode: [M][N] fp32 running sum of the splits
  // grouped products (256-wide fp32 tiles only): `groups` independent
  // products of the same shape, X stacked [groups * M][K], W stacked
  // [groups * N][K], product g written at Y + g * y_group
  int groups;
  int64_t y_group;
  // 1: the next kernel may start only once every thread of a CTA is past
  // its wait (the whole chain before this kernel has finished), so that it
  // can read that chain's tables before its own wait; 0: at once
  int late_trigger;
};

// The tile a unit index names: product g, weight-row tile, activation-row tile.
struct TileIdx {
  int g, m_tile, n_tile;
};
__device__ __forceinline__ TileIdx tile_of(const TcParams& p, int t) {
  const int per = p.m_tiles * p.n_tiles;
  return TileIdx{t / per, (t % per) / p.n_tiles, (t % per) % p.n_tiles};
}

constexpr int stage_bytes(int BN) { return BM * BK * 2 + BN * BK * 2; }
template <int BN, bool PERSIST>
__host__ __device__ constexpr int tmem_cols() {
  return PERSIST ? 512 : BN < 32 ? 32 : BN;
}
// Dynamic shared memory: the TMA ring, then (128-row persistent tiles only)
// the fp32 tile staged for the store, which in the cluster schedule aliases
// the idle ring instead; then the barriers.
// (256-wide SwiGLU tiles: the up half of one 32-column chunk, 64 rows with a
// padded stride of 33 floats, for the exchange between the epilogue warps.)
constexpr bool stages_tile(int BN, bool persist) { return persist && BN == kPersistBN; }
constexpr size_t kSwiXchBytes = 64 * 33 * 4;
constexpr size_t extra_bytes(int BN, bool persist, bool swi) {
  return stages_tile(BN, persist) ? (size_t)BN * BM * 4 : (persist && swi ? kSwiXchBytes : 0);
}
size_t smem_bytes(int BN, bool persist, bool swi, int stages) {
  return (size_t)stages * stage_bytes(BN) + extra_bytes(BN, persist, swi) + 1024 + kBarrierBytes;
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// Barrier of the four epilogue warps that also ORs a flag across them, so
// that all four take the same branch after it.
__device__ __forceinline__ bool epi_bar_or(bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)v)
      : "memory");
  return out != 0;
}

// Split s of the tile's K range, in 64-wide blocks.
__device__ __forceinline__ void split_range(const TcParams& p, int s, int& kb0, int& kb1) {
  kb0 = (int)((int64_t)s * p.kb_total / p.splits);
  kb1 = (int)((int64_t)(s + 1) * p.kb_total / p.splits);
}

// Walks this CTA's (tile, split) units in order, calling f(tile, split) for
// each; f returns false to stop.
template <bool PERSIST, typename F>
__device__ __forceinline__ void for_each_unit(const TcParams& p, F f) {
  const int tiles = p.m_tiles * p.n_tiles * p.groups;
  if (PERSIST) {
    for (int t = blockIdx.x; t < tiles; t += gridDim.x)
      for (int s = 0; s < p.splits; ++s)
        if (!f(t, s)) return;
  } else {
    f((int)blockIdx.x / p.splits, (int)blockIdx.x % p.splits);
  }
}

template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float* v) {
  if constexpr (N == 32) tmem_ld32(taddr, v);
  else tmem_ld16(taddr, v);
}

// Writes the tile's 4-feature groups [lo, hi) (group e = column c * rows/4
// + f/4, so consecutive threads write consecutive features) through the
// output mode.  get4(c, f) returns the fp32 sums of weight rows f..f+3 for
// token column c.  Loads are issued for U groups before any store depends on
// them; a group that crosses N, or an output without 16-byte rows, is
// written element by element.
template <bool SWI, typename Get4>
__device__ __forceinline__ void store_tile(const TcParams& p, int m_tile, int tok0, int lo, int hi, int tid, int nthr,
                                           Get4 get4) {
  constexpr int U = 2;
  constexpr int ROWS = SWI ? BM / 2 : BM;
  constexpr int G = ROWS / 4;
  const bool bf = SWI || p.mode == kResidBf16;
  for (int e0 = lo + tid; e0 < hi; e0 += U * nthr) {
    float4 v[U], w[U];
    void* yp[U];  // first output element of the group
    int nv[U];    // valid features of the group (0..4)
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = e0 + u * nthr;
      const int c = e / G, f = (e % G) * 4;
      const int t = tok0 + c, feat = m_tile * ROWS + f;
      nv[u] = (e < hi && t < p.M) ? max(0, min(4, p.N - feat)) : 0;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      w[u] = v[u];
      yp[u] = nullptr;
      if (!nv[u]) continue;
      if (p.yseg)
        yp[u] = reinterpret_cast<float*>(p.yseg[t / p.seg_rows]) + (int64_t)(t % p.seg_rows) * p.ldy + feat;
      else if (bf)
        yp[u] = reinterpret_cast<bf16*>(p.Y) + (int64_t)t * p.ldy + feat;
      else
        yp[u] = reinterpret_cast<float*>(p.Y) + (int64_t)t * p.ldy + feat;
      v[u] = get4(c, f);
      if (SWI) {
        w[u] = get4(c, f + BM / 2);
      } else if (p.mode == kResidBf16) {
        const bf16* h = reinterpret_cast<const bf16*>(yp[u]);
        if (nv[u] == 4 && p.vec) {
          const uint2 raw = *reinterpret_cast<const uint2*>(h);
          const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
          const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
          w[u] = make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
        } else {
          float* wf = reinterpret_cast<float*>(&w[u]);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < nv[u]) wf[i] = __bfloat162float(h[i]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!nv[u]) continue;
      float4 o;
      if (SWI) {
        const float* g = reinterpret_cast<const float*>(&v[u]);
        const float* up = reinterpret_cast<const float*>(&w[u]);
        float* of = reinterpret_cast<float*>(&o);
#pragma unroll
        for (int i = 0; i < 4; ++i) of[i] = g[i] / (1.f + expf(-g[i])) * up[i];
      } else if (p.mode == kResidBf16) {
        o = make_float4(w[u].x + v[u].x, w[u].y + v[u].y, w[u].z + v[u].z, w[u].w + v[u].w);
      } else {
        o = v[u];
      }
      if (bf) {
        bf16* y = reinterpret_cast<bf16*>(yp[u]);
        if (nv[u] == 4 && p.vec) {
          const __nv_bfloat162 a = __floats2bfloat162_rn(o.x, o.y), b = __floats2bfloat162_rn(o.z, o.w);
          uint2 raw;
          raw.x = *reinterpret_cast<const uint32_t*>(&a);
          raw.y = *reinterpret_cast<const uint32_t*>(&b);
          *reinterpret_cast<uint2*>(y) = raw;
        } else {
          const float* of = reinterpret_cast<const float*>(&o);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < nv[u]) y[i] = __float2bfloat16_rn(of[i]);
        }
      } else {
        float* y = reinterpret_cast<float*>(yp[u]);
        if (nv[u] == 4 && p.vec) {
          *reinterpret_cast<float4*>(y) = o;
        } else {
          const float* of = reinterpret_cast<const float*>(&o);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < nv[u]) y[i] = of[i];
        }
      }
    }
  }
}

// SWI: the 128-row weight tile is 64 gate rows then the 64 matching up rows
// (two TMA boxes from two matrices), and the epilogue writes silu(g) * u.
template <int BN, bool SWI, bool PERSIST>
__global__ void __launch_bounds__(kThreads, PERSIST ? 1 : 2) k_gemm_tc(const __grid_constant__ CUtensorMap tmW,
                                                                       const __grid_constant__ CUtensorMap tmW2,
                                                                       const __grid_constant__ CUtensorMap tmX,
                                                                       TcParams p) {
  const int STAGES = p.stages;
  constexpr int A_BYTES = BM * BK * 2;
  constexpr int B_BYTES = BN * BK * 2;
  constexpr uint32_t TX = A_BYTES + B_BYTES;
  constexpr int CH = BN < 32 ? BN : 32;
  constexpr int ROWS = SWI ? BM / 2 : BM;
  static_assert(!PERSIST || BN == kPersistBN || BN == kWideBN, "persistent tile widths");
  // 256-wide persistent tiles: the running sum of the splits lives in the fp32
  // output (kF32) or in p.ws (residual); SwiGLU tiles come with one split only
  constexpr bool WIDE = PERSIST && BN == kWideBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  float* stg = PERSIST ? reinterpret_cast<float*>(sB + STAGES * B_BYTES) : reinterpret_cast<float*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES + extra_bytes(BN, PERSIST, SWI));
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;  // [2] accumulator b holds a finished split
  uint64_t* acce = accf + 2;        // [2] accumulator b has been drained
  uint64_t* drain = acce + 2;       // MMAs still in flight when a CTA aborts
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!p.late_trigger) pdl_trigger();  // the next kernel may be scheduled as this one's CTAs retire
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmW) : "memory");
    if (SWI) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmW2) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmX) : "memory");
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, (uint32_t)tmem_cols<BN, PERSIST>());
    fence_before();
  }
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer ----
    uint64_t pol_w, pol_x;
    if (PERSIST) {
      // a weight tile is read by the CTAs of neighbouring tiles at about the same time
      asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol_w));
    } else {
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
    }
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_x));
    auto load_w = [&](int st, int t, int kb) {
      const TileIdx ti = tile_of(p, t);
      if (SWI) {
        tma_load_2d(sA + st * A_BYTES, &tmW, &full[st], kb * BK, ti.m_tile * (BM / 2), pol_w);
        tma_load_2d(sA + st * A_BYTES + A_BYTES / 2, &tmW2, &full[st], kb * BK, ti.m_tile * (BM / 2), pol_w);
      } else {
        tma_load_2d(sA + st * A_BYTES, &tmW, &full[st], kb * BK, ti.g * p.N + ti.m_tile * BM, pol_w);
      }
    };
    // Weights do not depend on the previous kernel: the first stages of them
    // are requested before waiting for it, so the weight stream starts while
    // the previous kernel drains.
    int it = 0;
    for_each_unit<PERSIST>(p, [&](int t, int s) {
      int kb0, kb1;
      split_range(p, s, kb0, kb1);
      for (int kb = kb0; kb < kb1 && it < STAGES; ++kb, ++it) {
        mbar_expect_tx(&full[it], TX);
        load_w(it, t, kb);
      }
      return it < STAGES;
    });
    const int pre = it;
    pdl_wait();
    if (p.late_trigger) pdl_trigger();
    it = 0;
    bool ok = true;
    for_each_unit<PERSIST>(p, [&](int t, int s) {
      int kb0, kb1;
      split_range(p, s, kb0, kb1);
      const TileIdx ti = tile_of(p, t);
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int st = it % STAGES;
        if (it >= pre) {
          if (!mbar_wait(&empty[st], ((uint32_t)(it / STAGES) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            return false;
          }
          mbar_expect_tx(&full[st], TX);
          load_w(st, t, kb);
        }
        tma_load_2d(sB + st * B_BYTES, &tmX, &full[st], kb * BK, ti.g * p.M + ti.n_tile * BN, pol_x);
      }
      return true;
    });
    if (!ok) {
      atomicOr(p.err, kErrBit);
      *abort_flag = 1;
      // let this CTA's own copies land before its shared memory is released
      for (int i = max(0, it - STAGES); i < it; ++i) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&full[i % STAGES], (uint32_t)(i / STAGES) & 1u) &&
               globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 0) {
    // The producer warp's other lanes are idle until the epilogue.  A CTA's
    // trigger counts once every one of its threads has executed it, so with a
    // late trigger they wait and trigger at once rather than at the end.
    if (p.late_trigger) {
      pdl_wait();
      pdl_trigger();
    }
  } else if (warp == 1) {
    // ---- MMA issuer: the whole warp runs the loop (every lane waits on the
    // barriers itself, decisions are taken together) and one elected lane
    // issues, so the MMAs queue without holding the warp up ----
    constexpr uint32_t idesc = idesc_bf16(BM, BN);
    int it = 0, j = 0;
    bool ok = true;
    if (p.late_trigger) {  // this warp reads no memory of earlier kernels: the wait costs it nothing
      pdl_wait();
      pdl_trigger();
    }
    for_each_unit<PERSIST>(p, [&](int, int s) {
      const int b = PERSIST ? (j & 1) : 0;
      if (PERSIST && j >= 2 &&
          !__all_sync(0xffffffffu, mbar_wait(&acce[b], (uint32_t)((j >> 1) - 1) & 1u, abort_flag))) {
        ok = false;
        return false;
      }
      fence_after();
      const uint32_t d = tmem + (uint32_t)(b * BN);
      int kb0, kb1;
      split_range(p, s, kb0, kb1);
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int st = it % STAGES;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (uint32_t)(it / STAGES) & 1u, abort_flag))) {
          ok = false;
          return false;
        }
        fence_after();
        const uint32_t a0 = smem_u32(sA + st * A_BYTES), b0 = smem_u32(sB + st * B_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          umma_bf16_warp(d, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), idesc, (kb > kb0 || k > 0) ? 1u : 0u);
        umma_commit_warp(&empty[st]);
      }
      umma_commit_warp(&accf[b]);  // arrives once every MMA of this split has completed
      ++j;
      return true;
    });
    if (!ok) {
      if (lane == 0) atomicOr(p.err, kErrBit);
      *abort_flag = 1;
      umma_commit_warp(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  } else if (warp >= 2) {
    // ---- epilogue: TMEM -> sums -> staged tile ----
    const int q = warp & 3;  // the TMEM lane quarter this warp may read
    const int row = q * 32 + lane;
    const uint32_t lanes = tmem + ((uint32_t)(q * 32) << 16);
    pdl_wait();  // the stores below read (residual) and write memory of earlier kernels
    if (p.late_trigger) pdl_trigger();
    int j = 0;
    for_each_unit<PERSIST>(p, [&](int t, int s) {
      const int b = PERSIST ? (j & 1) : 0;
      bool bad = !mbar_wait(&accf[b], PERSIST ? (uint32_t)(j >> 1) & 1u : 0u, abort_flag);
      if (PERSIST) bad = epi_bar_or(bad);
      if (bad) {
        if (lane == 0) atomicOr(p.err, kErrBit);
        *abort_flag = 1;
        return false;
      }
      fence_after();
      const uint32_t acc = lanes + (uint32_t)(b * BN);
      if constexpr (WIDE) {
        const TileIdx ti = tile_of(p, t);
        const int tok0 = ti.n_tile * BN, m_tile = ti.m_tile;
        const bool last = s == p.splits - 1;
        if constexpr (SWI) {
          // one split: gate rows 0..63 take the matching up row (64 + r) of
          // each 32-column chunk through shared memory
          const int r64 = row & 63, feat = m_tile * (BM / 2) + r64;
          bf16* y = reinterpret_cast<bf16*>(p.Y) + feat;
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 32) {
            float v[32];
            tmem_ld32(acc + c0, v);
            if (row >= 64) {
#pragma unroll
              for (int i = 0; i < 32; ++i) stg[r64 * 33 + i] = v[i];
            }
            epi_bar();
            const int nt = (row < 64 && feat < p.N) ? min(32, p.M - (tok0 + c0)) : 0;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < nt) {
                const float g = v[i], u = stg[r64 * 33 + i];
                y[(int64_t)(tok0 + c0 + i) * p.ldy] = __float2bfloat16_rn(g / (1.f + expf(-g)) * u);
              }
            epi_bar();
          }
        } else {
          // Y (fp32 output) or p.ws (residual) holds the running sum of the
          // splits so far, ((0 + P_0) + P_1) + ...; a thread only rereads what
          // it wrote for the split before (a tile's splits run in order here)
          const int feat = m_tile * BM + row;
          const bool resid = p.mode == kResidBf16;
          auto run_ptr = [&](int tok) -> float* {
            if (resid) return p.ws + (int64_t)tok * p.N + feat;
            if (p.yseg) return reinterpret_cast<float*>(p.yseg[tok / p.seg_rows]) + (int64_t)(tok % p.seg_rows) * p.ldy + feat;
            return reinterpret_cast<float*>(p.Y) + ti.g * p.y_group + (int64_t)tok * p.ldy + feat;
          };
          // 32 columns at a time for an fp32 output, 16 for the residual
          // stream (which also holds h in registers)
          auto chunk = [&](auto cw_tag, int c0) {
            constexpr int CW = decltype(cw_tag)::value;
            float v[CW];
            tmem_ld<CW>(acc + c0, v);
            const int nt = feat < p.N ? min(CW, p.M - (tok0 + c0)) : 0;
            if (s > 0) {
              float pr[CW];
#pragma unroll
              for (int i = 0; i < CW; ++i) pr[i] = i < nt ? *run_ptr(tok0 + c0 + i) : 0.f;
#pragma unroll
              for (int i = 0; i < CW; ++i) v[i] = pr[i] + v[i];
            } else {
#pragma unroll
              for (int i = 0; i < CW; ++i) v[i] = 0.f + v[i];
            }
            if (resid && last) {
              bf16* h = reinterpret_cast<bf16*>(p.Y) + feat;
              float hv[CW];
#pragma unroll
              for (int i = 0; i < CW; ++i) hv[i] = i < nt ? __bfloat162float(h[(int64_t)(tok0 + c0 + i) * p.ldy]) : 0.f;
#pragma unroll
              for (int i = 0; i < CW; ++i)
                if (i < nt) h[(int64_t)(tok0 + c0 + i) * p.ldy] = __float2bfloat16_rn(hv[i] + v[i]);
            } else {
#pragma unroll
              for (int i = 0; i < CW; ++i)
                if (i < nt) *run_ptr(tok0 + c0 + i) = v[i];
            }
          };
          if (resid) {
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 16) chunk(std::integral_constant<int, 16>(), c0);
          } else {
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) chunk(std::integral_constant<int, 32>(), c0);
          }
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[b]);
        ++j;
        return true;
      }
      const uint32_t run = lanes + (uint32_t)(2 * BN);  // running sum (persistent, split > 0)
      const bool last = s == p.splits - 1;
      if (!PERSIST || last) {
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += CH) {
          float v[CH];
          tmem_ld<CH>(acc + c0, v);
          if (PERSIST && p.splits > 1) {
            float r[CH];
            tmem_ld<CH>(run + c0, r);
#pragma unroll
            for (int i = 0; i < CH; ++i) v[i] = r[i] + v[i];
          }
#pragma unroll
          for (int i = 0; i < CH; ++i) stg[(c0 + i) * BM + row] = v[i];
        }
      } else {
        // running sum of the splits so far: (0 + P_0) + P_1 + ...
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32], r[32];
          tmem_ld32(acc + c0, v);
          if (s == 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0.f + v[i];
          } else {
            tmem_ld32(run + c0, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = r[i] + v[i];
          }
          tmem_st32(run + c0, r);
        }
      }
      // accumulator b may be refilled
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[b]);
      if (PERSIST && last) {
        epi_bar();  // the staged tile is complete
        store_tile<SWI>(p, t / p.n_tiles, (t % p.n_tiles) * BN, 0, BN * ROWS / 4, (int)threadIdx.x - 64, kEpiThreads,
                        [&](int c, int f) { return *reinterpret_cast<const float4*>(&stg[c * BM + f]); });
        epi_bar();  // staging is free for the next tile
      }
      ++j;
      return true;
    });
  }
  __syncwarp();

  if (!PERSIST) {
    // ---- split clusters: sum the partials in split order, then store ----
    pdl_wait();
    if (p.late_trigger) pdl_trigger();
    const int t = (int)blockIdx.x / p.splits;
    const int m_tile = t / p.n_tiles, tok0 = (t % p.n_tiles) * BN;
    const int E = BN * ROWS / 4;  // 4-feature groups of the tile
    if (p.splits == 1) {
      __syncthreads();
      if (!*abort_flag)
        store_tile<SWI>(p, m_tile, tok0, 0, E, threadIdx.x, kThreads,
                        [&](int c, int f) { return *reinterpret_cast<const float4*>(&stg[c * BM + f]); });
    } else {
      cg::cluster_group cl = cg::this_cluster();
      cl.sync();  // every partial of the tile is staged
      const int r = (int)cl.block_rank();
      const float4* peer[kMaxSplits];
#pragma unroll
      for (int i = 0; i < kMaxSplits; ++i)
        peer[i] = reinterpret_cast<const float4*>(i < p.splits ? cl.map_shared_rank(stg, i) : stg);
      const int lo = (int)((int64_t)r * E / p.splits), hi = (int)((int64_t)(r + 1) * E / p.splits);
      if (!*abort_flag)
        store_tile<SWI>(p, m_tile, tok0, lo, hi, threadIdx.x, kThreads, [&](int c, int f) {
          const int idx = (c * BM + f) / 4;
          float4 v[kMaxSplits];
#pragma unroll
          for (int i = 0; i < kMaxSplits; ++i) v[i] = i < p.splits ? peer[i][idx] : make_float4(0.f, 0.f, 0.f, 0.f);
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int i = 0; i < kMaxSplits; ++i)
            if (i < p.splits) {
              acc.x += v[i].x;
              acc.y += v[i].y;
              acc.z += v[i].z;
              acc.w += v[i].w;
            }
          return acc;
        });
      cluster_sync_relaxed();  // no CTA leaves while a peer still reads its partial
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tmem, (uint32_t)tmem_cols<BN, PERSIST>());
  }
}

}  // namespace

struct TcContext {
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  int num_sms = 0;
  int* err = nullptr;
  bool attr_set[16] = {};
};

const char* tc_last_error() { return g_tc_err.c_str(); }

static int tc_fail(const char* what, cudaError_t e = cudaSuccess) {
  char buf[256];
  snprintf(buf, sizeof buf, "%s%s%s", what, e != cudaSuccess ? ": " : "", e != cudaSuccess ? cudaGetErrorString(e) : "");
  g_tc_err = buf;
  return -1;
}

int tc_create(TcContext** out, int num_sms, int* err) {
  TcContext* c = new TcContext();
  c->num_sms = num_sms;
  c->err = err;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void**)&c->encode, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !c->encode) {
    delete c;
    return tc_fail("cuTensorMapEncodeTiled entry point", e);
  }
  *out = c;
  return 0;
}

void tc_destroy(TcContext* c) { delete c; }

static int encode_2d(TcContext* c, CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, int64_t ld_elems,
                     uint32_t box_rows) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {(cuuint64_t)ld_elems * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = c->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[128];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    g_tc_err = buf;
    return -1;
  }
  return 0;
}

int tc_encode_kv_maps(TcContext* c, const void* kv, int64_t cap, int d, int planes, CUtensorMap* out) {
  // K planes: [planes][cap][d], box {64 channels, 64 positions, 1 plane}
  {
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)cap, (cuuint64_t)planes};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)cap * d * 2};
    const cuuint32_t box[3] = {64, 64, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (c->encode(&out[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(kv), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return tc_fail("K plane tensor map");
  }
  // V^T planes: [planes][d][cap], box {64 positions, d channels, 1 plane}
  {
    const cuuint64_t dims[3] = {(cuuint64_t)cap, (cuuint64_t)d, (cuuint64_t)planes};
    const cuuint64_t strides[2] = {(cuuint64_t)cap * 2, (cuuint64_t)cap * d * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)d, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (c->encode(&out[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(kv), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return tc_fail("V plane tensor map");
  }
  return 0;
}

// Largest dynamic shared memory a k_gemm_tc launch asks for.
constexpr size_t kSmemMax = 227 * 1024;

template <int BN, bool SWI, bool PERSIST>
static int launch_bn(TcContext* c, const CUtensorMap& mw, const CUtensorMap& mw2, const CUtensorMap& mx,
                     const TcParams& p, int grid, int cluster, cudaStream_t st, int slot) {
  const size_t smem = smem_bytes(BN, PERSIST, SWI, p.stages);
  if (smem > kSmemMax || p.stages < 2 || p.stages > kMaxStages || (size_t)BN * BM * 4 > (size_t)p.stages * stage_bytes(BN))
    return tc_fail("tc_gemm: pipeline does not fit shared memory");
  if (!c->attr_set[slot]) {
    cudaError_t e =
        cudaFuncSetAttribute(k_gemm_tc<BN, SWI, PERSIST>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemMax);
    if (e != cudaSuccess) return tc_fail("smem attribute", e);
    c->attr_set[slot] = true;
  }
  const cudaError_t e = launch_kc(k_gemm_tc<BN, SWI, PERSIST>, grid, kThreads, smem, st, cluster, mw, mw2, mx, p);
  if (e != cudaSuccess) return tc_fail("k_gemm_tc launch", e);
  return 0;
}

template <bool SWI>
static int launch_mode(TcContext* c, int BN, bool persist, const CUtensorMap& mw, const CUtensorMap& mw2,
                       const CUtensorMap& mx, const TcParams& p, int grid, int cluster, cudaStream_t st) {
  const int base = SWI ? 6 : 0;
  if (persist && BN == kWideBN) return launch_bn<kWideBN, SWI, true>(c, mw, mw2, mx, p, grid, cluster, st, SWI ? 13 : 12);
  if (persist) return launch_bn<kPersistBN, SWI, true>(c, mw, mw2, mx, p, grid, cluster, st, base + 5);
  switch (BN) {
    case 16: return launch_bn<16, SWI, false>(c, mw, mw2, mx, p, grid, cluster, st, base + 0);
    case 32: return launch_bn<32, SWI, false>(c, mw, mw2, mx, p, grid, cluster, st, base + 1);
    case 64: return launch_bn<64, SWI, false>(c, mw, mw2, mx, p, grid, cluster, st, base + 2);
    default: return launch_bn<128, SWI, false>(c, mw, mw2, mx, p, grid, cluster, st, base + 3);
  }
}

int tc_gemm_grouped(TcContext* c, const void* X, int64_t ldx, const void* W, int64_t ldw, float* Y, int64_t ldy,
                    int64_t y_group, int M, int N, int K, int groups, cudaStream_t st) {
  if (M <= 0 || N <= 0 || groups <= 0) return 0;
  if (K % BK || ldx % 8 || ldw % 8 || ((uintptr_t)X & 15) || ((uintptr_t)W & 15))
    return tc_fail("tc_gemm_grouped: K must be a multiple of 64, strides multiples of 8, operands 16-byte aligned");
  const int m_tiles = (N + BM - 1) / BM, kb_total = K / BK;
  // the splits of one product of this shape, as tc_gemm chooses them
  int cap = std::max(1, std::min({2 * c->num_sms / m_tiles, kMaxSplits, std::max(1, kb_total / 2)}));
  int splits = 1;
  while (splits * 2 <= cap) splits *= 2;
  const int n_tiles = (M + kWideBN - 1) / kWideBN;
  const int tiles = m_tiles * n_tiles * groups;
  CUtensorMap mw, mx;
  if (encode_2d(c, &mw, W, (uint64_t)K, (uint64_t)N * groups, ldw, (uint32_t)BM)) return -1;
  if (encode_2d(c, &mx, X, (uint64_t)K, (uint64_t)M * groups, ldx, (uint32_t)kWideBN)) return -1;
  const size_t fixed = extra_bytes(kWideBN, true, false) + 1024 + kBarrierBytes;
  const int stages = (int)std::min<size_t>(kMaxStages, (kSmemMax - fixed) / stage_bytes(kWideBN));
  TcParams p{Y, ldy, M, N, kF32, m_tiles, n_tiles, splits, kb_total, 0, stages, nullptr, 0, c->err, nullptr, groups,
             y_group, 0};
  return launch_bn<kWideBN, false, true>(c, mw, mw, mx, p, std::min(tiles, c->num_sms), 1, st, 12);
}

int tc_gemm(TcContext* c, const void* X, int64_t ldx, const void* W, const void* W2, int64_t ldw, void* Y,
            int64_t ldy, int M, int N, int K, int mode, cudaStream_t st, void* const* yseg, int seg_rows, float* ws,
            int late_trigger) {
  if (M <= 0 || N <= 0) return 0;
  const bool swi = mode == kSwigluBf16;
  if (yseg && (mode != kF32 || seg_rows <= 0)) return tc_fail("tc_gemm: row segments need fp32 output");
  if (K % BK || ldx % 8 || ldw % 8 || ((uintptr_t)X & 15) || ((uintptr_t)W & 15) || (swi && ((uintptr_t)W2 & 15)))
    return tc_fail("tc_gemm: K must be a multiple of 64, strides multiples of 8, operands 16-byte aligned");
  if (mode < kF32 || mode > kSwigluBf16) return tc_fail("tc_gemm: unknown mode");
  const int rows_per_tile = swi ? BM / 2 : BM;
  const int m_tiles = (N + rows_per_tile - 1) / rows_per_tile, kb_total = K / BK;
  // The split of K fills about one wave of two CTAs per SM with the weight
  // tiles of a small call; it depends on N, K and the SM count only.  It is
  // a power of two: clusters of 3, 5, 6 or 7 CTAs pack the GPCs badly (a
  // 6-way split of a 48-tile product ran 1.5x slower than a 4-way one).
  int cap = std::max(1, std::min({2 * c->num_sms / m_tiles, kMaxSplits, std::max(1, kb_total / 2)}));
  int splits = 1;
  while (splits * 2 <= cap) splits *= 2;
  // Many rows: persistent 128-row tiles once they cover half of the SMs;
  // otherwise one CTA per (tile, split), the splits of a tile in a cluster.
  const int tiles128 = m_tiles * ((M + kPersistBN - 1) / kPersistBN);
  const bool persist = M > 128 && 2 * tiles128 >= c->num_sms;
  const bool wide = persist && (mode == kF32 || (mode == kResidBf16 && ws) || (swi && splits == 1));
  const int BN = wide ? kWideBN : persist ? kPersistBN : M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
  const int n_tiles = (M + BN - 1) / BN;
  const int tiles = m_tiles * n_tiles;
  CUtensorMap mw, mw2, mx;
  if (encode_2d(c, &mw, W, (uint64_t)K, (uint64_t)N, ldw, (uint32_t)rows_per_tile)) return -1;
  if (swi) {
    if (encode_2d(c, &mw2, W2, (uint64_t)K, (uint64_t)N, ldw, (uint32_t)rows_per_tile)) return -1;
  } else {
    mw2 = mw;
  }
  if (encode_2d(c, &mx, X, (uint64_t)K, (uint64_t)M, ldx, (uint32_t)BN)) return -1;
  const int vec = ldy % 4 == 0 && ((uintptr_t)Y & 15) == 0;
  const int grid = persist ? std::min(tiles, c->num_sms) : tiles * splits;
  // Pipeline depth from the shared memory of one CTA per SM when the grid
  // fits one per SM, else of two: each CTA's stream is latency-bound, so the
  // bytes in flight per SM set its bandwidth.
  const size_t fixed = extra_bytes(BN, persist, swi) + 1024 + kBarrierBytes;
  const size_t budget = (persist || grid <= c->num_sms) ? kSmemMax : 112 * 1024;
  const int stages = (int)std::min<size_t>(kMaxStages, (budget - fixed) / stage_bytes(BN));
  TcParams p{Y, ldy, M, N, mode, m_tiles, n_tiles, splits, kb_total, vec, stages, yseg, seg_rows, c->err, ws, 1, 0,
             late_trigger};
  const int cluster = persist ? 1 : splits;
  return swi ? launch_mode<true>(c, BN, persist, mw, mw2, mx, p, grid, cluster, st)
             : launch_mode<false>(c, BN, persist, mw, mw2, mx, p, grid, cluster, st);
}

}  // namespace dfl
