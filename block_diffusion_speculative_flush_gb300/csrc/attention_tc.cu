// Block attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA) for bf16
// drafts with head_dim 128: the n+1 block rows x the group's query heads of
// one KV head attend over one range of key positions (context, then the
// block's own rows), with the window limit and the causal / bidirectional
// in-block mask applied per query row (Laguna PR: the window is a per-query
// limit over [context | block]).
//
// One CTA per work item (session, KV head, key range starting on a multiple
// of 64).  Query rows (at most 128, zero padded) form the MMA's M = 128 side.
//   warps 8, 10   TMA, one producer per ring: 64-key K tiles [64 keys][128 d]
//                 into a 4-stage ring (warp 8) and the matching V^T tiles
//                 [128 d][64 keys] into a 5-stage ring (warp 10); the cache
//                 keeps V transposed so that both are K-major operand tiles.
//                 A K stage is free once S = Q K^T is done, a V stage once
//                 P V is done.
//   warp 9        MMA, the whole warp running one loop and one elected lane
//                 issuing (queued MMAs do not hold the warp up): S(t) = Q K^T
//                 into one of two TMEM buffers as soon as K(t) has landed and
//                 the softmax has read S(t-2) out of that buffer; O += P V^T,
//                 each stream's tiles in order, as soon as P(u) and V(u) are
//                 in shared memory.  P is a bf16 pair hi + lo (~16 bits of the
//                 probabilities): two MMAs per 16 keys.
//   warps 0..7    softmax, two threads per query row (warps w and w + 4 read
//                 the same TMEM lanes; each takes 32 keys of a tile and 64
//                 columns of O): S from TMEM, mask against the row's visible
//                 key range, online max in the exp2 domain with lazy
//                 rescaling (O and the sum are rescaled only when the row max
//                 grows by more than 2^8, so P <= 256), P = 2^(s k - m) with
//                 the scale k folded into one packed two-lane FMA, written to
//                 shared memory as the next MMA's A operand; finally O and
//                 (max, sum) go out as this key range's partial.
// Two streams when the query rows fit in 64 (R <= 64): TMEM lanes are tied to
// warp quarters, so 64 rows would leave the softmax to warps 0, 1, 4, 5 (two
// of the four SM sub-partitions).  Instead Q is stored twice (rows 64..127
// repeat rows 0..63); warps of quarters 0-1 take the even key tiles (S buffer
// 0, O region 0, rows 0..63) and warps of quarters 2-3 the odd ones (S buffer
// 1, O region 1, rows 64..127), each with its own online softmax.  Each
// stream has its own O accumulator in TMEM, so the streams' products never
// wait on each other; both write their 64 rows of the one P tile, and a
// product's rows of the other stream land in O rows of its region that are
// never read.  The two streams' (max, sum, O) merge in shared memory at the
// end.  TMEM: O0 [0,128), O1 [128,256), S0 [256,320), S1 [320,384).
// Every wait is bounded; an expired wait sets bit 8 of the error word.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "launch.h"
#include "tc_ptx.cuh"

namespace dfl {

namespace {

using namespace tc;
namespace cg = cooperative_groups;

constexpr int D = 128;                       // head dim
constexpr int KT = 64;                       // keys per tile (MMA N of S)
constexpr int KST = 4;                       // K stages
constexpr int VST = 5;                       // V^T stages
constexpr int QBYTES = 128 * D * 2;          // Q: two [128 rows][64 d] swizzled blocks
constexpr int KBYTES = KT * D * 2;           // K tile: two [64 keys][64 d] blocks
constexpr int VBYTES = D * KT * 2;           // V^T tile: one [128 d][64 keys] block
constexpr int PBYTES = 128 * KT * 2;         // P tile: one [128 rows][64 keys] block
constexpr int DATA_BYTES = QBYTES + KST * KBYTES + VST * VBYTES + 2 * PBYTES;  // + barriers and exchange
constexpr int THREADS = 352;
constexpr int SOFTMAX_THREADS = 256;
constexpr uint32_t TMEM_COLS = 512;          // O0 [0,128), O1 [128,256) (two streams), S0 [256,320), S1 [320,384)
constexpr uint32_t S_COL = 256;

// max(a, b, c) in one instruction
__device__ __forceinline__ float max3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}
// 2^x on the special-function unit (results below 2^-126 flush to zero)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2unpack(uint64_t r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
// Two probabilities P = 2^(s k + c) of two scores s as bf16 pairs hi + lo
// (hi the rounded P, lo the rounded remainder; returns hi, lo through `lo`);
// P is added to the pair of partial sums.  The affine step, the remainder
// and the sum run as packed two-lane fp32 instructions.
__device__ __forceinline__ uint32_t p_pair(float s0, float s1, uint64_t k2, uint64_t c2, uint64_t& sum2, uint32_t& lo) {
  uint64_t x;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(x) : "l"(f2pack(s0, s1)), "l"(k2), "l"(c2));
  const float2 e = f2unpack(x);
  const float p0 = ex2(e.x), p1 = ex2(e.y);
  const uint64_t pp = f2pack(p0, p1);
  const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
  const uint32_t b = *reinterpret_cast<const uint32_t*>(&h);
  uint64_t rr;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(rr) : "l"(pp), "l"(f2pack(__uint_as_float(b << 16), __uint_as_float(b & 0xffff0000u))));
  const float2 r = f2unpack(rr);
  const __nv_bfloat162 l2 = __floats2bfloat162_rn(r.x, r.y);
  lo = *reinterpret_cast<const uint32_t*>(&l2);
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(sum2) : "l"(pp));
  return b;
}

// byte offset of 16-byte chunk c of row r inside a [rows][128 B] swizzled block
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// Named barrier `id` over `count` threads that also ANDs a predicate over them.
__device__ __forceinline__ bool bar_and(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(THREADS, 1) k_attn_tc(const bf16* __restrict__ Q, const AttnItem* __restrict__ items,
                                                        SessTables tabs, AttnParams p, float* __restrict__ part,
                                                        int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + QBYTES;
  uint8_t* sV = sK + KST * KBYTES;
  uint8_t* sP = sV + VST * VBYTES;  // [hi, lo]
  uint64_t* k_full = (uint64_t*)(sP + 2 * PBYTES);
  uint64_t* k_empty = k_full + KST;
  uint64_t* v_full = k_empty + KST;
  uint64_t* v_empty = v_full + VST;
  uint64_t* s_full = v_empty + VST;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* o_done = pv_done + 2;
  uint32_t* tmem_slot = (uint32_t*)(o_done + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  // [3][2][128]: per-half row max (one buffer per tile parity, so a thread
  // never overwrites a value its partner has not read) and the final sum
  float* xch = (float*)(tmem_slot + 4);

  // Merged in-kernel, the output goes to the O product, which reads nothing of
  // this call's tables early: it may start at once.  Partials go to
  // k_attn_combine, which does read them early: it starts only once every
  // thread here is past its wait.
  if (p.cluster > 1) pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool dual = p.nrows * (p.Hq / p.Hkv) <= 64;
  const int tile_threads = dual ? SOFTMAX_THREADS / 2 : SOFTMAX_THREADS;  // softmax threads per key tile

  if (tid == 0) {
    for (int s = 0; s < KST; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], tile_threads);
      mbar_init(&p_full[b], tile_threads);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(o_done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    fence_before();
  }
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  // The work item, the session tables and every cache row older than this
  // forward were written before the kernel that precedes this one (k_qkv_post,
  // or the V^T writer after it) finished its own wait, and that kernel lets
  // this one start only then: they are read before this kernel's wait.  Q and
  // the rows this forward writes come from that kernel and are read after it.
  const AttnItem it = items[blockIdx.x];
  const int G = p.Hq / p.Hkv, R = p.nrows * G;
  const int64_t F = tabs.frontier[it.sess], cap = tabs.cap[it.sess];
  const CUtensorMap* kmap = tabs.kvmaps[it.sess];
  const CUtensorMap* vmap = kmap + 1;
  const int planeK = 2 * p.layer * p.Hkv + it.kvh, planeV = (2 * p.layer + 1) * p.Hkv + it.kvh;
  const int T = (int)((it.k1 - it.k0 + KT - 1) / KT);
  // key tiles [0, T_old) hold no row that this forward writes
  int T_old = 0;
  if (tabs.fresh) {
    const int64_t fresh = tabs.fresh[it.sess];
    T_old = fresh <= it.k0 ? 0 : (int)min((int64_t)T, (fresh - it.k0) / KT);
  }
  if (tid == 256) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)kmap) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)vmap) : "memory");
  }

  // everyone but the producers waits here; they first request the tiles of
  // older rows
  if (warp != 8 && warp != 10) {
    pdl_wait();
    if (p.cluster == 1) pdl_trigger();
  }
  // Q (and the gates) come from the kernel just before: read after the wait
  const bf16* Qw = after_wait(Q);
  const float* gates = after_wait(p.gates);
  // ---- Q rows of this KV head, zero padded to 128 (two streams: rows 0..63
  // twice), as the MMA's A tile
  if (warp < 8) {
    // all 8 loads of a thread are issued before the first store
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int e = tid + SOFTMAX_THREADS * k, r = dual ? (e >> 4) & 63 : e >> 4, c = e & 15;
      v[k] = make_uint4(0, 0, 0, 0);
      if (r < R) {
        const int i = r / G, g = r % G;
        v[k] = *reinterpret_cast<const uint4*>(Qw + (((int64_t)it.sess * p.nrows + i) * p.Hq + it.kvh * G + g) * D +
                                              c * 8);
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int e = tid + SOFTMAX_THREADS * k, r = e >> 4, c = e & 15;
      *reinterpret_cast<uint4*>(sQ + (c >> 3) * (QBYTES / 2) + swz(r, c & 7)) = v[k];
    }
    fence_proxy_async();
  }
  // Q staged: the MMA warp needs it (and the softmax warps wrote it); the
  // producers do not, and start their loads at once
  if (warp < 8 || warp == 9) asm volatile("bar.sync 7, %0;" ::"r"(SOFTMAX_THREADS + 32) : "memory");

  if (warp == 8 || warp == 10) {
    // ---- TMA producers, one per ring: warp 8 the K tiles, warp 10 the V^T
    // tiles, so that neither ring waits for the other's free stage
    const bool isK = warp == 8;
    const int NS = isK ? KST : VST;
    uint64_t* full = isK ? k_full : v_full;
    uint64_t* empty = isK ? k_empty : v_empty;
    auto load = [&](int t) {
      const int st = t % NS;
      const int slot0 = (int)((it.k0 + (int64_t)t * KT) % cap);
      if (isK) {
        mbar_expect_tx(&full[st], KBYTES);
        tma_load_3d(sK + st * KBYTES, kmap, &full[st], 0, slot0, planeK);
        tma_load_3d(sK + st * KBYTES + KBYTES / 2, kmap, &full[st], 64, slot0, planeK);
      } else {
        mbar_expect_tx(&full[st], VBYTES);
        tma_load_3d(sV + st * VBYTES, vmap, &full[st], slot0, 0, planeV);
      }
    };
    // the first stages, where they hold older rows only, while the previous
    // kernel drains; then the whole warp waits (its other lanes write the
    // clustered merge's output at the end); then the rest in order
    const int early = min(T_old, NS);
    if (lane == 0)
      for (int t = 0; t < early; ++t) load(t);
    __syncwarp();
    pdl_wait();
    if (p.cluster == 1) pdl_trigger();
    if (lane == 0) {
      int issued = early;
      for (int t = early; t < T; ++t) {
        if (t >= NS && !mbar_wait(&empty[t % NS], (uint32_t)((t / NS) - 1) & 1u, abort_flag)) {
          atomicOr(err, 8);
          *abort_flag = 1;
          break;
        }
        load(t);
        ++issued;
      }
      if (*abort_flag) {  // let this CTA's own copies land before leaving
        for (int t = issued - NS > 0 ? issued - NS : 0; t < issued; ++t) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&full[t % NS], (uint32_t)(t / NS) & 1u) && globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 9) {
    // ---- MMA issuer: the whole warp runs the loop and takes every decision
    // together (each lane waits on the barrier itself); one elected lane
    // issues each MMA and commit, which queue without holding up the warp
    constexpr uint32_t idS = idesc_bf16(128, KT), idPV = idesc_bf16(128, D);
    const uint32_t tO = tmem;
    auto issue_s = [&](int t) {
      const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK + (t % KST) * KBYTES);
      const uint32_t tS = tmem + S_COL + (t & 1) * KT;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        umma_bf16_warp(tS, sdesc_sw128(q0 + (ks >> 2) * (QBYTES / 2) + (ks & 3) * 32),
                       sdesc_sw128(k0 + (ks >> 2) * (KBYTES / 2) + (ks & 3) * 32), idS, ks > 0 ? 1u : 0u);
      umma_commit_warp(&s_full[t & 1]);
      umma_commit_warp(&k_empty[t % KST]);  // the K stage is free once S(t) is done
    };
    // two streams: stream u & 1 accumulates into its own O region, so the
    // streams' products never wait on each other
    const int nst = dual ? 2 : 1;
    auto issue_pv = [&](int u) {
      const uint32_t ph = smem_u32(sP), pl = ph + PBYTES, v0 = smem_u32(sV + (u % VST) * VBYTES);
      const uint32_t tOu = tO + (dual ? (uint32_t)((u & 1) * D) : 0u);
#pragma unroll
      for (int ks = 0; ks < KT / 16; ++ks)
        umma_bf16_warp(tOu, sdesc_sw128(ph + ks * 32), sdesc_sw128(v0 + ks * 32), idPV, (u >= nst || ks > 0) ? 1u : 0u);
#pragma unroll
      for (int ks = 0; ks < KT / 16; ++ks) umma_bf16_warp(tOu, sdesc_sw128(pl + ks * 32), sdesc_sw128(v0 + ks * 32), idPV, 1u);
      umma_commit_warp(&pv_done[u & 1]);
      umma_commit_warp(&v_empty[u % VST]);
    };
    // S(t) as soon as K(t) has landed and the softmax has read S(t-2) out of
    // the same TMEM buffer, P V(u) (each stream's in tile order) as soon as
    // P(u) and V(u) are in place: S of a stream's next tile is computed while
    // the stream still works on its current one.  A test counts only once
    // every lane has seen the phase complete.
    int ns = 0, npv[2] = {0, 1};  // next S; next P V of each stream
    if (!dual) npv[1] = T;
    bool ok = true;
    uint64_t t0 = globaltimer_ns();
    for (uint32_t spin = 1; npv[0] < T || npv[1] < T; ++spin) {
      if (ns < T && __all_sync(0xffffffffu, mbar_test_wait(&k_full[ns % KST], (uint32_t)(ns / KST) & 1u) &&
                                                (ns < 2 || mbar_test_wait(&s_free[ns & 1], (uint32_t)((ns >> 1) - 1) & 1u)))) {
        fence_after();
        issue_s(ns++);
        t0 = globaltimer_ns();
        continue;
      }
      bool issued = false;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int u = npv[x];
        if (u < ns && __all_sync(0xffffffffu, mbar_test_wait(&p_full[u & 1], (uint32_t)(u >> 1) & 1u) &&
                                                  mbar_test_wait(&v_full[u % VST], (uint32_t)(u / VST) & 1u))) {
          fence_after();
          issue_pv(u);
          npv[x] = u + nst;
          issued = true;
        }
      }
      if (issued) {
        t0 = globaltimer_ns();
        continue;
      }
      if ((spin & 63u) == 0 && __any_sync(0xffffffffu, *abort_flag != 0 || globaltimer_ns() - t0 > kWaitLimitNs)) {
        ok = false;
        break;
      }
    }
    if (!ok) {
      if (lane == 0) atomicOr(err, 8);
      *abort_flag = 1;
    }
    umma_commit_warp(o_done);  // arrives once every MMA issued above has completed
  } else if (warp < 8) {
    // ---- softmax: two threads per TMEM row (row = TMEM lane)
    const int r = (warp & 3) * 32 + lane;
    const int half = warp >> 2;                // keys [32 half, +32) of a tile, O columns [64 half, +64)
    const int stream = dual ? (warp & 3) >> 1 : 0;  // key tiles stream, stream + tstep, ...
    const int tstep = dual ? 2 : 1;
    const int qr = r - 64 * stream;            // the query row this TMEM row holds
    const bool rv = qr < R;
    // warps w and w + 4 share their rows: the per-tile exchange is a barrier
    // of the pair alone, and it also makes the pair's decision to stop on an
    // expired wait a common one, so the two always meet the same barriers
    const int pair_bar = 1 + (warp & 3);
    // a warp whose 32 rows are all padding (qr >= R) computes nothing: the
    // P rows it would write only meet O rows that are never read.  It keeps
    // the barrier protocol (one arrival per tile on s_free and p_full, the
    // pair barrier), so no phase runs ahead of the others.
    const bool live = (warp & 3) * 32 - 64 * stream < R;
    const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t ocol = (uint32_t)(stream * D);  // this stream's O region (O1 only with two streams)
    const float sl2 = p.scale * 1.4426950408889634f;
    // the row's visible key positions form one interval [vlo, vhi]
    int64_t vlo = it.k0, vhi = it.k1 - 1;
    if (rv) {
      const int64_t qpos = F + qr / G;
      if (p.window) vlo = vlo > qpos - p.window + 1 ? vlo : qpos - p.window + 1;
      if (p.causal) vhi = vhi < qpos ? vhi : qpos;
    } else {
      vlo = 1;
      vhi = 0;
    }
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = stream; t < T; t += tstep) {
      const int sb = t & 1;
      bool w = ok && __all_sync(0xffffffffu, mbar_wait(&s_full[sb], (uint32_t)(t >> 1) & 1u, abort_flag));
      float s[32], mt = -INFINITY;
      if (w) {
        if (live) {
          fence_after();
          tmem_ld32(tmem + lrow + S_COL + sb * KT + 32 * half, s);
          fence_before();
        }
        mbar_arrive(&s_free[sb]);
      }
      if (w && live) {
        const int64_t kt = it.k0 + (int64_t)t * KT + 32 * half;
        const int64_t lo64 = vlo - kt, hi64 = vhi - kt;
        const int lo = lo64 < 0 ? 0 : (lo64 > 32 ? 32 : (int)lo64);
        const int hi = hi64 < -1 ? -1 : (hi64 > 31 ? 31 : (int)hi64);
        // the max of the raw scores (the scale is positive): the scale
        // folds into the exponent below
        if (!__all_sync(0xffffffffu, lo == 0 && hi == 31)) {
          // keys outside the row's visible range (a window, the causal
          // block, the end of the range); without them (the common case)
          // the half-tile needs no mask
#pragma unroll
          for (int j = 0; j < 32; ++j) s[j] = (j >= lo && j <= hi) ? s[j] : -INFINITY;
        }
        float m0 = fmaxf(s[0], s[1]), m1 = fmaxf(s[2], s[3]);
#pragma unroll
        for (int j = 4; j < 32; j += 4) {
          m0 = max3(m0, s[j], s[j + 1]);
          m1 = max3(m1, s[j + 2], s[j + 3]);
        }
        mt = fmaxf(m0, m1);
      }
      // both threads of a row agree on the tile max (a buffer per parity of
      // the stream's own tile count: a value is read before it is rewritten)
      float* xt = xch + ((dual ? t >> 1 : t) & 1) * 256;
      xt[half * 128 + r] = mt;
      if (!bar_and(pair_bar, 64, w)) {
        ok = false;
        break;
      }
      if (!live) {
        mbar_arrive(&p_full[sb]);
        continue;
      }
      mt = fmaxf(mt, xt[(half ^ 1) * 128 + r]) * sl2;  // the exp2 domain
      // lazy rescale: move the reference max only when it grows past 2^8
      const bool grow = mt > m_used + 8.f;
      const float m_new = grow ? mt : m_used;
      const float f = (grow && m_used != -INFINITY) ? exp2f(m_used - m_new) : 1.f;
      if (__any_sync(0xffffffffu, f != 1.f)) {
        // O must hold every earlier tile's product before it is scaled; the
        // later ones wait for this tile's P.  (Two streams: only the stream's
        // own products write its O region.)
        const int tp = t - tstep;
        if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[tp & 1], (uint32_t)(tp >> 1) & 1u, abort_flag))) {
          ok = false;  // the pair stops together at the next tile's barrier
          continue;
        }
        fence_after();
#pragma unroll 1
        for (int c = 64 * half; c < 64 * half + 64; c += 32) {
          float o[32];
          tmem_ld32(tmem + lrow + ocol + c, o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] *= f;
          tmem_st32(tmem + lrow + ocol + c, o);
        }
      }
      l *= f;
      m_used = m_new;
      uint32_t hi2[16], lo2[16];
      // while a row has seen no visible key its max is -inf and every score
      // is -inf too: exponentiate against 0 so that P = exp2(-inf) = 0
      const float mref = m_used == -INFINITY ? 0.f : m_used;
      const uint64_t k2 = f2pack(sl2, sl2), c2 = f2pack(-mref, -mref);
      uint64_t ls2 = f2pack(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 32; j += 2) hi2[j / 2] = p_pair(s[j], s[j + 1], k2, c2, ls2, lo2[j / 2]);
      const float2 ls = f2unpack(ls2);
      l += ls.x + ls.y;
      // One P tile (hi, lo) serves every tile: this thread's rows are free
      // once the product of its stream's previous tile is done.  (With two
      // streams each writes its own 64 rows; each product reads all 128, but
      // the other stream's rows only reach O rows of that product's region
      // that are never read.)
      if (t >= tstep) {
        const int tw = t - tstep;
        if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[tw & 1], (uint32_t)(tw >> 1) & 1u, abort_flag))) {
          ok = false;
          continue;
        }
      }
      uint8_t* ph = sP;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int cc = 4 * half + c;
        *reinterpret_cast<uint4*>(ph + swz(r, cc)) = make_uint4(hi2[4 * c], hi2[4 * c + 1], hi2[4 * c + 2], hi2[4 * c + 3]);
        *reinterpret_cast<uint4*>(ph + PBYTES + swz(r, cc)) = make_uint4(lo2[4 * c], lo2[4 * c + 1], lo2[4 * c + 2], lo2[4 * c + 3]);
      }
      fence_proxy_async();
      fence_before();
      mbar_arrive(&p_full[sb]);
    }
    if (!ok) {
      atomicOr(err, 8);
      *abort_flag = 1;
    }
    // ---- partial of this key range: (max in natural-log units, sum, -, -, O)
    if (!mbar_wait(o_done, 0, abort_flag) && !mbar_wait(o_done, 0, abort_flag)) atomicOr(err, 8);
    fence_after();
    float* xl = xch + 2 * 256;
    xl[half * 128 + r] = l;
    bar_and(pair_bar, 64, true);
    float lsum = xl[r] + xl[128 + r], we = 1.f, wo = 0.f;
    // two streams: the odd stream's rows go through idle V stages (every
    // copy has landed and every MMA has completed) to the even stream's
    float* xo = reinterpret_cast<float*>(sV + 2 * VBYTES) + (rv ? qr : 0) * (D + 4);
    if (dual) {
      if (stream == 1 && live) {
        if (rv && half == 0) *reinterpret_cast<float2*>(xo) = make_float2(m_used, lsum);
        // Stream 1 owns the odd tiles.  With a single tile it ran no product
        // and its TMEM O region still holds whatever an earlier kernel left
        // there, not necessarily finite numbers; its weight below is zero, and
        // zero times a NaN is a NaN, so it hands over zeros instead.
#pragma unroll 1
        for (int c = 64 * half; c < 64 * half + 64; c += 32) {
          float o[32];
          if (T > 1) {
            tmem_ld32(tmem + lrow + ocol + c, o);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = 0.f;
          }
          if (rv) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(xo + 4 + c + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
          }
        }
      }
      // warps of quarters q and q + 2 (and their partners) hold the same query rows
      bar_and(5 + (warp & 1), 128, true);
      if (stream == 0 && rv) {
        const float2 mo = *reinterpret_cast<const float2*>(xo);
        const float M = fmaxf(m_used, mo.x);
        we = m_used == -INFINITY ? 0.f : exp2f(m_used - M);
        wo = mo.x == -INFINITY ? 0.f : exp2f(mo.x - M);
        lsum = lsum * we + mo.y * wo;
        m_used = M;
      }
    }
    // the partial goes to global memory, or (clustered) to this CTA's idle K/V stages
    float* pr = p.cluster > 1 ? reinterpret_cast<float*>(sK) + (rv ? qr : 0) * (D + 4)
                              : part + ((int64_t)blockIdx.x * R + (rv ? qr : 0)) * (D + 4);
    if (stream == 0 && rv && half == 0) {
      *reinterpret_cast<float4*>(pr) =
          make_float4(m_used == -INFINITY ? -INFINITY : m_used * 0.6931471805599453f, lsum, 0.f, 0.f);
    }
#pragma unroll 1
    for (int c = 64 * half; c < 64 * half + 64 && live && stream == 0; c += 32) {
      float o[32];
      tmem_ld32(tmem + lrow + ocol + c, o);
      if (rv) {
        if (dual) {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = o[j] * we + xo[4 + c + j] * wo;
        }
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(pr + 4 + c + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
      }
    }
  }
  if (p.cluster > 1) {
    // ---- merge of the cluster's key ranges, in range order: rank q owns rows
    // [q R / S, (q+1) R / S); 32 threads per row, 4 output columns each
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();  // every range's partial is staged
    const int S = p.cluster, q = (int)cl.block_rank();
    const int r0 = q * R / S, r1 = (q + 1) * R / S;
    const int ln = lane;
    float* mine = reinterpret_cast<float*>(sK);
    for (int rr = r0 + warp; rr < r1; rr += THREADS / 32) {
      float mi = -INFINITY, li = 0.f;
      if (ln < S) {
        const float* pp = cl.map_shared_rank(mine, ln) + rr * (D + 4);
        mi = pp[0];
        li = pp[1];
      }
      const float M = warp_max(mi);
      const float wi = (ln < S && mi != -INFINITY) ? expf(mi - M) : 0.f;
      const float L = warp_sum(li * wi);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int sidx = 0; sidx < S; ++sidx) {
        const float ws = __shfl_sync(0xffffffffu, wi, sidx);
        if (ws == 0.f) continue;  // a range with no visible key holds no O
        const float4 v = *reinterpret_cast<const float4*>(cl.map_shared_rank(mine, sidx) + rr * (D + 4) + 4 + 4 * ln);
        acc.x += ws * v.x;
        acc.y += ws * v.y;
        acc.z += ws * v.z;
        acc.w += ws * v.w;
      }
      const int i = rr / G, g = rr % G, hq = it.kvh * G + g;
      const int64_t orow = (int64_t)it.sess * p.nrows + i;
      const float sc = (gates ? gates[orow * p.Hq + hq] : 1.f) / L;
      const __nv_bfloat162 a = __floats2bfloat162_rn(acc.x * sc, acc.y * sc);
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc.z * sc, acc.w * sc);
      uint2 raw;
      raw.x = *reinterpret_cast<const uint32_t*>(&a);
      raw.y = *reinterpret_cast<const uint32_t*>(&b2);
      *reinterpret_cast<uint2*>(reinterpret_cast<bf16*>(p.out) + (orow * p.Hq + hq) * D + 4 * ln) = raw;
    }
    cluster_sync_relaxed();  // no CTA leaves while a peer still reads its partial
  }
  fence_before();
  __syncthreads();
  if (warp == 9) {
    fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

int launch_attention_tc(const void* Q, const AttnItem* items, int n_items, SessTables tabs, AttnParams p, float* part,
                        int* err, cudaStream_t st) {
  const int R = p.nrows * (p.Hq / p.Hkv);
  if (p.d != D || R > 128 || !tabs.kvmaps) return 0;
  if (n_items <= 0) return 1;
  const size_t smem = (size_t)DATA_BYTES + 1024 + 256 + 3 * 1024;
  static bool attrs = false;
  if (!attrs) {
    cudaFuncSetAttribute(k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaFuncSetAttribute(k_attn_tc, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    attrs = true;
  }
  if (p.cluster > 1 && p.cluster <= kAttnMaxCluster && n_items % p.cluster == 0 && p.out) {
    if (launch_kc(k_attn_tc, n_items, THREADS, smem, st, p.cluster, (const bf16*)Q, items, tabs, p, part, err) ==
        cudaSuccess)
      return 2;
    cudaGetLastError();  // the cluster did not fit: the same ranges, merged by k_attn_combine
  }
  p.cluster = 1;
  launch_k(k_attn_tc, n_items, THREADS, smem, st, (const bf16*)Q, items, tabs, p, part, err);
  return 1;
}

}  // namespace dfl
