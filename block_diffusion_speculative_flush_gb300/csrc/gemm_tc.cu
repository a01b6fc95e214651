// Weight-streaming GEMM for the DFlash draft on sm_103a: tcgen05.mma with the
// accumulator in tensor memory, both operands brought into shared memory by
// TMA (cp.async.bulk.tensor) with 128-byte swizzle.
//
// Shape of the work.  The draft's products are skinny: a few to a few
// hundred activation rows (16 block rows per sequence, plus the pending
// context rows) against weight matrices of 10^7..10^9 elements, so the
// weight stream from HBM is the cost.  The MMA's 128-row side therefore
// takes 128 weight rows (output features) and its N side takes the
// activation rows ("swap AB"): D[feature][row] = W[feature][:] . X[row][:].
// One CTA owns one 128-feature tile, one token tile of BN rows and one
// contiguous range of K; when K is split, the CTA that finishes a tile last
// sums the partials in split order (no spin, no atomics on data), so results
// are deterministic and a row's value never depends on how many rows share
// the call.
//
// Roles in a 128-thread CTA: thread 0 issues TMA loads into a STAGES-deep
// ring, thread 32 issues the MMAs (4 x K=16 per 64-wide stage) and commits
// each stage back to the producer, then all four warps read TMEM (warp w owns
// lanes 32w..32w+31) and store.  Every wait is bounded: a wait that runs past
// its limit sets an error bit and the CTA drains and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <string>

#include "common.cuh"
#include "gemm_tc.h"
#include "launch.h"

namespace dfl {

namespace {

using bf16 = __nv_bfloat16;

thread_local std::string g_tc_err;

constexpr int BM = 128;  // weight rows per tile (MMA M)
constexpr int BK = 64;   // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct TcParams {
  void* Y;         // fp32 output, bf16 residual stream, or bf16 SwiGLU product
  int64_t ldy;
  int M, N;        // activation rows; output features
  int mode;        // TcMode
  int n_tiles, splits, kb_total;
  float* ws;       // split partials [tile][split][BN][BM]
  int* counters;   // [tile] arrivals, returned to zero by the last CTA
  int* err;
};

constexpr int kMaxSplits = 16;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase of `parity` to complete; false if the CTA was told to
// abort or the wait ran past its limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte
// swizzle layout: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address (16-byte units)
  d |= (uint64_t)1 << 16;                    // leading byte offset (unused when swizzled)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;                    // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (both K-major), fp32 D.
template <int BN>
__host__ __device__ constexpr uint32_t idesc_bf16() {
  return (1u << 4)                          // D format fp32
         | (1u << 7)                        // A format bf16
         | (1u << 10)                       // B format bf16
         | ((uint32_t)(BN >> 3) << 17)      // N
         | ((uint32_t)(BM >> 4) << 24);     // M
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float* v);

template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <int BN>
__host__ __device__ constexpr int stages_for() {
  return BN <= 16 ? 6 : BN <= 32 ? 5 : BN <= 64 ? 4 : BN <= 128 ? 3 : 4;
}
template <int BN>
__host__ __device__ constexpr int tmem_cols() {
  return BN < 32 ? 32 : BN;
}
template <int BN>
__host__ __device__ constexpr size_t smem_bytes() {
  return (size_t)stages_for<BN>() * (BM * BK * 2 + BN * BK * 2) + 1024 + 256;
}

// SWI: the 128-row weight tile is 64 gate rows then the 64 matching up rows
// (two TMA boxes from two matrices), and the epilogue writes silu(g) * u.
template <int BN, bool SWI>
__global__ void __launch_bounds__(128, 1) k_gemm_tc(const __grid_constant__ CUtensorMap tmW,
                                                    const __grid_constant__ CUtensorMap tmW2,
                                                    const __grid_constant__ CUtensorMap tmX, TcParams p) {
  constexpr int STAGES = stages_for<BN>();
  constexpr int A_BYTES = BM * BK * 2;
  constexpr int B_BYTES = BN * BK * 2;
  constexpr uint32_t TX = A_BYTES + B_BYTES;
  constexpr int CH = BN < 32 ? BN : 32;
  static_assert((size_t)BN * BM * 4 <= (size_t)STAGES * (A_BYTES + B_BYTES), "epilogue tile must fit the pipeline");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* full = (uint64_t*)(sB + STAGES * B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* done = empty + STAGES;
  uint32_t* tmem_slot = (uint32_t*)(done + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  int* last_flag = (int*)(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int w = blockIdx.x;
  const int split = w % p.splits;
  w /= p.splits;
  const int n_tile = w % p.n_tiles;
  const int m_tile = w / p.n_tiles;
  const int kb0 = (int)((int64_t)split * p.kb_total / p.splits);
  const int kb1 = (int)((int64_t)(split + 1) * p.kb_total / p.splits);
  const int nkb = kb1 - kb0;

  pdl_trigger();  // the next kernel may be scheduled as this one's CTAs retire
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmW) : "memory");
    if (SWI) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmW2) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tmX) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"((uint32_t)tmem_cols<BN>())
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {
    // ---- TMA producer ----
    uint64_t pol_w, pol_x;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_x));
    auto load_w = [&](int i, int s) {
      if (SWI) {
        tma_load_2d(sA + s * A_BYTES, &tmW, &full[s], (kb0 + i) * BK, m_tile * (BM / 2), pol_w);
        tma_load_2d(sA + s * A_BYTES + A_BYTES / 2, &tmW2, &full[s], (kb0 + i) * BK, m_tile * (BM / 2), pol_w);
      } else {
        tma_load_2d(sA + s * A_BYTES, &tmW, &full[s], (kb0 + i) * BK, m_tile * BM, pol_w);
      }
    };
    // Weights do not depend on the previous kernel: the first stages of them
    // are requested before waiting for it, so the weight stream starts while
    // the previous kernel drains.
    const int pre = nkb < STAGES ? nkb : STAGES;
    for (int i = 0; i < pre; ++i) {
      mbar_expect_tx(&full[i], TX);
      load_w(i, i);
    }
    pdl_wait();
    for (int i = 0; i < pre; ++i) tma_load_2d(sB + i * B_BYTES, &tmX, &full[i], (kb0 + i) * BK, n_tile * BN, pol_x);
    int issued = pre;
    for (int i = pre; i < nkb; ++i) {
      const int s = i % STAGES;
      const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
      if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag)) {
        atomicOr(p.err, 4);
        *abort_flag = 1;
        break;
      }
      mbar_expect_tx(&full[s], TX);
      load_w(i, s);
      tma_load_2d(sB + s * B_BYTES, &tmX, &full[s], (kb0 + i) * BK, n_tile * BN, pol_x);
      ++issued;
    }
    if (*abort_flag) {
      // let this CTA's own copies land before its shared memory is released
      for (int i = max(0, issued - STAGES); i < issued; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&full[s], ph) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (threadIdx.x == 32) {
    // ---- MMA issuer ----
    constexpr uint32_t idesc = idesc_bf16<BN>();
    for (int i = 0; i < nkb; ++i) {
      const int s = i % STAGES;
      const uint32_t ph = (uint32_t)(i / STAGES) & 1u;
      if (!mbar_wait(&full[s], ph, abort_flag)) {
        atomicOr(p.err, 4);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA + s * A_BYTES), b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
      for (int k = 0; k < BK / 16; ++k)
        umma_bf16(tmem, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), idesc, (i | k) != 0);
      umma_commit(&empty[s]);
    }
    umma_commit(done);  // arrives once every MMA issued above has completed
  }
  __syncwarp();
  pdl_wait();  // the epilogue reads (residual) and writes memory the previous kernels use

  // ---- epilogue: TMEM -> registers -> global ----
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(done, 0)) {
    if (globaltimer_ns() - t0 > 2 * kWaitLimitNs) {
      atomicOr(p.err, 4);
      break;
    }
  }
  tc_fence_after();
  const int row = warp * 32 + lane;   // TMEM lane = weight row within the tile
  const int tok0 = n_tile * BN;
  const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
  // The pipeline buffers are idle once every MMA has completed: the final
  // tile is staged there as S[col][row] (fp32) for a coalesced store.
  float* S = reinterpret_cast<float*>(smem);
  bool store = true;
  if (p.splits == 1) {
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += CH) {
      float v[CH];
      tmem_ld<CH>(taddr + c0, v);
#pragma unroll
      for (int j = 0; j < CH; ++j) S[(c0 + j) * BM + row] = v[j];
    }
  } else {
    const int tile = m_tile * p.n_tiles + n_tile;
    float* mine = p.ws + ((int64_t)(tile * p.splits + split) * BN) * BM;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += CH) {
      float v[CH];
      tmem_ld<CH>(taddr + c0, v);
#pragma unroll
      for (int j = 0; j < CH; ++j) __stcg(mine + (int64_t)(c0 + j) * BM + row, v[j]);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *last_flag = atomicAdd(&p.counters[tile], 1) == p.splits - 1;
    __syncthreads();
    store = *last_flag != 0;
    if (store) {
      // the last CTA of the tile sums the partials in split order; all loads
      // of a column group are issued before the adds
      __threadfence();
      const float* base = p.ws + (int64_t)tile * p.splits * BN * BM + row;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 4) {
        float v[kMaxSplits][4];
#pragma unroll
        for (int sp = 0; sp < kMaxSplits; ++sp)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            v[sp][j] = sp < p.splits ? __ldcg(base + ((int64_t)sp * BN + c0 + j) * BM) : 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float acc = 0.f;
#pragma unroll
          for (int sp = 0; sp < kMaxSplits; ++sp)
            if (sp < p.splits) acc += v[sp][j];
          S[(c0 + j) * BM + row] = acc;
        }
      }
      if (threadIdx.x == 0) p.counters[tile] = 0;
    }
  }
  __syncthreads();
  if (store) {
    if (SWI) {
      // rows 0..63 of the tile are gate rows, 64..127 the matching up rows
      bf16* out = reinterpret_cast<bf16*>(p.Y);
      for (int e = threadIdx.x; e < BN * (BM / 2); e += blockDim.x) {
        const int c = e / (BM / 2), f = e % (BM / 2);
        const int t = tok0 + c, feat = m_tile * (BM / 2) + f;
        if (t < p.M && feat < p.N) {
          const float g = S[c * BM + f], u = S[c * BM + BM / 2 + f];
          out[(int64_t)t * p.ldy + feat] = __float2bfloat16_rn(g / (1.f + expf(-g)) * u);
        }
      }
    } else if (p.mode == kResidBf16) {
      bf16* h = reinterpret_cast<bf16*>(p.Y);
      for (int e = threadIdx.x; e < BN * BM; e += blockDim.x) {
        const int c = e / BM, f = e % BM;
        const int t = tok0 + c, feat = m_tile * BM + f;
        if (t < p.M && feat < p.N) {
          bf16* hp = h + (int64_t)t * p.ldy + feat;
          *hp = __float2bfloat16_rn(__bfloat162float(*hp) + S[c * BM + f]);
        }
      }
    } else {
      float* Y = reinterpret_cast<float*>(p.Y);
      for (int e = threadIdx.x; e < BN * BM; e += blockDim.x) {
        const int c = e / BM, f = e % BM;
        const int t = tok0 + c, feat = m_tile * BM + f;
        if (t < p.M && feat < p.N) Y[(int64_t)t * p.ldy + feat] = S[c * BM + f];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)tmem_cols<BN>())
                 : "memory");
  }
}

}  // namespace

struct TcContext {
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  int num_sms = 0;
  float* ws = nullptr;
  size_t ws_cap = 0;
  int* counters = nullptr;
  size_t cnt_cap = 0;
  int* err = nullptr;
  bool attr_set[10] = {};
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

void tc_destroy(TcContext* c) {
  if (!c) return;
  cudaFree(c->ws);
  cudaFree(c->counters);
  delete c;
}

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

template <int BN, bool SWI>
static int launch_bn(TcContext* c, const CUtensorMap& mw, const CUtensorMap& mw2, const CUtensorMap& mx,
                     const TcParams& p, int grid, cudaStream_t st, int slot) {
  const size_t smem = smem_bytes<BN>();
  if (!c->attr_set[slot]) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_tc<BN, SWI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return tc_fail("smem attribute", e);
    c->attr_set[slot] = true;
  }
  const cudaError_t e = launch_k(k_gemm_tc<BN, SWI>, grid, 128, smem, st, mw, mw2, mx, p);
  if (e != cudaSuccess) return tc_fail("k_gemm_tc launch", e);
  return 0;
}

int tc_gemm(TcContext* c, const void* X, int64_t ldx, const void* W, const void* W2, int64_t ldw, void* Y,
            int64_t ldy, int M, int N, int K, int mode, cudaStream_t st) {
  if (M <= 0 || N <= 0) return 0;
  const bool swi = mode == kSwigluBf16;
  if (K % BK || ldx % 8 || ldw % 8 || ((uintptr_t)X & 15) || ((uintptr_t)W & 15) || (swi && ((uintptr_t)W2 & 15)))
    return tc_fail("tc_gemm: K must be a multiple of 64, strides multiples of 8, operands 16-byte aligned");
  if (mode < kF32 || mode > kSwigluBf16) return tc_fail("tc_gemm: unknown mode");
  const int BN = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
  const int rows_per_tile = swi ? BM / 2 : BM;
  const int m_tiles = (N + rows_per_tile - 1) / rows_per_tile, n_tiles = (M + BN - 1) / BN, kb_total = K / BK;
  // Split K so that the weight tiles fill one wave of resident CTAs (two per
  // SM up to BN = 128, one at 256); the split depends on N and K only.
  const int slots = c->num_sms * (BN <= 128 ? 2 : 1);
  int splits = slots / m_tiles;
  splits = std::max(1, std::min({splits, kMaxSplits, std::max(1, kb_total / 2)}));
  const int tiles = m_tiles * n_tiles;
  if (splits > 1) {
    const size_t need = (size_t)tiles * splits * BN * BM * sizeof(float);
    if (need > c->ws_cap) {
      cudaError_t e = cudaStreamSynchronize(st);
      if (e == cudaSuccess) e = cudaFree(c->ws);
      c->ws = nullptr;
      c->ws_cap = 0;
      if (e == cudaSuccess) e = cudaMalloc(&c->ws, need + need / 4);
      if (e != cudaSuccess) return tc_fail("split workspace", e);
      c->ws_cap = need + need / 4;
    }
    if ((size_t)tiles > c->cnt_cap) {
      cudaError_t e = cudaStreamSynchronize(st);
      if (e == cudaSuccess) e = cudaFree(c->counters);
      c->counters = nullptr;
      c->cnt_cap = 0;
      const size_t want = (size_t)tiles * 2;
      if (e == cudaSuccess) e = cudaMalloc(&c->counters, want * sizeof(int));
      if (e == cudaSuccess) e = cudaMemsetAsync(c->counters, 0, want * sizeof(int), st);
      if (e != cudaSuccess) return tc_fail("split counters", e);
      c->cnt_cap = want;
    }
  }
  CUtensorMap mw, mw2, mx;
  if (encode_2d(c, &mw, W, (uint64_t)K, (uint64_t)N, ldw, (uint32_t)rows_per_tile)) return -1;
  if (swi) {
    if (encode_2d(c, &mw2, W2, (uint64_t)K, (uint64_t)N, ldw, (uint32_t)rows_per_tile)) return -1;
  } else {
    mw2 = mw;
  }
  if (encode_2d(c, &mx, X, (uint64_t)K, (uint64_t)M, ldx, (uint32_t)BN)) return -1;
  TcParams p{Y, ldy, M, N, mode, n_tiles, splits, kb_total, c->ws, c->counters, c->err};
  const int grid = tiles * splits;
  if (swi) {
    switch (BN) {
      case 16: return launch_bn<16, true>(c, mw, mw2, mx, p, grid, st, 5);
      case 32: return launch_bn<32, true>(c, mw, mw2, mx, p, grid, st, 6);
      case 64: return launch_bn<64, true>(c, mw, mw2, mx, p, grid, st, 7);
      case 128: return launch_bn<128, true>(c, mw, mw2, mx, p, grid, st, 8);
      default: return launch_bn<256, true>(c, mw, mw2, mx, p, grid, st, 9);
    }
  }
  switch (BN) {
    case 16: return launch_bn<16, false>(c, mw, mw2, mx, p, grid, st, 0);
    case 32: return launch_bn<32, false>(c, mw, mw2, mx, p, grid, st, 1);
    case 64: return launch_bn<64, false>(c, mw, mw2, mx, p, grid, st, 2);
    case 128: return launch_bn<128, false>(c, mw, mw2, mx, p, grid, st, 3);
    default: return launch_bn<256, false>(c, mw, mw2, mx, p, grid, st, 4);
  }
}

}  // namespace dfl
