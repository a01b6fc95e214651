// Host runtime behind the C ABI of include/dflash.h: model validation, the
// drafter session state machine, workspace management and the launch
// sequence of one batched flush / propose / verify.
//
// The session cursors follow ollama's mlxrunner/dflash.go (committed,
// takePending, commitBlock, flush, propose): ctxOffset F is the slot after
// the last feature row written; P rows are held past it; F + P is the slot
// after the last reported token.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "dflash.h"
#include "gemm_tc.h"
#include "kernels.h"

using namespace dfl;

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define CU_TRY(expr)                                                                              \
  do {                                                                                            \
    cudaError_t e_ = (expr);                                                                      \
    if (e_ != cudaSuccess)                                                                        \
      return fail(e_ == cudaErrorMemoryAllocation ? DFLASH_ERR_OOM : DFLASH_ERR_CUDA, "%s: %s (%s:%d)", #expr, \
                  cudaGetErrorString(e_), __FILE__, __LINE__);                                    \
  } while (0)

#define ST_TRY(expr)        \
  do {                      \
    int s_ = (expr);        \
    if (s_ != DFLASH_OK) return s_; \
  } while (0)

inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// A device buffer that only grows.  Growing waits for the stream so that no
// queued kernel still reads the old allocation.
struct Buf {
  void* p = nullptr;
  size_t cap = 0;
  int ensure(size_t bytes, cudaStream_t st) {
    if (bytes <= cap) return DFLASH_OK;
    if (p) {
      CU_TRY(cudaStreamSynchronize(st));
      CU_TRY(cudaFree(p));
      p = nullptr;
      cap = 0;
    }
    size_t want = std::max<size_t>(bytes, 4096);
    want = (size_t)align_up((int64_t)want + want / 4, 256);
    CU_TRY(cudaMalloc(&p, want));
    CU_TRY(cudaMemsetAsync(p, 0, want, st));
    cap = want;
    return DFLASH_OK;
  }
  void release() {
    if (p) cudaFree(p);
    p = nullptr;
    cap = 0;
  }
  template <typename T> T* as() const { return (T*)p; }
};

// Packs the small per-call tables into one host block.  Up to
// kTableParamMax bytes it travels as the parameter of a one-CTA kernel in the
// launch chain (launch_table_write); a larger block is copied from a ring of
// pinned host slots guarded by events, so that a slot is never rewritten
// while its copy is still queued.
struct TablePack {
  std::vector<char> host;
  size_t add(const void* src, size_t bytes) {
    const size_t off = (size_t)align_up((int64_t)host.size(), 16);
    host.resize(off + bytes);
    if (bytes) memcpy(host.data() + off, src, bytes);
    return off;
  }
  template <typename T> size_t add(const std::vector<T>& v) { return add(v.data(), v.size() * sizeof(T)); }
};

struct HostRing {
  static constexpr int kSlots = 8;
  char* slot[kSlots] = {};
  size_t cap[kSlots] = {};
  cudaEvent_t ev[kSlots] = {};
  int next = 0;
  int upload(const TablePack& t, Buf& dev, cudaStream_t st) {
    const size_t bytes = std::max<size_t>(t.host.size(), 16);
    ST_TRY(dev.ensure(bytes, st));
    if (t.host.size() <= (size_t)kTableParamMax) {
      // small tables go through the launch chain as a kernel parameter
      if (launch_table_write(dev.p, t.host.data(), t.host.size(), st)) return fail(DFLASH_ERR_CUDA, "table write launch");
      return DFLASH_OK;
    }
    const int i = next;
    next = (next + 1) % kSlots;
    if (!ev[i]) CU_TRY(cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming));
    CU_TRY(cudaEventSynchronize(ev[i]));
    if (cap[i] < bytes) {
      if (slot[i]) cudaFreeHost(slot[i]);
      slot[i] = nullptr;
      const size_t want = (size_t)align_up((int64_t)bytes * 2, 4096);
      CU_TRY(cudaMallocHost((void**)&slot[i], want));
      cap[i] = want;
    }
    memcpy(slot[i], t.host.data(), t.host.size());
    CU_TRY(cudaMemcpyAsync(dev.p, slot[i], t.host.size(), cudaMemcpyHostToDevice, st));
    CU_TRY(cudaEventRecord(ev[i], st));
    return DFLASH_OK;
  }
  void release() {
    for (int i = 0; i < kSlots; ++i) {
      if (ev[i]) {
        cudaEventSynchronize(ev[i]);
        cudaEventDestroy(ev[i]);
      }
      if (slot[i]) cudaFreeHost(slot[i]);
      ev[i] = nullptr;
      slot[i] = nullptr;
    }
  }
};

struct LayerW {
  const void *in_norm, *w_qkv, *q_norm, *k_norm, *w_g, *w_o, *post_norm, *w_gate, *w_up, *w_down;
  void* w_qkvg = nullptr;  // owned: [w_qkv ; w_g] rows, one product for q, k, v and the gate
  const void *conv_norm = nullptr, *w_dc = nullptr;  // DFlash2's dynamic convolution
};

}  // namespace

struct dflash_model {
  dflash_config cfg{};
  DT dt = DT::F32;
  size_t esz = 4;
  const void *aux_norms, *w_fc, *hidden_norm, *final_norm, *embed, *unembed;
  const void *sel_prev = nullptr, *sel_next = nullptr;  // DFlash2's selector tables
  bool dflash2 = false;
  // context-only forwards of many rows: every layer's K/V rows of the fused
  // projection packed into one matrix [L][2 Hkv d][H] (owned), and device
  // tables of the layers' input-norm and k-norm gains [2][L]
  void* w_kv = nullptr;
  const void** d_gains = nullptr;
  std::vector<LayerW> layers;
  int qkv_rows = 0;   // (Hq + 2 Hkv) d
  int qkv_cols = 0;   // qkv_rows (+ Hq for the gate)
  int num_sms = 0;
  int64_t rope_len = 0;  // positions the RoPE table (rope) holds
  bool use_tc = false;
  int32_t* d_err = nullptr;
  TcContext* tc = nullptr;
  // measurement
  bool timing = false;
  int64_t launches = 0;
  struct Rec { cudaEvent_t e0, e1; int cls; double bytes, flops; };
  std::vector<Rec> recs;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev_pool;
  size_t ev_used = 0;
  // workspace
  Buf tables, u, fcout, c, h, x, qkv, rope, Q, G, O, tmp, y, a, z, logits, spart, apart, vstat, vpart, vbonus, cutbuf,
      vpen, vpen_tab, d2part, d2cand, xall, kvall;
  HostRing ring;
};

struct dflash_session {
  dflash_model* m = nullptr;
  cudaStream_t stream = nullptr;
  int64_t F = 0;      // ctxOffset
  int32_t P = 0;      // pendingCount
  bool block_outstanding = false;
  int64_t max_ctx = 0, cap = 0;
  void* kv = nullptr;       // [L][2][Hkv][cap][d]
  void* pending = nullptr;  // [PENDING_FLUSH_TOKENS][K*H_t]
  float* plogits = nullptr; // [B_s-1][V] logits of the last proposal
  float* plse = nullptr;    // [B_s-1]
  int32_t* ptok = nullptr;  // [B_s-1]
  uint64_t* pcut = nullptr; // [B_s-1] truncation cut of each proposal row (when last_trunc)
  long long* d_accepted = nullptr;
  CUtensorMap* d_maps = nullptr;  // {K planes, V^T planes} for the tensor-core attention, or NULL
  bool has_prop = false;
  int last_n = 0;
  float last_T = 0.f;
  Trunc trunc{0, 1.f, 0.f, 0};  // the sampler's truncation (top_k 0: full distributions)
  bool last_trunc = false;      // the last proposal was drawn from a truncated distribution
  int64_t rounds = 0, proposed = 0, flushes = 0, flushed_rows = 0;
  int device = 0;               // the CUDA device that was current at dflash_open
  Penalty pen{1.f, 0.f, 0.f, 0, nullptr};  // the sampler's penalties (hist: the session's copy)
  int32_t* d_hist = nullptr;    // [kMaxPenaltyHistory] committed history for the penalties
  int32_t* pcand_ids = nullptr;  // DFlash2: [n][sel_candidates] candidates of the last proposal
  float* pcand_probs = nullptr;  // DFlash2: their probabilities (one-hot on the token at T = 0)
};

namespace {
bool penalties_on(const Penalty& p) { return p.repeat != 1.f || p.presence != 0.f || p.frequency != 0.f; }
}  // namespace

namespace {

// ---------------------------------------------------------------------------
// measurement: CUDA events around instrumented launches
// ---------------------------------------------------------------------------
enum TimeClass { kGemmTc = 0, kGemmSimt, kAttention, kSample, kVerify, kClasses };
const char* const kClassNames[kClasses] = {"gemm_tc", "gemm_simt", "attention", "sample", "verify"};

struct Timed {
  dflash_model* m;
  cudaStream_t st;
  size_t idx = (size_t)-1;
  Timed(dflash_model* m_, int cls, double bytes, double flops, cudaStream_t st_) : m(m_), st(st_) {
    if (!m->timing) return;
    if (m->ev_used == m->ev_pool.size()) {
      cudaEvent_t a = nullptr, b = nullptr;
      if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) return;
      m->ev_pool.push_back({a, b});
    }
    auto ev = m->ev_pool[m->ev_used++];
    idx = m->recs.size();
    m->recs.push_back(dflash_model::Rec{ev.first, ev.second, cls, bytes, flops});
    cudaEventRecord(ev.first, st);
  }
  ~Timed() {
    if (idx != (size_t)-1) cudaEventRecord(m->recs[idx].e1, st);
  }
};

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------
int check_config(const dflash_config& c) {
  if (c.dtype != DFLASH_DTYPE_F32 && c.dtype != DFLASH_DTYPE_BF16) return fail(DFLASH_ERR_INVALID_ARG, "dtype %d", c.dtype);
  if (c.n_taps < 1 || c.target_hidden < 1 || c.hidden < 1 || c.n_layers < 1 || c.n_q_heads < 1 || c.n_kv_heads < 1 ||
      c.intermediate < 1 || c.vocab < 2)
    return fail(DFLASH_ERR_SHAPE, "non-positive dimension in config");
  if (c.block_size < 2 || c.block_size > 512) return fail(DFLASH_ERR_SHAPE, "block_size %d outside 2..512", c.block_size);
  if (c.n_taps > kMaxTaps) return fail(DFLASH_ERR_SHAPE, "n_taps %d above %d", c.n_taps, kMaxTaps);
  if (c.window != 0 && (c.window < 2 || c.window > (1 << 20)))
    return fail(DFLASH_ERR_SHAPE, "window %d outside 2..2^20", c.window);
  if (c.head_dim != 64 && c.head_dim != 128) return fail(DFLASH_ERR_SHAPE, "head_dim %d (64 or 128 supported)", c.head_dim);
  if (c.n_q_heads % c.n_kv_heads) return fail(DFLASH_ERR_SHAPE, "n_q_heads %d not a multiple of n_kv_heads %d", c.n_q_heads, c.n_kv_heads);
  if (c.n_q_heads / c.n_kv_heads * c.block_size > 512)
    return fail(DFLASH_ERR_SHAPE, "query rows per KV head (group x block) above 512");
  if (c.mask_token < 0 || c.mask_token >= c.vocab) return fail(DFLASH_ERR_SHAPE, "mask_token %d outside vocab", c.mask_token);
  if (c.causal_block != 0 && c.causal_block != 1) return fail(DFLASH_ERR_INVALID_ARG, "causal_block must be 0 or 1");
  if (c.gated_attention != 0 && c.gated_attention != 1) return fail(DFLASH_ERR_INVALID_ARG, "gated_attention must be 0 or 1");
  if (!(c.rope_theta > 1.f) || !(c.rms_eps >= 0.f)) return fail(DFLASH_ERR_INVALID_ARG, "rope_theta / rms_eps");
  if (c.variant != DFLASH_VARIANT_DFLASH && c.variant != DFLASH_VARIANT_DFLASH2)
    return fail(DFLASH_ERR_INVALID_ARG, "variant %d", c.variant);
  if (c.variant == DFLASH_VARIANT_DFLASH2) {
    if (c.conv_taps < 1 || c.conv_taps > kMaxConvTaps) return fail(DFLASH_ERR_SHAPE, "conv_taps %d outside 1..%d", c.conv_taps, kMaxConvTaps);
    if (c.sel_rank < 1 || c.sel_rank > 256) return fail(DFLASH_ERR_SHAPE, "sel_rank %d outside 1..256", c.sel_rank);
    if (c.sel_candidates < 1 || c.sel_candidates > kMaxCandidates || c.sel_candidates > c.vocab)
      return fail(DFLASH_ERR_SHAPE, "sel_candidates %d outside 1..%d (and at most vocab)", c.sel_candidates, kMaxCandidates);
    if (c.hidden % c.n_q_heads) return fail(DFLASH_ERR_SHAPE, "hidden %d not a multiple of n_q_heads", c.hidden);
  }
  if (c.dtype == DFLASH_DTYPE_BF16) {
    const int w[] = {c.target_hidden, c.hidden, c.intermediate, c.n_q_heads * c.head_dim};
    for (int x : w)
      if (x % 64) return fail(DFLASH_ERR_SHAPE, "bf16 widths must be multiples of 64 (got %d)", x);
  }
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------
// matrix products: Y[M][N] (fp32) = X[M][K] . W[N][K]^T
// ---------------------------------------------------------------------------
int gemm(dflash_model* m, const void* X, int64_t ldx, const void* W, int64_t ldw, float* Y, int64_t ldy, int M, int N,
         int K, cudaStream_t st, bool late_trigger = false) {
  if (M <= 0) return DFLASH_OK;
  const double bytes = (double)N * K * m->esz + (double)M * K * m->esz + (double)M * N * 4;
  Timed tm(m, m->use_tc ? kGemmTc : kGemmSimt, bytes, 2.0 * M * N * K, st);
  m->launches++;
  if (m->use_tc) {
    const int rc = tc_gemm(m->tc, X, ldx, W, nullptr, ldw, Y, ldy, M, N, K, kF32, st, nullptr, 0, nullptr,
                           late_trigger ? 1 : 0);
    if (rc) return fail(DFLASH_ERR_CUDA, "tcgen05 GEMM: %s", tc_last_error());
  } else {
    launch_gemm_simt(m->dt, X, ldx, W, ldw, Y, ldy, M, N, K, st);
  }
  return DFLASH_OK;
}

// Y rows [j*seg_rows, (j+1)*seg_rows) into yseg[j] (device table); tensor-core path only.
int gemm_rows(dflash_model* m, const void* X, int64_t ldx, const void* W, int64_t ldw, void* const* yseg, int seg_rows,
              int64_t ldy, int M, int N, int K, cudaStream_t st) {
  if (M <= 0) return DFLASH_OK;
  const double bytes = (double)N * K * m->esz + (double)M * K * m->esz + (double)M * N * 4;
  Timed tm(m, kGemmTc, bytes, 2.0 * M * N * K, st);
  m->launches++;
  if (tc_gemm(m->tc, X, ldx, W, nullptr, ldw, nullptr, ldy, M, N, K, kF32, st, yseg, seg_rows))
    return fail(DFLASH_ERR_CUDA, "tcgen05 GEMM: %s", tc_last_error());
  return DFLASH_OK;
}

// h[M][N] = storage(h + X W^T): the residual add after the attention output
// and after the MLP down projection.
int gemm_resid(dflash_model* m, const void* X, int64_t ldx, const void* W, void* h, float* tmp, int M, int N, int K,
               cudaStream_t st) {
  if (M <= 0) return DFLASH_OK;
  if (!m->use_tc) {
    ST_TRY(gemm(m, X, ldx, W, K, tmp, N, M, N, K, st));
    launch_residual(m->dt, h, tmp, N, M, N, st);
    m->launches++;
    return DFLASH_OK;
  }
  const double bytes = (double)N * K * 2 + (double)M * K * 2 + (double)M * N * 4;
  Timed tm(m, kGemmTc, bytes, 2.0 * M * N * K, st);
  m->launches++;
  // tmp ([M][N] fp32, idle on this path) carries the split sums of many-row calls
  if (tc_gemm(m->tc, X, ldx, W, nullptr, K, h, N, M, N, K, kResidBf16, st, nullptr, 0, tmp))
    return fail(DFLASH_ERR_CUDA, "tcgen05 GEMM: %s", tc_last_error());
  return DFLASH_OK;
}

// a[M][I] = storage(silu(Y Wg^T) * (Y Wu^T)).
int gemm_swiglu(dflash_model* m, const void* Y, const void* Wg, const void* Wu, void* a, float* tmp, int M, int I,
                int H, cudaStream_t st) {
  if (M <= 0) return DFLASH_OK;
  if (!m->use_tc) {
    ST_TRY(gemm(m, Y, H, Wg, H, tmp, 2 * I, M, I, H, st));
    ST_TRY(gemm(m, Y, H, Wu, H, tmp + I, 2 * I, M, I, H, st));
    launch_swiglu(m->dt, tmp, 2 * I, M, I, I, a, st);
    m->launches++;
    return DFLASH_OK;
  }
  const double bytes = 2.0 * I * H * 2 + (double)M * H * 2 + (double)M * I * 2;
  Timed tm(m, kGemmTc, bytes, 4.0 * M * I * H, st);
  m->launches++;
  if (tc_gemm(m->tc, Y, H, Wg, Wu, H, a, I, M, I, H, kSwigluBf16, st))
    return fail(DFLASH_ERR_CUDA, "tcgen05 GEMM: %s", tc_last_error());
  return DFLASH_OK;
}

int launch_check(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(DFLASH_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------
// one batched forward: context rows (flush) and optionally block rows
// ---------------------------------------------------------------------------
struct CtxRow {
  const void* tap[kMaxTaps];  // the row's n_taps target hidden states
  int32_t sess;               // compact session index
  int64_t pos;                // slot
};

struct Forward {
  std::vector<dflash_session*> sess;  // compact sessions
  std::vector<CtxRow> ctx;
  // block part
  int n = 0;                          // block rows are n + 1 per session (0: flush only)
  const int32_t* current = nullptr;   // device [batch]
  std::vector<int32_t> sess_map;      // compact -> caller index
  float temperature = 0.f;
  uint64_t seed = 0;
  uint64_t rnd = 0;
  int32_t* out_tokens = nullptr;
  float* out_q = nullptr;
  float* out_logits = nullptr;
};

int run_forward(dflash_model* m, Forward& fw, cudaStream_t st) {
  const dflash_config& c = m->cfg;
  const int Bc = (int)fw.sess.size();
  const int Mc = (int)fw.ctx.size();
  const bool block = fw.n > 0;
  const int nrows = fw.n + 1;
  const int Mb = block ? Bc * nrows : 0;
  const int M = Mc + Mb;
  if (M == 0) return DFLASH_OK;
  const int H = c.hidden, d = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads, I = c.intermediate, V = c.vocab;
  const int KHt = c.n_taps * c.target_hidden;
  const size_t es = m->esz;

  // ---- per-call tables ---------------------------------------------------
  TablePack tp;
  std::vector<const void*> rowsrc((size_t)Mc * c.n_taps);  // [Mc][K]: tap k of context row r
  std::vector<RowMeta> meta(M);
  for (int r = 0; r < Mc; ++r) {
    for (int k = 0; k < c.n_taps; ++k) rowsrc[(size_t)r * c.n_taps + k] = fw.ctx[r].tap[k];
    meta[r] = RowMeta{fw.ctx[r].sess, -1, fw.ctx[r].pos};
  }
  std::vector<void*> kvb(Bc);
  std::vector<const CUtensorMap*> mapv(Bc);
  std::vector<int64_t> capv(Bc), front(Bc), fresh(Bc);
  std::vector<int32_t> seqv(Bc);
  bool have_maps = true;
  for (int j = 0; j < Bc; ++j) {
    mapv[j] = fw.sess[j]->d_maps;
    have_maps = have_maps && mapv[j] != nullptr;
    kvb[j] = fw.sess[j]->kv;
    capv[j] = fw.sess[j]->cap;
    front[j] = fw.sess[j]->F;
    fresh[j] = fw.sess[j]->F;  // the block's rows start at F
    seqv[j] = block ? fw.sess_map[j] : j;
  }
  for (int r = 0; r < Mc; ++r) fresh[fw.ctx[r].sess] = std::min(fresh[fw.ctx[r].sess], fw.ctx[r].pos);
  for (int j = 0; j < Bc && block; ++j)
    for (int i = 0; i < nrows; ++i) meta[Mc + j * nrows + i] = RowMeta{j, j * nrows + i, fw.sess[j]->F + i};
  // attention work items: split every (session, KV head) key range in chunks
  std::vector<AttnItem> items;
  std::vector<int32_t> ifirst(Bc), icount(Bc);
  int max_splits = 0;
  // in-kernel merge of the key ranges: one session on the tensor-core path
  const bool attn_cluster_ok = block && Bc == 1 && m->dt == DT::BF16 && d == 128 && nrows * (Hq / Hkv) <= 128;
  int attn_cluster = 1;
  if (block) {
    int64_t total = 0;
    std::vector<int64_t> k0v(Bc), k1v(Bc);
    for (int j = 0; j < Bc; ++j) {
      const int64_t F = fw.sess[j]->F;
      // ranges start on a multiple of 64 (a whole tensor-core key tile);
      // positions before the window are masked per query
      k0v[j] = (c.window ? std::max<int64_t>(0, F - c.window + 1) : 0) & ~(int64_t)63;
      k1v[j] = F + nrows;
      total += (k1v[j] - k0v[j]) * Hkv;
    }
    // The key range length of the work items: one CTA runs per SM, so the
    // items run in waves of num_sms, and a wave lasts as long as its longest
    // item.  Among lengths that are multiples of 64 (at least 128), take the
    // one that minimises waves x (length + a fixed cost per item, about four
    // tiles of keys).  Fewer, longer ranges also keep the split partials
    // (R x (d + 4) floats per item) small next to the K/V bytes.
    int64_t maxlen = 1;
    for (int j = 0; j < Bc; ++j) maxlen = std::max<int64_t>(maxlen, k1v[j] - k0v[j]);
    const int64_t top = std::max<int64_t>(128, align_up(maxlen, 64));
    int64_t chunk = top;
    double best = 1e300;
    for (int64_t ch = 128; ch <= top; ch += ch < 1024 ? 64 : 256) {
      int64_t n_items = 0;
      for (int j = 0; j < Bc; ++j) n_items += (int64_t)Hkv * ((k1v[j] - k0v[j] + ch - 1) / ch);
      const int64_t waves = (n_items + m->num_sms - 1) / std::max(1, m->num_sms);
      const double cost = (double)waves * (double)(std::min(ch, maxlen) + 256);
      if (cost < best) {
        best = cost;
        chunk = ch;
      }
    }
    (void)total;
    const int64_t tiles0 = (k1v[0] - k0v[0] + 63) / 64;
    if (attn_cluster_ok && tiles0 > 1 && tiles0 <= kAttnMaxCluster) {
      // one session with a short key range per KV head (a window): one
      // 64-key tile per CTA, the head's tiles one cluster merged in-kernel.
      // Longer ranges keep partials + k_attn_combine: on GB300 clusters of
      // CTAs that stream several tiles each did not beat it.
      chunk = 64;
      attn_cluster = (int)tiles0;
    }
    for (int j = 0; j < Bc; ++j) {
      const int S = (int)((k1v[j] - k0v[j] + chunk - 1) / chunk);
      ifirst[j] = (int32_t)items.size();
      icount[j] = S;
      max_splits = std::max(max_splits, S);
      for (int h = 0; h < Hkv; ++h)
        for (int s = 0; s < S; ++s)
          items.push_back(AttnItem{j, h, k0v[j] + s * chunk, std::min(k1v[j], k0v[j] + (s + 1) * chunk)});
    }
  }
  // each session's proposal state, written in place by the unembedding and the draw
  std::vector<float*> plog(Bc), plse(Bc);
  std::vector<int32_t*> ptok(Bc);
  for (int j = 0; j < Bc; ++j) {
    plog[j] = fw.sess[j]->plogits;
    plse[j] = fw.sess[j]->plse;
    ptok[j] = fw.sess[j]->ptok;
  }
  const size_t o_plog = tp.add(plog), o_plse = tp.add(plse), o_ptok = tp.add(ptok);
  // truncated draws (T > 0 and a session with a top_k): per-session settings and cut rows
  bool any_trunc = false;
  size_t o_trunc = 0, o_pcut = 0;
  if (block && fw.temperature > 0.f) {
    std::vector<Trunc> trv(Bc);
    std::vector<uint64_t*> pcv(Bc);
    for (int j = 0; j < Bc; ++j) {
      trv[j] = fw.sess[j]->trunc;
      pcv[j] = fw.sess[j]->pcut;
      any_trunc = any_trunc || trv[j].top_k > 0;
    }
    if (any_trunc) {
      o_trunc = tp.add(trv);
      o_pcut = tp.add(pcv);
    }
  }
  // the sessions' penalties (propose only; none active: no launch)
  std::vector<Penalty> pen_tab;
  bool o_pen = false;
  for (int j = 0; j < Bc && block; ++j)
    if (penalties_on(fw.sess[j]->pen) && fw.sess[j]->pen.n_hist > 0) o_pen = true;
  if (o_pen) {
    pen_tab.resize(Bc);
    for (int j = 0; j < Bc; ++j) {
      pen_tab[j] = fw.sess[j]->pen;
      if (!penalties_on(pen_tab[j])) pen_tab[j].n_hist = 0;
    }
  }
  const size_t o_rowsrc = tp.add(rowsrc), o_meta = tp.add(meta), o_kv = tp.add(kvb), o_cap = tp.add(capv),
               o_front = tp.add(front), o_seq = tp.add(seqv), o_items = tp.add(items), o_ifirst = tp.add(ifirst),
               o_icount = tp.add(icount), o_map = tp.add(fw.sess_map), o_maps = tp.add(mapv),
               o_fresh = tp.add(fresh);
  // RoPE cos/sin: the model's table indexed by position (angle pos *
  // theta^(-2j/d) in double), extended when a call reaches past it; it grows
  // geometrically, so a steady stream of rounds computes no trigonometry
  int64_t maxpos = 0;
  for (int r = 0; r < M; ++r) maxpos = std::max<int64_t>(maxpos, meta[r].pos + 1);
  if (maxpos > m->rope_len) {
    const int64_t want = std::max<int64_t>({maxpos, 2 * m->rope_len, 4096});
    ST_TRY(m->rope.ensure((size_t)want * (d / 2) * sizeof(float2), st));
    launch_rope_table(nullptr, 0, (int)want, d, c.rope_theta, m->rope.as<float2>(), st);
    m->launches++;
    m->rope_len = want;
  }
  ST_TRY(m->ring.upload(tp, m->tables, st));
  char* tb = m->tables.as<char>();
  SessTables tabs{(void* const*)(tb + o_kv), (const int64_t*)(tb + o_cap), (const int64_t*)(tb + o_front),
                  (const int32_t*)(tb + o_seq), have_maps ? (const CUtensorMap* const*)(tb + o_maps) : nullptr,
                  (const int64_t*)(tb + o_fresh)};
  const RowMeta* dmeta = (const RowMeta*)(tb + o_meta);

  // ---- buffers -----------------------------------------------------------
  ST_TRY(m->x.ensure((size_t)M * H * es, st));
  ST_TRY(m->qkv.ensure((size_t)M * m->qkv_cols * 4, st));
  if (Mc) {
    ST_TRY(m->u.ensure((size_t)Mc * KHt * es, st));
    ST_TRY(m->fcout.ensure((size_t)Mc * H * 4, st));
    ST_TRY(m->c.ensure((size_t)Mc * H * es, st));
  }
  if (block) {
    ST_TRY(m->h.ensure((size_t)Mb * H * es, st));
    ST_TRY(m->Q.ensure((size_t)Mb * Hq * d * es, st));
    ST_TRY(m->G.ensure((size_t)Mb * Hq * 4, st));
    ST_TRY(m->O.ensure((size_t)Mb * Hq * d * es, st));
    ST_TRY(m->tmp.ensure((size_t)Mb * std::max(H, 2 * I) * 4, st));
    ST_TRY(m->y.ensure((size_t)Mb * H * es, st));
    ST_TRY(m->a.ensure((size_t)Mb * I * es, st));
    ST_TRY(m->z.ensure((size_t)Bc * fw.n * H * es, st));
    const int R = nrows * (Hq / Hkv);
    ST_TRY(m->apart.ensure(std::max<size_t>(items.size(), 1) * R * (d + 4) * 4, st));
  }

  // ---- context path: aux_hidden_norms -> fc -> hidden_norm ----------------
  if (Mc) {
    launch_tap_norm(m->dt, (const void* const*)(tb + o_rowsrc), Mc, m->aux_norms, m->u.p, c.n_taps, c.target_hidden,
                    c.rms_eps, st);
    ST_TRY(gemm(m, m->u.p, KHt, m->w_fc, KHt, m->fcout.as<float>(), H, Mc, H, KHt, st));
    launch_rmsnorm(m->dt, true, m->fcout.p, Mc, nullptr, H, m->hidden_norm, m->c.p, H, Mc, H, Mc, 0, 0, c.rms_eps, st);
    m->launches += 2;
  }
  if (block) {
    launch_embed(m->dt, m->embed, fw.current, (const int32_t*)(tb + o_map), c.mask_token, V, Bc, nrows, H, m->h.p,
                 m->d_err, st);
    m->launches++;
  }
  const float2* rope = m->rope.as<float2>();
  ST_TRY(launch_check("context path"));
  const int qd = Hq * d, kd = Hkv * d;
  const void* const* d_in_gains = m->d_gains;
  const void* const* d_k_gains = m->d_gains + c.n_layers;
  if (!block && m->use_tc && M > 128) {
    // many context rows: every layer's input norm in one launch, every
    // layer's K/V product as one grouped product (each layer's sums as its
    // own call would make them), every layer's cache write in one launch
    const int L = c.n_layers;
    ST_TRY(m->xall.ensure((size_t)L * M * H * es, st));
    ST_TRY(m->kvall.ensure((size_t)L * M * 2 * kd * 4, st));
    launch_rmsnorm_layers(m->dt, m->c.p, H, d_in_gains, m->xall.p, H, (int64_t)M * H, M, L, H, c.rms_eps, st);
    {
      const double bytes = (double)L * (2.0 * kd * H * es + (double)M * H * es + (double)M * 2 * kd * 4);
      Timed tm(m, kGemmTc, bytes, 2.0 * L * M * 2 * kd * H, st);
      if (tc_gemm_grouped(m->tc, m->xall.p, H, m->w_kv, H, m->kvall.as<float>(), 2 * kd, (int64_t)M * 2 * kd, M,
                          2 * kd, H, L, st))
        return fail(DFLASH_ERR_CUDA, "tcgen05 GEMM: %s", tc_last_error());
    }
    launch_kv_ctx(m->dt, m->kvall.as<float>(), 2 * kd, 0, kd, (int64_t)M * 2 * kd, dmeta, M, rope, d_k_gains, Hkv, d,
                  c.rms_eps, tabs, 0, L, st);
    m->launches += 3;
    return launch_check("grouped context forward");
  }

  AttnParams ap{Hq, Hkv, d, nrows, c.window, c.causal_block, c.n_layers, 0, 1.f / std::sqrt((float)d)};
  double attn_bytes = 0, attn_flops = 0;  // per layer: K/V read once, Q read, O written
  for (const AttnItem& it : items) {
    attn_bytes += (double)(it.k1 - it.k0) * d * 2 * es;
    attn_flops += 4.0 * (it.k1 - it.k0) * d * nrows * (Hq / Hkv);
  }
  attn_bytes += 2.0 * Mb * Hq * d * es;
  for (int l = 0; l < c.n_layers; ++l) {
    const LayerW& w = m->layers[l];
    // input_layernorm over [context rows ; block rows]
    launch_rmsnorm(m->dt, false, m->c.p, Mc, m->h.p, H, w.in_norm, m->x.p, H, M, H, M, 0, 0, c.rms_eps, st);
    m->launches++;
    if (block) {
      // k_qkv_post, next, reads its row and session tables before its wait
      // (the tensor-core product lets it start only once they are written)
      const void* wq = w.w_qkvg ? w.w_qkvg : w.w_qkv;
      ST_TRY(gemm(m, m->x.p, H, wq, H, m->qkv.as<float>(), m->qkv_cols, M, m->qkv_cols, H, st, true));
    } else {
      // context-only forward: the K/V rows of the fused projection only
      const char* wkv = (const char*)w.w_qkv + (size_t)qd * H * es;
      ST_TRY(gemm(m, m->x.p, H, wkv, H, m->qkv.as<float>() + qd, m->qkv_cols, M, 2 * kd, H, st));
    }
    if (!block) {
      // context rows only: K and V straight into the caches, 32 rows per CTA
      launch_kv_ctx(m->dt, m->qkv.as<float>(), m->qkv_cols, qd, qd + kd, 0, dmeta, M, rope, d_k_gains + l, Hkv, d,
                    c.rms_eps, tabs, l, 1, st);
      m->launches++;
      ST_TRY(launch_check("kv"));
      continue;
    }
    m->launches += launch_qkv_post(m->dt, m->qkv.as<float>(), m->qkv_cols, dmeta, M, rope, w.q_norm, w.k_norm, Hq,
                                   Hkv, d, c.gated_attention, c.rms_eps, tabs, c.n_layers, l, m->Q.p,
                                   m->G.as<float>(), st, m->use_tc ? 1 : 0);
    ST_TRY(launch_check("qkv"));
    ap.layer = l;
    {
      Timed tm(m, kAttention, attn_bytes, attn_flops, st);
      const AttnItem* ditems = (const AttnItem*)(tb + o_items);
      ap.cluster = attn_cluster;
      ap.out = m->O.p;
      ap.gates = c.gated_attention ? m->G.as<float>() : nullptr;
      int how = 0;
      if (m->dt == DT::BF16)
        how = launch_attention_tc(m->Q.p, ditems, (int)items.size(), tabs, ap, m->apart.as<float>(), m->d_err, st);
      if (how == 0)
        launch_attention_simt(m->dt, m->Q.p, ditems, (int)items.size(), tabs, ap, m->apart.as<float>(), st);
      if (how != 2)
        launch_attention_combine(m->dt, m->apart.as<float>(), (const int32_t*)(tb + o_ifirst),
                                 (const int32_t*)(tb + o_icount), Bc, ap, c.gated_attention ? m->G.as<float>() : nullptr,
                                 m->O.p, st, max_splits, how == 1 ? 1 : 0);
      m->launches += 2;
    }
    ST_TRY(launch_check("attention"));
    ST_TRY(gemm_resid(m, m->O.p, qd, w.w_o, m->h.p, m->tmp.as<float>(), Mb, H, qd, st));
    if (m->dflash2) {
      // DFlash2's block-local dynamic convolution: x = RMSNorm(h; conv_norm)
      // (into y, free until the post-norm below), the kernel logits W_dc x
      // (into tmp), then h_i += sum_j softmax(...)_j x_{i-j} within the block
      const int GK = Hq * c.conv_taps;
      launch_rmsnorm(m->dt, false, m->h.p, Mb, nullptr, H, w.conv_norm, m->y.p, H, Mb, H, Mb, 0, 0, c.rms_eps, st);
      ST_TRY(gemm(m, m->y.p, H, w.w_dc, H, m->tmp.as<float>(), GK, Mb, GK, H, st));
      launch_dynconv(m->dt, m->h.p, m->y.p, m->tmp.as<float>(), Mb, nrows, H, Hq, c.conv_taps, st);
      m->launches += 2;
      ST_TRY(launch_check("dynamic convolution"));
    }
    launch_rmsnorm(m->dt, false, m->h.p, Mb, nullptr, H, w.post_norm, m->y.p, H, Mb, H, Mb, 0, 0, c.rms_eps, st);
    m->launches++;
    ST_TRY(gemm_swiglu(m, m->y.p, w.w_gate, w.w_up, m->a.p, m->tmp.as<float>(), Mb, I, H, st));
    ST_TRY(gemm_resid(m, m->a.p, I, w.w_down, m->h.p, m->tmp.as<float>(), Mb, H, I, st));
    ST_TRY(launch_check("mlp"));
  }
  if (!block) return DFLASH_OK;

  // ---- rows 1..n: final norm, unembedding, one batched draw ----------------
  const int n = fw.n, Rz = Bc * n;
  launch_rmsnorm(m->dt, false, m->h.p, Mb, nullptr, H, m->final_norm, m->z.p, H, Rz, H, n, nrows, 1, c.rms_eps, st);
  m->launches++;
  // The tensor-core unembedding writes each session's rows straight into its
  // proposal buffer; the CUDA-core path writes one block that is copied out.
  float* lg = nullptr;
  const bool seg = m->use_tc && Bc > 1;
  if (Bc == 1) {
    lg = fw.sess[0]->plogits;
  } else if (!seg) {
    ST_TRY(m->logits.ensure((size_t)Rz * V * 4, st));
    lg = m->logits.as<float>();
  }
  if (seg) {
    ST_TRY(gemm_rows(m, m->z.p, H, m->unembed, H, (void* const*)(tb + o_plog), n, V, Rz, V, H, st));
  } else {
    ST_TRY(gemm(m, m->z.p, H, m->unembed, H, lg, V, Rz, V, H, st));
  }
  // the sessions' rows of logits, and the copies that finish a draw: the
  // logits block of a CUDA-core batch into each session, and out_logits
  auto session_rows = [&]() {
    std::vector<float*> rows(Bc);
    for (int j = 0; j < Bc; ++j) rows[j] = (seg || Bc == 1) ? fw.sess[j]->plogits : lg + (size_t)j * n * V;
    return rows;
  };
  auto finish_copies = [&]() -> int {
    for (int j = 0; j < Bc; ++j) {
      dflash_session* s = fw.sess[j];
      if (Bc > 1 && !seg)
        CU_TRY(cudaMemcpyAsync(s->plogits, lg + (size_t)j * n * V, (size_t)n * V * 4, cudaMemcpyDeviceToDevice, st));
      if (fw.out_logits)
        CU_TRY(cudaMemcpyAsync(fw.out_logits + (size_t)fw.sess_map[j] * n * V, s->plogits, (size_t)n * V * 4,
                               cudaMemcpyDeviceToDevice, st));
    }
    return DFLASH_OK;
  };
  if (m->dflash2) {
    // DFlash2's selector (dflash.go selectBlock, the BlockSelector branch):
    // the candidates of every row, then each session's positions in order,
    // at the request temperature only (no truncation, no penalties)
    const int kc = c.sel_candidates, nch = topk_chunks(V);
    std::vector<int32_t*> sid(Bc);
    std::vector<float*> spr(Bc);
    for (int j = 0; j < Bc; ++j) {
      sid[j] = fw.sess[j]->pcand_ids;
      spr[j] = fw.sess[j]->pcand_probs;
    }
    TablePack pk;
    const size_t o_r = pk.add(session_rows()), o_i = pk.add(sid), o_p = pk.add(spr);
    ST_TRY(m->ring.upload(pk, m->vpen_tab, st));
    char* pb = m->vpen_tab.as<char>();
    ST_TRY(m->d2part.ensure((size_t)Rz * nch * kc * sizeof(uint64_t), st));
    ST_TRY(m->d2cand.ensure((size_t)Rz * kc * 8, st));
    int32_t* cid = m->d2cand.as<int32_t>();
    float* clg = reinterpret_cast<float*>(cid + (size_t)Rz * kc);
    {
      Timed tm(m, kSample, (double)Rz * V * 4, 2.0 * Rz * V, st);
      launch_topk_candidates((const float* const*)(pb + o_r), n, V, V, kc, Rz, m->d2part.as<uint64_t>(), cid, clg, st);
      SelectArgs sel{};
      sel.B = Bc;
      sel.n = n;
      sel.kc = kc;
      sel.rank = c.sel_rank;
      sel.V = V;
      sel.temperature = fw.temperature;
      sel.seed = fw.seed;
      sel.rnd = (uint32_t)fw.rnd;
      sel.current = fw.current;
      sel.sess_map = (const int32_t*)(tb + o_map);
      sel.seq_ids = tabs.seq;
      sel.sel_prev = m->sel_prev;
      sel.sel_next = m->sel_next;
      sel.cand_ids = cid;
      sel.cand_logit = clg;
      sel.sess_tok = (int32_t* const*)(tb + o_ptok);
      sel.sess_ids = (int32_t* const*)(pb + o_i);
      sel.sess_probs = (float* const*)(pb + o_p);
      sel.out_tokens = fw.out_tokens;
      sel.out_q = fw.out_q;
      sel.err = m->d_err;
      launch_select(m->dt, sel, st);
      m->launches += 4;
    }
    ST_TRY(launch_check("selector"));
    return finish_copies();
  }
  if (o_pen) {
    // every row of a session's block gets the same committed-history penalties
    TablePack pk;
    const size_t o_p = pk.add(pen_tab), o_r = pk.add(session_rows());
    ST_TRY(m->ring.upload(pk, m->vpen_tab, st));
    char* pb = m->vpen_tab.as<char>();
    launch_penalize_rows((const Penalty*)(pb + o_p), (float* const*)(pb + o_r), n, V, V, Bc, st);
    m->launches += 2;
    ST_TRY(launch_check("penalties"));
  }
  const int chunk = sample_chunk(Rz, V, m->num_sms), chunks = (V + chunk - 1) / chunk;
  ST_TRY(m->spart.ensure((size_t)Rz * chunks * sizeof(float4), st));
  ST_TRY(m->vstat.ensure((size_t)Rz * 8, st));
  SampleArgs sa{};
  sa.logits = lg;
  sa.seq_logits = seg ? (const float* const*)(tb + o_plog) : nullptr;
  if (any_trunc) ST_TRY(m->cutbuf.ensure((size_t)Rz * 8, st));
  sa.sess_tok = (int32_t* const*)(tb + o_ptok);
  sa.sess_lse = (float* const*)(tb + o_plse);
  sa.ld = V;
  sa.rows = Rz;
  sa.V = V;
  sa.in_bf16 = 0;
  sa.temperature = fw.temperature;
  sa.gumbel = fw.temperature > 0.f;
  sa.seed = fw.seed;
  sa.rnd = (uint32_t)fw.rnd;
  sa.rows_per_seq = n;
  sa.row_offset = 1;
  sa.seq_ids = tabs.seq;
  sa.err = m->d_err;
  {
    Timed tm(m, kSample, (double)Rz * V * 4, 6.0 * Rz * V, st);
    if (any_trunc) {
      uint64_t* cut = m->cutbuf.as<uint64_t>();
      launch_trunc_cut(sa, (const Trunc*)(tb + o_trunc), cut, (uint64_t* const*)(tb + o_pcut), st);
      sa.cut = cut;
      m->launches++;
    }
    launch_sample_partials(sa, chunk, m->spart.as<float4>(), st);
    // tokens and log-sum-exp into the sessions, tokens and q(token) in caller order
    sa.out_map = (const int32_t*)(tb + o_map);
    launch_sample_combine(sa, chunks, m->spart.as<float4>(), fw.out_tokens, fw.out_q, nullptr, st);
    m->launches += 2;
  }
  ST_TRY(launch_check("sample"));
  return finish_copies();
}

// Context rows of one session's held features (and optionally extra rows
// straight from the caller), with the window drop applied.  F advances
// past every row; P returns to zero.
// The held rows (staged, concatenated taps) and then extra_rows new rows read
// in place: tap k of new row j at extra[k] + j * extra_stride bytes.
void take_pending(dflash_session* s, int32_t sess_idx, const char* const* extra, int64_t extra_stride, int extra_rows,
                  std::vector<CtxRow>& out) {
  const dflash_config& c = s->m->cfg;
  const size_t tapb = (size_t)c.target_hidden * s->m->esz, rowb = (size_t)c.n_taps * tapb;
  const int64_t first = s->F;
  const int total = s->P + extra_rows;
  const int64_t Fnew = first + total;
  for (int r = 0; r < total; ++r) {
    const int64_t slot = first + r;
    if (c.window && slot <= Fnew - c.window) continue;  // no later query can see it
    CtxRow row{};
    row.sess = sess_idx;
    row.pos = slot;
    for (int k = 0; k < c.n_taps; ++k)
      row.tap[k] = r < s->P ? (const char*)s->pending + (size_t)r * rowb + k * tapb
                            : extra[k] + (size_t)(r - s->P) * extra_stride;
    out.push_back(row);
  }
  s->flushed_rows += total;
  s->F = Fnew;
  s->P = 0;
}

void commit_block(dflash_session* s) {
  if (!s->block_outstanding) return;
  s->block_outstanding = false;  // the block's slots past F are free again
}

int check_sessions(dflash_session* const* s, int32_t batch) {
  if (!s || batch < 1) return fail(DFLASH_ERR_INVALID_ARG, "null session array or batch < 1");
  for (int b = 0; b < batch; ++b) {
    if (!s[b]) return fail(DFLASH_ERR_INVALID_ARG, "session %d is null", b);
    if (s[b]->m != s[0]->m) return fail(DFLASH_ERR_INVALID_ARG, "sessions of different models in one batch");
    for (int j = 0; j < b; ++j)
      if (s[j] == s[b]) return fail(DFLASH_ERR_INVALID_ARG, "session %d repeated in batch", b);
  }
  return DFLASH_OK;
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

// Internal accessors for the allocation-free verify (verify_noalloc.cu);
// hidden symbols, not part of the ABI.
int dflash__set_error(int code, const char* msg) { return fail(code, "%s", msg); }

int dflash__session_truncation(const dflash_session* s, Trunc* trunc, const uint64_t** proposal_cut) {
  *trunc = s->trunc;
  *proposal_cut = s->last_trunc ? s->pcut : nullptr;
  return DFLASH_OK;
}

int dflash__session_proposal(const dflash_session* s, const float** logits, const float** lse,
                             const int32_t** tokens, float* temperature, int32_t* n, long long** accepted,
                             void** stream, int32_t* vocab, int32_t* draft_limit, int32_t** err, const void** model) {
  *logits = s->plogits;
  *lse = s->plse;
  *tokens = s->ptok;
  *temperature = s->last_T;
  *n = s->has_prop ? s->last_n : 0;
  *accepted = s->d_accepted;
  *stream = (void*)s->stream;
  *vocab = s->m->cfg.vocab;
  *draft_limit = s->m->cfg.block_size - 1;
  *err = s->m->d_err;
  *model = s->m;
  return DFLASH_OK;
}

int dflash__session_device(const dflash_session* s) { return s->device; }
int dflash__session_penalties(const dflash_session* s) { return penalties_on(s->pen) ? 1 : 0; }

// A Timed bracket that the allocation-free verify can open and close across
// its launches (the class is kVerify); the handle is an index into the
// model's records, or -1 while timing is off.
long long dflash__verify_timing_begin(const void* model, double bytes, double flops, void* stream) {
  dflash_model* m = (dflash_model*)model;
  Timed t(m, kVerify, bytes, flops, (cudaStream_t)stream);
  const long long idx = t.idx == (size_t)-1 ? -1 : (long long)t.idx;
  t.idx = (size_t)-1;  // closed by dflash__verify_timing_end
  return idx;
}

void dflash__verify_timing_end(const void* model, long long idx, void* stream) {
  dflash_model* m = (dflash_model*)model;
  if (idx >= 0 && (size_t)idx < m->recs.size()) cudaEventRecord(m->recs[(size_t)idx].e1, (cudaStream_t)stream);
}

void dflash__count_launches(const void* model, int n) { ((dflash_model*)model)->launches += n; }

const char* dflash_last_error(void) { return g_err.c_str(); }
int dflash_version(void) { return 200; }

int dflash_model_create(const dflash_config* cfg, const dflash_weights* w, dflash_model** out) {
  if (!cfg || !w || !out) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  ST_TRY(check_config(*cfg));
  const dflash_config& c = *cfg;
  if (!w->aux_norms || !w->w_fc || !w->hidden_norm || !w->final_norm || !w->embed || !w->unembed || !w->layers)
    return fail(DFLASH_ERR_INVALID_ARG, "null model weight");
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_layer_weights& lw = w->layers[l];
    if (!lw.in_norm || !lw.w_qkv || !lw.q_norm || !lw.k_norm || !lw.w_o || !lw.post_norm || !lw.w_gate || !lw.w_up ||
        !lw.w_down)
      return fail(DFLASH_ERR_INVALID_ARG, "null weight in layer %d", l);
    if (c.gated_attention && !lw.w_g) return fail(DFLASH_ERR_SHAPE, "layer %d: gated attention without g_proj", l);
    if (c.variant == DFLASH_VARIANT_DFLASH2 && (!lw.conv_norm || !lw.w_dc))
      return fail(DFLASH_ERR_INVALID_ARG, "layer %d: DFlash2 without conv_norm / w_dc", l);
    if (!c.gated_attention && lw.w_g) return fail(DFLASH_ERR_SHAPE, "layer %d: g_proj given but gating is off", l);
  }
  if (c.variant == DFLASH_VARIANT_DFLASH2 && (!w->sel_prev || !w->sel_next))
    return fail(DFLASH_ERR_INVALID_ARG, "DFlash2 without the selector tables");
  dflash_model* m = new dflash_model();
  m->cfg = c;
  m->dflash2 = c.variant == DFLASH_VARIANT_DFLASH2;
  if (m->dflash2) {
    m->sel_prev = w->sel_prev;
    m->sel_next = w->sel_next;
  }
  m->dt = c.dtype == DFLASH_DTYPE_BF16 ? DT::BF16 : DT::F32;
  m->esz = dt_size(m->dt);
  m->aux_norms = w->aux_norms;
  m->w_fc = w->w_fc;
  m->hidden_norm = w->hidden_norm;
  m->final_norm = w->final_norm;
  m->embed = w->embed;
  m->unembed = w->unembed;
  m->qkv_rows = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
  m->qkv_cols = m->qkv_rows + (c.gated_attention ? c.n_q_heads : 0);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaMalloc(&m->d_err, 16);
  if (e == cudaSuccess) e = cudaMemset(m->d_err, 0, 16);
  if (e != cudaSuccess) {
    delete m;
    return fail(DFLASH_ERR_CUDA, "device setup: %s", cudaGetErrorString(e));
  }
  m->layers.resize(c.n_layers);
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash_layer_weights& lw = w->layers[l];
    LayerW& L = m->layers[l];
    L = LayerW{lw.in_norm, lw.w_qkv, lw.q_norm, lw.k_norm, lw.w_g, lw.w_o, lw.post_norm, lw.w_gate, lw.w_up, lw.w_down,
               nullptr, m->dflash2 ? lw.conv_norm : nullptr, m->dflash2 ? lw.w_dc : nullptr};
    if (c.gated_attention) {
      // one product for q | k | v | gate: a packed copy of the two matrices
      const size_t a = (size_t)m->qkv_rows * c.hidden * m->esz, g = (size_t)c.n_q_heads * c.hidden * m->esz;
      e = cudaMalloc(&L.w_qkvg, a + g);
      if (e == cudaSuccess) e = cudaMemcpy(L.w_qkvg, lw.w_qkv, a, cudaMemcpyDeviceToDevice);
      if (e == cudaSuccess) e = cudaMemcpy((char*)L.w_qkvg + a, lw.w_g, g, cudaMemcpyDeviceToDevice);
      if (e != cudaSuccess) {
        dflash_model_destroy(m);
        return fail(e == cudaErrorMemoryAllocation ? DFLASH_ERR_OOM : DFLASH_ERR_CUDA, "packing qkv+g: %s",
                    cudaGetErrorString(e));
      }
    }
  }
  m->use_tc = m->dt == DT::BF16 && !(c.flags & DFLASH_FLAG_SIMT_GEMM);
  if (m->use_tc) {
    if (tc_create(&m->tc, m->num_sms, m->d_err)) {
      const std::string msg = tc_last_error();
      dflash_model_destroy(m);
      return fail(DFLASH_ERR_CUDA, "tcgen05 setup: %s", msg.c_str());
    }
  }
  {
    // the gain tables, and (tensor-core path) the packed K/V weight rows
    std::vector<const void*> gains(2 * (size_t)c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
      gains[l] = m->layers[l].in_norm;
      gains[c.n_layers + l] = m->layers[l].k_norm;
    }
    e = cudaMalloc((void**)&m->d_gains, gains.size() * sizeof(void*));
    if (e == cudaSuccess) e = cudaMemcpy(m->d_gains, gains.data(), gains.size() * sizeof(void*), cudaMemcpyHostToDevice);
    const size_t kvb = (size_t)2 * c.n_kv_heads * c.head_dim * c.hidden * m->esz;
    const size_t qb = (size_t)c.n_q_heads * c.head_dim * c.hidden * m->esz;
    if (e == cudaSuccess && m->use_tc) e = cudaMalloc(&m->w_kv, kvb * c.n_layers);
    for (int l = 0; l < c.n_layers && e == cudaSuccess && m->use_tc; ++l)
      e = cudaMemcpy((char*)m->w_kv + kvb * l, (const char*)m->layers[l].w_qkv + qb, kvb, cudaMemcpyDeviceToDevice);
    if (e != cudaSuccess) {
      dflash_model_destroy(m);
      return fail(e == cudaErrorMemoryAllocation ? DFLASH_ERR_OOM : DFLASH_ERR_CUDA, "gain tables / packed K/V: %s",
                  cudaGetErrorString(e));
    }
  }
  *out = m;
  return DFLASH_OK;
}

int dflash_model_destroy(dflash_model* m) {
  if (!m) return fail(DFLASH_ERR_INVALID_ARG, "null model");
  cudaDeviceSynchronize();
  for (auto& L : m->layers)
    if (L.w_qkvg) cudaFree(L.w_qkvg);
  Buf* bufs[] = {&m->tables, &m->u, &m->fcout, &m->c, &m->h, &m->x, &m->qkv, &m->rope, &m->Q, &m->G,
                 &m->O, &m->tmp, &m->y, &m->a, &m->z, &m->logits, &m->spart, &m->apart, &m->vstat, &m->vpart, &m->cutbuf,
                 &m->vbonus, &m->vpen, &m->vpen_tab, &m->d2part, &m->d2cand, &m->xall, &m->kvall};
  for (Buf* b : bufs) b->release();
  m->ring.release();
  for (auto& e : m->ev_pool) {
    cudaEventDestroy(e.first);
    cudaEventDestroy(e.second);
  }
  if (m->d_err) cudaFree(m->d_err);
  if (m->w_kv) cudaFree(m->w_kv);
  if (m->d_gains) cudaFree(m->d_gains);
  if (m->tc) tc_destroy(m->tc);
  delete m;
  return DFLASH_OK;
}

int dflash_draft_limit(const dflash_model* m) {
  if (!m) return fail(DFLASH_ERR_INVALID_ARG, "null model");
  return m->cfg.block_size - 1;
}

int dflash_device_status(dflash_model* m) {
  if (!m) return fail(DFLASH_ERR_INVALID_ARG, "null model");
  int32_t e = 0;
  CU_TRY(cudaDeviceSynchronize());
  CU_TRY(cudaMemcpy(&e, m->d_err, 4, cudaMemcpyDeviceToHost));
  CU_TRY(cudaMemset(m->d_err, 0, 4));
  if (e) {
    std::string why;
    if (e & 1) why += "anchor token id outside the vocabulary; ";
    if (e & 2) why += "draft token id outside the vocabulary; ";
    if (e & 4) why += "tensor-core GEMM pipeline wait expired; ";
    if (e & 8) why += "tensor-core attention pipeline wait expired; ";
    if (e & 16) why += "a logits row had no comparable score (non-finite values); ";
    return fail(DFLASH_ERR_DEVICE, "device reported: %s", why.c_str());
  }
  return DFLASH_OK;
}

int dflash_open(dflash_model* m, int64_t restored_offset, int64_t max_ctx, void* stream, dflash_session** out) {
  if (!m || !out) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  const dflash_config& c = m->cfg;
  if (max_ctx < 1 || restored_offset < 0 || restored_offset > max_ctx)
    return fail(DFLASH_ERR_INVALID_ARG, "max_ctx %lld / restored_offset %lld", (long long)max_ctx,
                (long long)restored_offset);
  dflash_session* s = new dflash_session();
  s->m = m;
  s->stream = (cudaStream_t)stream;
  if (cudaGetDevice(&s->device) != cudaSuccess) s->device = 0;
  s->F = restored_offset;
  s->max_ctx = max_ctx;
  s->cap = c.window ? align_up((int64_t)c.window + c.block_size, 64) : align_up(max_ctx + c.block_size, 64);
  const size_t kvb = (size_t)c.n_layers * 2 * c.n_kv_heads * s->cap * c.head_dim * m->esz;
  const size_t pend = (size_t)DFLASH_PENDING_FLUSH_TOKENS * c.n_taps * c.target_hidden * m->esz;
  const size_t nb = (size_t)(c.block_size - 1);
  cudaError_t e = cudaMalloc(&s->kv, kvb);
  if (e == cudaSuccess) e = cudaMemsetAsync(s->kv, 0, kvb, s->stream);
  if (e == cudaSuccess) e = cudaMalloc(&s->pending, pend);
  if (e == cudaSuccess) e = cudaMalloc((void**)&s->plogits, nb * c.vocab * 4);
  if (e == cudaSuccess) e = cudaMalloc((void**)&s->plse, nb * 4);
  if (e == cudaSuccess) e = cudaMalloc((void**)&s->ptok, nb * 4);
  if (e == cudaSuccess) e = cudaMalloc((void**)&s->pcut, nb * 8);
  if (e == cudaSuccess) e = cudaMalloc((void**)&s->d_accepted, 8);
  if (e == cudaSuccess && m->dflash2) e = cudaMalloc((void**)&s->pcand_ids, nb * c.sel_candidates * 4);
  if (e == cudaSuccess && m->dflash2) e = cudaMalloc((void**)&s->pcand_probs, nb * c.sel_candidates * 4);
  if (e == cudaSuccess) e = cudaMemsetAsync(s->d_accepted, 0, 8, s->stream);
  // the model's RoPE table covers every position this session can reach
  // (committed rows stop at max_ctx; a block adds block_size), so no call of
  // the session has to grow it
  const int64_t positions = max_ctx + c.block_size;
  if (e == cudaSuccess && positions > m->rope_len) {
    e = cudaDeviceSynchronize();  // no call of any stream may still read the old table
    if (e == cudaSuccess && m->rope.ensure((size_t)positions * (c.head_dim / 2) * sizeof(float2), s->stream) != DFLASH_OK)
      e = cudaErrorMemoryAllocation;
    if (e == cudaSuccess) {
      launch_rope_table(nullptr, 0, (int)positions, c.head_dim, c.rope_theta, m->rope.as<float2>(), s->stream);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) m->rope_len = positions;
  }
  if (e == cudaSuccess && m->use_tc && c.head_dim == 128) {
    CUtensorMap maps[2];
    if (tc_encode_kv_maps(m->tc, s->kv, s->cap, c.head_dim, 2 * c.n_layers * c.n_kv_heads, maps) != 0) {
      e = cudaErrorInvalidValue;
    } else {
      e = cudaMalloc((void**)&s->d_maps, sizeof maps);
      if (e == cudaSuccess) e = cudaMemcpy(s->d_maps, maps, sizeof maps, cudaMemcpyHostToDevice);
    }
  }
  if (e != cudaSuccess) {
    cudaFree(s->kv);
    cudaFree(s->pending);
    cudaFree(s->plogits);
    cudaFree(s->plse);
    cudaFree(s->ptok);
    cudaFree(s->pcut);
    cudaFree(s->d_accepted);
    cudaFree(s->d_maps);
    cudaFree(s->pcand_ids);
    cudaFree(s->pcand_probs);
    delete s;
    return fail(e == cudaErrorMemoryAllocation ? DFLASH_ERR_OOM : DFLASH_ERR_CUDA, "session buffers: %s",
                cudaGetErrorString(e));
  }
  *out = s;
  return DFLASH_OK;
}

// committed for a run whose tap k of row j is at taps[k] + j * row_bytes;
// concat: the taps are the consecutive slices of one feature row.
static int committed_impl(dflash_session* s, const char* const* taps, int64_t row_bytes, bool concat, int32_t n_rows,
                   int64_t position) {
  const dflash_config& c = s->m->cfg;
  const int64_t width = (int64_t)c.n_taps * c.target_hidden;
  const int64_t start = s->F + s->P - position;
  if (start < 0)
    return fail(DFLASH_ERR_CONTEXT_GAP, "committed run at %lld leaves a context gap at %lld", (long long)position,
                (long long)(s->F + s->P));
  if (start >= n_rows) return DFLASH_OK;  // restored prefix: nothing new
  const int add = (int)(n_rows - start);
  if (s->F + s->P + add > s->max_ctx)
    return fail(DFLASH_ERR_CAPACITY, "context would reach %lld rows, max_ctx %lld", (long long)(s->F + s->P + add),
                (long long)s->max_ctx);
  const size_t es = s->m->esz;
  const char* src[kMaxTaps];
  for (int k = 0; k < c.n_taps; ++k) src[k] = taps[k] + (size_t)start * row_bytes;
  if (s->P + add < DFLASH_PENDING_FLUSH_TOKENS) {
    char* dst = (char*)s->pending + (size_t)s->P * width * es;
    if (concat) {
      launch_copy_rows(dst, (int64_t)(width * es), src[0], row_bytes, (int64_t)(width * es), add, s->stream);
    } else {
      TapSrc ts{};
      for (int k = 0; k < c.n_taps; ++k) ts.p[k] = src[k];
      launch_copy_taps(dst, (int64_t)(width * es), ts, c.n_taps, row_bytes, (int64_t)c.target_hidden * es, add,
                       s->stream);
    }
    ST_TRY(launch_check("pending rows"));
    s->P += add;
    return DFLASH_OK;
  }
  // the held rows reach the flush threshold: one context-only forward over
  // the staged rows and the new rows read in place
  commit_block(s);
  Forward fw;
  fw.sess = {s};
  const int64_t F0 = s->F;
  const int32_t P0 = s->P;
  take_pending(s, 0, src, row_bytes, add, fw.ctx);
  const int rc = run_forward(s->m, fw, s->stream);
  if (rc != DFLASH_OK) {
    s->F = F0;
    s->P = P0;
    return rc;
  }
  s->flushes++;
  return DFLASH_OK;
}

int dflash_committed(dflash_session* s, const void* features, int64_t row_stride, int32_t n_rows, int64_t position) {
  if (!s) return fail(DFLASH_ERR_INVALID_ARG, "null session");
  const dflash_config& c = s->m->cfg;
  const int64_t width = (int64_t)c.n_taps * c.target_hidden;
  if (n_rows < 0 || position < 0) return fail(DFLASH_ERR_INVALID_ARG, "n_rows %d / position %lld", n_rows, (long long)position);
  if (n_rows > 0 && (!features || row_stride < width))
    return fail(DFLASH_ERR_INVALID_ARG, "features null or row_stride %lld < %lld", (long long)row_stride, (long long)width);
  const char* taps[kMaxTaps] = {};
  if (features)
    for (int k = 0; k < c.n_taps; ++k) taps[k] = (const char*)features + (size_t)k * c.target_hidden * s->m->esz;
  return committed_impl(s, taps, row_stride * (int64_t)s->m->esz, true, n_rows, position);
}

int dflash_committed_taps(dflash_session* s, const void* const* taps, int64_t row_stride, int32_t n_rows,
                          int64_t position) {
  if (!s) return fail(DFLASH_ERR_INVALID_ARG, "null session");
  const dflash_config& c = s->m->cfg;
  if (n_rows < 0 || position < 0) return fail(DFLASH_ERR_INVALID_ARG, "n_rows %d / position %lld", n_rows, (long long)position);
  if (n_rows > 0 && (!taps || row_stride < c.target_hidden))
    return fail(DFLASH_ERR_INVALID_ARG, "taps null or row_stride %lld < %d", (long long)row_stride, c.target_hidden);
  const char* tp[kMaxTaps] = {};
  for (int k = 0; k < c.n_taps && n_rows > 0; ++k) {
    if (!taps[k]) return fail(DFLASH_ERR_INVALID_ARG, "tap %d is null", k);
    tp[k] = (const char*)taps[k];
  }
  return committed_impl(s, tp, row_stride * (int64_t)s->m->esz, false, n_rows, position);
}

int dflash_committed_batch(dflash_session* const* s, int32_t batch, const void* const* features, int64_t row_stride,
                           const int32_t* n_rows, const int64_t* position) {
  ST_TRY(check_sessions(s, batch));
  if (!features || !n_rows || !position) return fail(DFLASH_ERR_INVALID_ARG, "null features / n_rows / position");
  dflash_model* m = s[0]->m;
  const dflash_config& c = m->cfg;
  const int64_t width = (int64_t)c.n_taps * c.target_hidden;
  const size_t es = m->esz;
  // every check first, so that an error changes no session
  for (int b = 0; b < batch; ++b) {
    if (n_rows[b] < 0 || position[b] < 0)
      return fail(DFLASH_ERR_INVALID_ARG, "session %d: n_rows %d / position %lld", b, n_rows[b], (long long)position[b]);
    if (n_rows[b] > 0 && (!features[b] || row_stride < width))
      return fail(DFLASH_ERR_INVALID_ARG, "session %d: features null or row_stride %lld < %lld", b,
                  (long long)row_stride, (long long)width);
    const int64_t start = s[b]->F + s[b]->P - position[b];
    if (start < 0)
      return fail(DFLASH_ERR_CONTEXT_GAP, "session %d: committed run at %lld leaves a context gap at %lld", b,
                  (long long)position[b], (long long)(s[b]->F + s[b]->P));
    const int64_t add = std::max<int64_t>(0, n_rows[b] - start);
    if (s[b]->F + s[b]->P + add > s[b]->max_ctx)
      return fail(DFLASH_ERR_CAPACITY, "session %d: context would reach %lld rows, max_ctx %lld", b,
                  (long long)(s[b]->F + s[b]->P + add), (long long)s[b]->max_ctx);
  }
  Forward fw;
  std::vector<int64_t> F0(batch);
  std::vector<int32_t> P0(batch);
  // the staged rows of every session go in one launch per kMaxRowCopies sessions
  RowCopies cp;
  cp.n = 0;
  cp.row_bytes = width * (int64_t)es;
  for (int b = 0; b < batch; ++b) {
    dflash_session* x = s[b];
    F0[b] = x->F;
    P0[b] = x->P;
    const int64_t start = x->F + x->P - position[b];
    if (start >= n_rows[b]) continue;  // restored prefix: nothing new
    const int add = (int)(n_rows[b] - start);
    const char* src[kMaxTaps];
    for (int k = 0; k < c.n_taps; ++k)
      src[k] = (const char*)features[b] + ((size_t)start * row_stride + (size_t)k * c.target_hidden) * es;
    if (x->P + add < DFLASH_PENDING_FLUSH_TOKENS) {
      if (cp.n == kMaxRowCopies) {
        launch_copy_rows_batch(cp, s[0]->stream);
        cp.n = 0;
      }
      cp.dst[cp.n] = (char*)x->pending + (size_t)x->P * width * es;
      cp.src[cp.n] = src[0];
      cp.src_ld[cp.n] = row_stride * (int64_t)es;
      cp.rows[cp.n] = add;
      ++cp.n;
      x->P += add;
      continue;
    }
    // this session reaches the threshold: its held rows and the new rows
    // (read in place) join the one context-only forward of the call
    commit_block(x);
    const int32_t j = (int32_t)fw.sess.size();
    fw.sess.push_back(x);
    take_pending(x, j, src, row_stride * (int64_t)es, add, fw.ctx);
  }
  launch_copy_rows_batch(cp, s[0]->stream);
  int rc = launch_check("pending rows");
  if (rc == DFLASH_OK && !fw.sess.empty()) rc = run_forward(m, fw, s[0]->stream);
  if (rc != DFLASH_OK) {
    for (int b = 0; b < batch; ++b) {
      s[b]->F = F0[b];
      s[b]->P = P0[b];
    }
    return rc;
  }
  for (auto* x : fw.sess) x->flushes++;
  return DFLASH_OK;
}

int dflash_commit_block(dflash_session* const* s, int32_t batch) {
  ST_TRY(check_sessions(s, batch));
  for (int b = 0; b < batch; ++b) commit_block(s[b]);
  return DFLASH_OK;
}

int dflash_flush(dflash_session* const* s, int32_t batch) {
  ST_TRY(check_sessions(s, batch));
  Forward fw;
  std::vector<int64_t> F0(batch);
  std::vector<int32_t> P0(batch);
  for (int b = 0; b < batch; ++b) {
    commit_block(s[b]);
    F0[b] = s[b]->F;
    P0[b] = s[b]->P;
    if (s[b]->P == 0) continue;
    const int32_t j = (int32_t)fw.sess.size();
    fw.sess.push_back(s[b]);
    take_pending(s[b], j, nullptr, 0, 0, fw.ctx);
  }
  if (fw.sess.empty()) return DFLASH_OK;
  const int rc = run_forward(s[0]->m, fw, s[0]->stream);
  if (rc != DFLASH_OK) {
    for (int b = 0; b < batch; ++b) {
      s[b]->F = F0[b];
      s[b]->P = P0[b];
    }
    return rc;
  }
  for (auto* x : fw.sess) x->flushes++;
  return DFLASH_OK;
}

int dflash_settle(dflash_session* s) { return dflash_flush(&s, 1); }

int dflash_propose(dflash_session* const* s, int32_t batch, const int32_t* current, int32_t max_tokens,
                   float temperature, uint64_t seed, uint64_t round, int32_t* out_tokens, float* out_q,
                   float* out_logits, int32_t* out_n) {
  ST_TRY(check_sessions(s, batch));
  if (!out_n) return fail(DFLASH_ERR_INVALID_ARG, "out_n is null");
  if (!(temperature >= 0.f) || std::isinf(temperature)) return fail(DFLASH_ERR_INVALID_ARG, "temperature");
  dflash_model* m = s[0]->m;
  int n = std::min<int>(max_tokens, m->cfg.block_size - 1);
  for (int b = 0; b < batch; ++b) out_n[b] = 0;
  if (n <= 0) return DFLASH_OK;
  // dflash.go dflash2Depth: a DFlash2 session drafts seven tokens every round
  if (m->dflash2) n = std::min<int>(kDflash2Depth, m->cfg.block_size - 1);
  if (!current || !out_tokens || !out_q) return fail(DFLASH_ERR_INVALID_ARG, "null current / out_tokens / out_q");
  Forward fw;
  fw.n = n;
  fw.current = current;
  fw.temperature = temperature;
  fw.seed = seed;
  fw.rnd = round;
  fw.out_tokens = out_tokens;
  fw.out_q = out_q;
  fw.out_logits = out_logits;
  struct Saved { int64_t F; int32_t P; bool bo, hp; };
  std::vector<Saved> saved(batch);
  for (int b = 0; b < batch; ++b) {
    dflash_session* x = s[b];
    saved[b] = Saved{x->F, x->P, x->block_outstanding, x->has_prop};
    if (x->F + x->P == 0) continue;  // nothing committed yet: nil
    if (x->F + x->P + n >= x->cap && !m->cfg.window)
      return fail(DFLASH_ERR_CAPACITY, "session %d: block would pass the cache end", b);
    commit_block(x);
    const int32_t j = (int32_t)fw.sess.size();
    fw.sess.push_back(x);
    fw.sess_map.push_back(b);
    take_pending(x, j, nullptr, 0, 0, fw.ctx);
  }
  if (fw.sess.empty()) return DFLASH_OK;
  const int rc = run_forward(m, fw, s[0]->stream);
  if (rc != DFLASH_OK) {
    for (int b = 0; b < batch; ++b) {
      s[b]->F = saved[b].F;
      s[b]->P = saved[b].P;
      s[b]->block_outstanding = saved[b].bo;
      s[b]->has_prop = saved[b].hp;
    }
    return rc;
  }
  for (size_t j = 0; j < fw.sess.size(); ++j) {
    dflash_session* x = fw.sess[j];
    x->block_outstanding = true;
    x->has_prop = true;
    x->last_n = n;
    x->last_T = temperature;
    x->last_trunc = temperature > 0.f && x->trunc.top_k > 0;  // the forward drew it truncated
    x->rounds++;
    x->proposed += n;
    out_n[fw.sess_map[j]] = n;
  }
  return DFLASH_OK;
}

int dflash_verify(dflash_session* const* s, int32_t batch, const void* target_logits, int32_t logits_dtype,
                  const int32_t* draft_tokens, int32_t n, float temperature, uint64_t seed, uint64_t round,
                  int32_t* out_accept, int32_t* out_bonus) {
  ST_TRY(check_sessions(s, batch));
  if (!target_logits || !draft_tokens || !out_accept || !out_bonus) return fail(DFLASH_ERR_INVALID_ARG, "null pointer");
  if (logits_dtype != DFLASH_DTYPE_F32 && logits_dtype != DFLASH_DTYPE_BF16)
    return fail(DFLASH_ERR_INVALID_ARG, "logits_dtype %d", logits_dtype);
  if (!(temperature >= 0.f) || std::isinf(temperature)) return fail(DFLASH_ERR_INVALID_ARG, "temperature");
  dflash_model* m = s[0]->m;
  if (n < 1 || n > m->cfg.block_size - 1) return fail(DFLASH_ERR_INVALID_ARG, "n = %d", n);
  for (int b = 0; b < batch; ++b)
    if (temperature > 0.f && (!s[b]->has_prop || s[b]->last_n != n))
      return fail(DFLASH_ERR_STATE, "session %d has no proposal of %d tokens to verify against", b, n);
  cudaStream_t st = s[0]->stream;
  const int V = m->cfg.vocab, rows = batch * (n + 1);
  TablePack tp;
  std::vector<const float*> dl(batch), dlse(batch);
  std::vector<const int32_t*> dtok(batch);
  std::vector<float> dT(batch);
  std::vector<long long*> acc(batch);
  std::vector<int32_t> seqv(batch);
  std::vector<Trunc> trv(batch);
  std::vector<const uint64_t*> dcut(batch);
  bool any_trunc = false, any_dcut = false;
  for (int b = 0; b < batch; ++b) {
    dl[b] = s[b]->plogits;
    dlse[b] = s[b]->plse;
    dtok[b] = s[b]->ptok;
    dT[b] = s[b]->last_T;
    acc[b] = s[b]->d_accepted;
    seqv[b] = b;
    trv[b] = s[b]->trunc;
    dcut[b] = s[b]->last_trunc ? s[b]->pcut : nullptr;
    any_trunc = any_trunc || (temperature > 0.f && trv[b].top_k > 0);
    any_dcut = any_dcut || (temperature > 0.f && dcut[b]);
  }
  // penalties: target row r of session b counts b's history plus d_1..d_r
  std::vector<Penalty> penv(batch);
  bool any_pen = false;
  for (int b = 0; b < batch; ++b) {
    penv[b] = s[b]->pen;
    any_pen = any_pen || penalties_on(penv[b]);
  }
  const size_t o_dl = tp.add(dl), o_dlse = tp.add(dlse), o_dtok = tp.add(dtok), o_dT = tp.add(dT), o_acc = tp.add(acc),
               o_seq = tp.add(seqv);
  const size_t o_trunc = any_trunc ? tp.add(trv) : 0, o_dcut = any_dcut ? tp.add(dcut) : 0;
  const size_t o_pen = any_pen ? tp.add(penv) : 0;
  // DFlash2: q of each position is its candidate distribution
  size_t o_cid = 0, o_cpr = 0;
  if (m->dflash2) {
    std::vector<const int32_t*> cid(batch);
    std::vector<const float*> cpr(batch);
    for (int b = 0; b < batch; ++b) {
      cid[b] = s[b]->pcand_ids;
      cpr[b] = s[b]->pcand_probs;
    }
    o_cid = tp.add(cid);
    o_cpr = tp.add(cpr);
  }
  ST_TRY(m->ring.upload(tp, m->tables, st));
  char* tb = m->tables.as<char>();
  const int chunk = sample_chunk(rows, V, m->num_sms), chunks = (V + chunk - 1) / chunk;
  ST_TRY(m->vpart.ensure((size_t)rows * chunks * sizeof(float4), st));
  ST_TRY(m->vstat.ensure((size_t)rows * 8, st));
  int32_t* amax = m->vstat.as<int32_t>();
  float* lse = (float*)(amax + rows);
  SampleArgs sa{};
  sa.logits = target_logits;
  sa.ld = V;
  sa.rows = rows;
  sa.V = V;
  sa.in_bf16 = logits_dtype == DFLASH_DTYPE_BF16;
  sa.temperature = temperature;
  sa.gumbel = 0;
  sa.rows_per_seq = n + 1;
  sa.row_offset = 0;
  sa.err = m->d_err;
  const double tbytes = (double)rows * V * (sa.in_bf16 ? 2 : 4) + (double)batch * V * 4;
  Timed tm(m, kVerify, tbytes, 4.0 * rows * V, st);
  if (any_pen) {
    // the penalised target rows go to a workspace copy (fp32); the caller's
    // logits are never written
    ST_TRY(m->vpen.ensure((size_t)rows * V * 4, st));
    launch_penalize_target((const Penalty*)(tb + o_pen), target_logits, sa.in_bf16, m->vpen.as<float>(),
                           draft_tokens, batch, n, V, st);
    m->launches++;
    sa.logits = m->vpen.p;
    sa.in_bf16 = 0;
  }
  if (any_trunc) {
    ST_TRY(m->cutbuf.ensure((size_t)rows * 8, st));
    launch_trunc_cut(sa, (const Trunc*)(tb + o_trunc), m->cutbuf.as<uint64_t>(), nullptr, st);
    sa.cut = m->cutbuf.as<uint64_t>();
    m->launches++;
  }
  launch_sample_partials(sa, chunk, m->vpart.as<float4>(), st);
  launch_sample_combine(sa, chunks, m->vpart.as<float4>(), amax, nullptr, lse, st);
  m->launches += 3;
  VerifyArgs va{};
  va.target = sa.logits;
  va.in_bf16 = sa.in_bf16;
  va.B = batch;
  va.n = n;
  va.V = V;
  va.temperature = temperature;
  va.seed = seed;
  va.rnd = (uint32_t)round;
  va.seq_ids = (const int32_t*)(tb + o_seq);
  va.draft = draft_tokens;
  va.lse_t = lse;
  va.amax_t = amax;
  va.dlogits = (const float* const*)(tb + o_dl);
  va.dlse = (const float* const*)(tb + o_dlse);
  va.dtok = (const int32_t* const*)(tb + o_dtok);
  va.dtemp = (const float*)(tb + o_dT);
  va.accept = out_accept;
  va.bonus = out_bonus;
  va.accepted_total = (long long* const*)(tb + o_acc);
  va.err = m->d_err;
  va.cut_t = sa.cut;
  va.dcut = any_dcut ? (const uint64_t* const*)(tb + o_dcut) : nullptr;
  if (m->dflash2) {
    va.cand_ids = (const int32_t* const*)(tb + o_cid);
    va.cand_probs = (const float* const*)(tb + o_cpr);
    va.ncand = m->cfg.sel_candidates;
  }
  const int bchunks = verify_bonus_chunks(V);
  ST_TRY(m->vbonus.ensure((size_t)batch * bchunks * sizeof(VerifyPart) + (size_t)batch * 4, st));
  va.rej = (int32_t*)(m->vbonus.as<char>() + (size_t)batch * bchunks * sizeof(VerifyPart));
  launch_verify_accept(va, m->vbonus.as<VerifyPart>(), st);
  m->launches += temperature > 0.f ? 2 : 1;  // bonus draw (T > 0) and finish
  return launch_check("verify");
}

int dflash_candidates(const dflash_session* s, int32_t* out_ids, float* out_probs) {
  if (!s || !out_ids || !out_probs) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  if (!s->m->dflash2) return fail(DFLASH_ERR_STATE, "the model is not a DFlash2 draft");
  if (!s->has_prop) return fail(DFLASH_ERR_STATE, "no proposal yet");
  const size_t bytes = (size_t)s->last_n * s->m->cfg.sel_candidates * 4;
  CU_TRY(cudaMemcpyAsync(out_ids, s->pcand_ids, bytes, cudaMemcpyDeviceToDevice, s->stream));
  CU_TRY(cudaMemcpyAsync(out_probs, s->pcand_probs, bytes, cudaMemcpyDeviceToDevice, s->stream));
  return DFLASH_OK;
}

int dflash__session_candidates(const dflash_session* s, const int32_t** ids, const float** probs, int32_t* kc) {
  *ids = s->m->dflash2 ? s->pcand_ids : nullptr;
  *probs = s->m->dflash2 ? s->pcand_probs : nullptr;
  *kc = s->m->dflash2 ? s->m->cfg.sel_candidates : 0;
  return DFLASH_OK;
}

int dflash_set_penalties(dflash_session* s, float repeat_penalty, float presence_penalty, float frequency_penalty,
                         const int32_t* history, int32_t n_history) {
  if (!s) return fail(DFLASH_ERR_INVALID_ARG, "null session");
  if (!(repeat_penalty > 0.f) || std::isinf(repeat_penalty) || !std::isfinite(presence_penalty) ||
      !std::isfinite(frequency_penalty))
    return fail(DFLASH_ERR_INVALID_ARG, "repeat_penalty must be positive and finite; the others finite");
  if (n_history < 0 || n_history > kMaxPenaltyHistory)
    return fail(DFLASH_ERR_INVALID_ARG, "n_history %d outside [0, %d]", n_history, kMaxPenaltyHistory);
  if (n_history > 0 && !history) return fail(DFLASH_ERR_INVALID_ARG, "null history");
  if (n_history > 0 && !s->d_hist) CU_TRY(cudaMalloc((void**)&s->d_hist, (size_t)kMaxPenaltyHistory * 4));
  if (n_history > 0)
    CU_TRY(cudaMemcpyAsync(s->d_hist, history, (size_t)n_history * 4, cudaMemcpyDeviceToDevice, s->stream));
  s->pen = Penalty{repeat_penalty, presence_penalty, frequency_penalty, n_history, s->d_hist};
  return DFLASH_OK;
}

int dflash_set_sampler(dflash_session* s, int32_t top_k, float top_p, float min_p) {
  if (!s) return fail(DFLASH_ERR_INVALID_ARG, "null session");
  if (top_k < 0 || top_k > kTruncMaxK) return fail(DFLASH_ERR_INVALID_ARG, "top_k %d outside [0, %d]", top_k, kTruncMaxK);
  if (!(top_p > 0.f && top_p <= 1.f)) return fail(DFLASH_ERR_INVALID_ARG, "top_p outside (0, 1]");
  if (!(min_p >= 0.f && min_p <= 1.f)) return fail(DFLASH_ERR_INVALID_ARG, "min_p outside [0, 1]");
  if (top_k == 0 && (top_p < 1.f || min_p > 0.f))
    return fail(DFLASH_ERR_INVALID_ARG, "top_p and min_p act inside a top_k of 1..%d", kTruncMaxK);
  s->trunc = Trunc{top_k, top_p, min_p, 0};
  return DFLASH_OK;
}

int dflash_close(dflash_session* s) {
  if (!s) return fail(DFLASH_ERR_INVALID_ARG, "null session");
  const int rc = dflash_flush(&s, 1);
  cudaStreamSynchronize(s->stream);
  cudaFree(s->kv);
  cudaFree(s->pending);
  cudaFree(s->plogits);
  cudaFree(s->plse);
  cudaFree(s->ptok);
  cudaFree(s->pcut);
  cudaFree(s->d_accepted);
  cudaFree(s->d_maps);
  cudaFree(s->d_hist);
  cudaFree(s->pcand_ids);
  cudaFree(s->pcand_probs);
  delete s;
  return rc;
}

int dflash_stats(const dflash_session* s, dflash_counters* out) {
  if (!s || !out) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  long long acc = 0;
  CU_TRY(cudaStreamSynchronize(s->stream));
  CU_TRY(cudaMemcpy(&acc, s->d_accepted, 8, cudaMemcpyDeviceToHost));
  out->rounds = s->rounds;
  out->proposed = s->proposed;
  out->accepted = acc;
  out->flushes = s->flushes;
  out->flushed_rows = s->flushed_rows;
  return DFLASH_OK;
}

int dflash_session_state(const dflash_session* s, int64_t* ctx_offset, int32_t* pending, int32_t* block_outstanding) {
  if (!s) return fail(DFLASH_ERR_INVALID_ARG, "null session");
  if (ctx_offset) *ctx_offset = s->F;
  if (pending) *pending = s->P;
  if (block_outstanding) *block_outstanding = s->block_outstanding ? 1 : 0;
  return DFLASH_OK;
}

static int kv_range_ok(const dflash_session* s, int32_t layer, int64_t first, int32_t n) {
  const dflash_config& c = s->m->cfg;
  if (layer < 0 || layer >= c.n_layers || first < 0 || n < 0) return fail(DFLASH_ERR_INVALID_ARG, "layer / range");
  if (first + n > s->max_ctx + c.block_size) return fail(DFLASH_ERR_CAPACITY, "rows past the cache");
  if (c.window && n > s->cap) return fail(DFLASH_ERR_CAPACITY, "more rows than the ring holds");
  return DFLASH_OK;
}

int dflash_kv_export(const dflash_session* s, int32_t layer, int64_t first_slot, int32_t n_rows, void* k_out,
                     void* v_out) {
  if (!s || !k_out || !v_out) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  ST_TRY(kv_range_ok(s, layer, first_slot, n_rows));
  const dflash_config& c = s->m->cfg;
  const size_t plane = (size_t)c.n_kv_heads * s->cap * c.head_dim * s->m->esz;
  char* base = (char*)s->kv + (size_t)(2 * layer) * plane;
  launch_kv_copy(s->m->dt, base, s->cap, first_slot, k_out, n_rows, c.n_kv_heads, c.head_dim, false, false, s->stream);
  launch_kv_copy(s->m->dt, base + plane, s->cap, first_slot, v_out, n_rows, c.n_kv_heads, c.head_dim, false, true,
                 s->stream);
  return launch_check("kv_export");
}

int dflash_kv_import(dflash_session* s, int32_t layer, int64_t first_slot, int32_t n_rows, const void* k_in,
                     const void* v_in) {
  if (!s || !k_in || !v_in) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  ST_TRY(kv_range_ok(s, layer, first_slot, n_rows));
  const dflash_config& c = s->m->cfg;
  const size_t plane = (size_t)c.n_kv_heads * s->cap * c.head_dim * s->m->esz;
  char* base = (char*)s->kv + (size_t)(2 * layer) * plane;
  launch_kv_copy(s->m->dt, base, s->cap, first_slot, const_cast<void*>(k_in), n_rows, c.n_kv_heads, c.head_dim, true,
                 false, s->stream);
  launch_kv_copy(s->m->dt, base + plane, s->cap, first_slot, const_cast<void*>(v_in), n_rows, c.n_kv_heads, c.head_dim,
                 true, true, s->stream);
  return launch_check("kv_import");
}

int dflash_timing_enable(dflash_model* m, int32_t on) {
  if (!m) return fail(DFLASH_ERR_INVALID_ARG, "null model");
  if (on) {
    CU_TRY(cudaDeviceSynchronize());
    m->recs.clear();
    m->ev_used = 0;
    m->launches = 0;
  }
  m->timing = on != 0;
  return DFLASH_OK;
}

int dflash_timing_read(dflash_model* m, dflash_kernel_time* out, int32_t max_entries, int32_t* n_entries) {
  if (!m || !out || !n_entries || max_entries < 0) return fail(DFLASH_ERR_INVALID_ARG, "null argument");
  CU_TRY(cudaDeviceSynchronize());
  dflash_kernel_time acc[kClasses + 1];
  memset(acc, 0, sizeof acc);
  for (int k = 0; k < kClasses; ++k) snprintf(acc[k].name, sizeof acc[k].name, "%s", kClassNames[k]);
  snprintf(acc[kClasses].name, sizeof acc[kClasses].name, "all");
  acc[kClasses].launches = m->launches;
  for (const auto& r : m->recs) {
    float ms = 0.f;
    CU_TRY(cudaEventElapsedTime(&ms, r.e0, r.e1));
    acc[r.cls].launches++;
    acc[r.cls].total_ms += ms;
    acc[r.cls].bytes += r.bytes;
    acc[r.cls].flops += r.flops;
  }
  int n = 0;
  for (int k = 0; k <= kClasses && n < max_entries; ++k)
    if (acc[k].launches) out[n++] = acc[k];
  *n_entries = n;
  return DFLASH_OK;
}

}  // extern "C"
