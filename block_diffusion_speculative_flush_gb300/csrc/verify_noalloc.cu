// Speculative verification that allocates no device memory.
//
// dflash_verify keeps its row statistics, bonus-draw partials and per-call
// tables in a model workspace that grows with cudaMalloc the first time a
// larger batch or vocabulary shows up.  Some callers cannot allow that: a
// serving runtime that hands out all device memory up front under a fixed
// budget, or a decode loop that must not meet cudaMalloc's implicit device
// synchronisation between two rounds.  This variant runs the same kernels on
// a fixed scratch area that lives in the library image itself (a file-scope
// __device__ array, present on every GPU that loads the library until the
// process exits), so it never calls cudaMalloc, cudaFree or an allocating
// library routine.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "dflash.h"
#include "kernels.h"

using namespace dfl;

// Accessors into the session, the model's measurement state and the error
// string (dflash_capi.cu; not exported).
extern "C" int dflash__session_proposal(const dflash_session* s, const float** logits, const float** lse,
                                        const int32_t** tokens, float* temperature, int32_t* n,
                                        long long** accepted, void** stream, int32_t* vocab, int32_t* draft_limit,
                                        int32_t** err, const void** model);
extern "C" int dflash__session_truncation(const dflash_session* s, Trunc* trunc, const uint64_t** proposal_cut);
extern "C" int dflash__session_device(const dflash_session* s);
extern "C" int dflash__session_penalties(const dflash_session* s);
extern "C" int dflash__session_candidates(const dflash_session* s, const int32_t** ids, const float** probs,
                                          int32_t* kc);
extern "C" long long dflash__verify_timing_begin(const void* model, double bytes, double flops, void* stream);
extern "C" void dflash__verify_timing_end(const void* model, long long idx, void* stream);
extern "C" void dflash__count_launches(const void* model, int n);
extern "C" int dflash__set_error(int code, const char* msg);

namespace {

// Size of the static scratch: 4 MiB.  It holds, per call, the per-session
// pointer tables (at most kMaxBatch sessions), the row statistics of the
// batch * (n + 1) target rows (one float4 partial per vocabulary chunk of
// the sampling partials, then log-sum-exp and argmax) and the bonus-draw
// partials.
constexpr size_t kScratchBytes = 4u << 20;
constexpr int kMaxBatch = 128;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};

// Device address of the scratch on device `dev`, looked up once per device
// with that device current (the host-side symbol is only a stand-in, not a
// device address).  The caller has made `dev` current.
int scratch_on_device(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return dflash__set_error(DFLASH_ERR_CUDA, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_verify_scratch);
    if (e != cudaSuccess) return dflash__set_error(DFLASH_ERR_CUDA, cudaGetErrorString(e));
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return DFLASH_OK;
}

// Makes the sessions' device current for the life of the object and puts
// the caller's device back afterwards.
struct DeviceScope {
  int prev = -1;
  bool ok = false;
  explicit DeviceScope(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = prev == dev || cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceScope() {
    if (ok && prev >= 0) cudaSetDevice(prev);
  }
};

constexpr size_t up16(size_t x) { return (x + 15) & ~(size_t)15; }

}  // namespace

extern "C" DFLASH_API int dflash_verify_noalloc(dflash_session* const* s, int32_t batch, const void* target_logits,
                                                int32_t logits_dtype, const int32_t* draft_tokens, int32_t n,
                                                float temperature, uint64_t seed, uint64_t round, int32_t* out_accept,
                                                int32_t* out_bonus) {
  char msg[256];
  if (!s || batch < 1) return dflash__set_error(DFLASH_ERR_INVALID_ARG, "null session array or batch < 1");
  if (batch > kMaxBatch) {
    snprintf(msg, sizeof msg, "batch %d exceeds the %d sessions the static verify scratch holds", batch, kMaxBatch);
    return dflash__set_error(DFLASH_ERR_CAPACITY, msg);
  }
  if (!target_logits || !draft_tokens || !out_accept || !out_bonus)
    return dflash__set_error(DFLASH_ERR_INVALID_ARG, "null pointer");
  if (logits_dtype != DFLASH_DTYPE_F32 && logits_dtype != DFLASH_DTYPE_BF16)
    return dflash__set_error(DFLASH_ERR_INVALID_ARG, "logits_dtype");
  if (!(temperature >= 0.f) || std::isinf(temperature)) return dflash__set_error(DFLASH_ERR_INVALID_ARG, "temperature");

  // host copies of the per-session tables (fixed-size, on the stack)
  const float* dl[kMaxBatch];
  const float* dlse[kMaxBatch];
  const int32_t* dtok[kMaxBatch];
  float dT[kMaxBatch];
  long long* acc[kMaxBatch];
  int32_t seq[kMaxBatch];
  Trunc trv[kMaxBatch];
  const uint64_t* dcut[kMaxBatch];
  const int32_t* cid[kMaxBatch];
  const float* cpr[kMaxBatch];
  int32_t kc = 0;
  bool any_trunc = false, any_dcut = false;
  void* stream = nullptr;
  int32_t V = 0, limit = 0;
  int32_t* err = nullptr;
  const void* model = nullptr;
  for (int b = 0; b < batch; ++b) {
    if (!s[b]) return dflash__set_error(DFLASH_ERR_INVALID_ARG, "null session");
    int32_t pn = 0, vb = 0, lim = 0;
    int32_t* eb = nullptr;
    void* st = nullptr;
    const void* mb = nullptr;
    dflash__session_proposal(s[b], &dl[b], &dlse[b], &dtok[b], &dT[b], &pn, &acc[b], &st, &vb, &lim, &eb, &mb);
    if (b == 0) {
      stream = st;
      V = vb;
      limit = lim;
      err = eb;
      model = mb;
    } else if (mb != model) {
      return dflash__set_error(DFLASH_ERR_INVALID_ARG, "sessions of different models in one batch");
    }
    for (int j = 0; j < b; ++j)
      if (s[j] == s[b]) return dflash__set_error(DFLASH_ERR_INVALID_ARG, "session repeated in batch");
    if (temperature > 0.f && pn != n) {
      snprintf(msg, sizeof msg, "session %d has no proposal of %d tokens to verify against", b, n);
      return dflash__set_error(DFLASH_ERR_STATE, msg);
    }
    if (dflash__session_penalties(s[b]))
      return dflash__set_error(DFLASH_ERR_INVALID_ARG,
                               "a session has penalties set: their penalised target rows need dflash_verify's workspace");
    seq[b] = b;
    dflash__session_candidates(s[b], &cid[b], &cpr[b], &kc);
    dflash__session_truncation(s[b], &trv[b], &dcut[b]);
    any_trunc = any_trunc || (temperature > 0.f && trv[b].top_k > 0);
    any_dcut = any_dcut || (temperature > 0.f && dcut[b]);
  }
  if (n < 1 || n > limit) return dflash__set_error(DFLASH_ERR_INVALID_ARG, "n out of range");

  // scratch layout
  const int rows = batch * (n + 1);
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dflash__session_device(s[0])) != cudaSuccess)
    return dflash__set_error(DFLASH_ERR_CUDA, "cannot read the sessions' device");
  const int chunk = sample_chunk(rows, V, sms), chunks = (V + chunk - 1) / chunk;
  size_t off = 0;
  const size_t o_dl = off;
  off = up16(off + batch * sizeof(void*));
  const size_t o_dlse = off;
  off = up16(off + batch * sizeof(void*));
  const size_t o_dtok = off;
  off = up16(off + batch * sizeof(void*));
  const size_t o_dT = off;
  off = up16(off + batch * sizeof(float));
  const size_t o_acc = off;
  off = up16(off + batch * sizeof(void*));
  const size_t o_seq = off;
  off = up16(off + batch * sizeof(int32_t));
  const size_t o_trunc = off;
  off = up16(off + batch * sizeof(Trunc));
  const size_t o_dcut = off;
  off = up16(off + batch * sizeof(void*));
  const size_t o_cid = off;
  off = up16(off + batch * sizeof(void*));
  const size_t o_cpr = off;
  off = up16(off + batch * sizeof(void*));
  const size_t tables_end = off;
  const size_t o_cut = off;
  off = up16(off + (any_trunc ? (size_t)rows * sizeof(uint64_t) : 0));
  const size_t o_part = off;
  off = up16(off + (size_t)rows * chunks * sizeof(float4));
  const size_t o_amax = off;
  off = up16(off + (size_t)rows * sizeof(int32_t));
  const size_t o_lse = off;
  off = up16(off + (size_t)rows * sizeof(float));
  const size_t o_bonus = off;
  off = up16(off + (size_t)batch * verify_bonus_chunks(V) * sizeof(VerifyPart));
  const size_t o_rej = off;
  off = up16(off + (size_t)batch * sizeof(int32_t));
  if (off > kScratchBytes) {
    snprintf(msg, sizeof msg,
             "verify of %d sessions x %d rows x %d vocabulary chunks needs %zu bytes of scratch; the static "
             "scratch holds %zu",
             batch, n + 1, chunks, off, kScratchBytes);
    return dflash__set_error(DFLASH_ERR_CAPACITY, msg);
  }
  // the scratch and the launches belong to the sessions' device, whatever
  // device the caller has current
  const int dev = dflash__session_device(s[0]);
  DeviceScope scope(dev);
  if (!scope.ok) return dflash__set_error(DFLASH_ERR_CUDA, "cannot make the sessions' device current");
  void* scratch = nullptr;
  int rc = scratch_on_device(dev, &scratch);
  if (rc != DFLASH_OK) return rc;
  char* base = (char*)scratch;
  cudaStream_t st = (cudaStream_t)stream;

  // tables: staged on the stack, then written by a one-CTA kernel that takes
  // them as its parameter, in stream order (no host-to-device copy, so the
  // call never waits for the stream; the block is at most ~8 KB)
  alignas(16) char host[up16(kMaxBatch * sizeof(void*)) * 7 + up16(kMaxBatch * sizeof(float)) +
                        up16(kMaxBatch * sizeof(int32_t)) + up16(kMaxBatch * sizeof(Trunc))];
  static_assert(sizeof(host) <= (size_t)kTableParamMax, "verify tables exceed a kernel parameter block");
  memcpy(host + o_dl, dl, batch * sizeof(void*));
  memcpy(host + o_dlse, dlse, batch * sizeof(void*));
  memcpy(host + o_dtok, dtok, batch * sizeof(void*));
  memcpy(host + o_dT, dT, batch * sizeof(float));
  memcpy(host + o_acc, acc, batch * sizeof(void*));
  memcpy(host + o_seq, seq, batch * sizeof(int32_t));
  memcpy(host + o_trunc, trv, batch * sizeof(Trunc));
  memcpy(host + o_dcut, dcut, batch * sizeof(void*));
  memcpy(host + o_cid, cid, batch * sizeof(void*));
  memcpy(host + o_cpr, cpr, batch * sizeof(void*));
  const double tbytes = (double)rows * V * (logits_dtype == DFLASH_DTYPE_BF16 ? 2 : 4) + (double)batch * V * 4;
  const long long timed = dflash__verify_timing_begin(model, tbytes, 4.0 * rows * V, stream);
  if (launch_table_write(base, host, tables_end, st)) {
    dflash__verify_timing_end(model, timed, stream);
    return dflash__set_error(DFLASH_ERR_CUDA, "verify table write launch");
  }
  cudaError_t e = cudaSuccess;
  // nothing in the scratch has to start at zero: every partial, statistic and
  // the rejection index are written before they are read

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
  sa.err = err;
  float4* part = (float4*)(base + o_part);
  int32_t* amax = (int32_t*)(base + o_amax);
  float* lse = (float*)(base + o_lse);
  if (any_trunc) {
    launch_trunc_cut(sa, (const Trunc*)(base + o_trunc), (uint64_t*)(base + o_cut), nullptr, st);
    sa.cut = (const uint64_t*)(base + o_cut);
  }
  launch_sample_partials(sa, chunk, part, st);
  launch_sample_combine(sa, chunks, part, amax, nullptr, lse, st);
  VerifyArgs va{};
  va.target = target_logits;
  va.in_bf16 = sa.in_bf16;
  va.B = batch;
  va.n = n;
  va.V = V;
  va.temperature = temperature;
  va.seed = seed;
  va.rnd = (uint32_t)round;
  va.seq_ids = (const int32_t*)(base + o_seq);
  va.draft = draft_tokens;
  va.lse_t = lse;
  va.amax_t = amax;
  va.dlogits = (const float* const*)(base + o_dl);
  va.dlse = (const float* const*)(base + o_dlse);
  va.dtok = (const int32_t* const*)(base + o_dtok);
  va.dtemp = (const float*)(base + o_dT);
  va.accept = out_accept;
  va.bonus = out_bonus;
  va.accepted_total = (long long* const*)(base + o_acc);
  va.err = err;
  va.rej = (int32_t*)(base + o_rej);
  va.cut_t = sa.cut;
  va.dcut = any_dcut ? (const uint64_t* const*)(base + o_dcut) : nullptr;
  if (kc > 0) {
    va.cand_ids = (const int32_t* const*)(base + o_cid);
    va.cand_probs = (const float* const*)(base + o_cpr);
    va.ncand = kc;
  }
  launch_verify_accept(va, (VerifyPart*)(base + o_bonus), st);
  dflash__verify_timing_end(model, timed, stream);
  dflash__count_launches(model, 3 + (any_trunc ? 1 : 0) + (temperature > 0.f ? 2 : 1));
  e = cudaGetLastError();
  if (e != cudaSuccess) return dflash__set_error(DFLASH_ERR_CUDA, cudaGetErrorString(e));
  return DFLASH_OK;
}
