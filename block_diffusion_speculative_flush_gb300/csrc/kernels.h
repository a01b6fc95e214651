// Internal launch interface of the DFlash kernels (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfl {

enum class DT : int { F32 = 0, BF16 = 1 };

inline size_t dt_size(DT t) { return t == DT::F32 ? 4 : 2; }

// One row of a layer's fused QKV product: a context row being flushed or a
// block row being drafted.
struct RowMeta {
  int32_t sess;  // index into the call's per-session tables
  int32_t blk;   // block row index into the Q / gate buffers, -1 for context rows
  int64_t pos;   // absolute position; also the cache slot (modulo the ring)
};

// Per-session device tables of one batched call.
// Cache layout of one session, per layer l and KV head h: the K plane
// (2l)*Hkv + h holds [cap slots][d] (row per position) and the V plane
// (2l+1)*Hkv + h holds [d][cap slots] (V transposed, row per channel), so
// that a 64-position tile of either is a K-major operand tile for the
// tensor cores.
struct SessTables {
  void* const* kv;         // [B] session cache base: 2 * L * Hkv planes of cap * d elements
  const int64_t* cap;      // [B] cache slots (ring size when the draft has a window)
  const int64_t* frontier; // [B] F: position of the block's anchor row
  const int32_t* seq;      // [B] seq id used by the random streams
  const CUtensorMap* const* kvmaps;  // [B] -> {K planes, V^T planes} TMA maps (bf16, d = 128), or NULL
  // [B] lowest position whose K/V this forward writes (its context rows,
  // then the block), or NULL: every older row of the cache is left as it was
  const int64_t* fresh;
};

// One attention work item: keys [k0, k1) (positions) of one session / KV head.
struct AttnItem {
  int32_t sess, kvh;
  int64_t k0, k1;
};

struct AttnParams {
  int Hq, Hkv, d, nrows;    // nrows = n + 1 block rows per session
  int window, causal;
  int L, layer;
  float scale;
  // Split-key merge inside the attention kernel (tensor-core path): the
  // `cluster` key ranges of one (session, KV head) form a thread-block
  // cluster and merge their partials through distributed shared memory into
  // out (bf16 [rows][Hq][d], times gates [rows][Hq] when given).  1: partials
  // go to global memory for k_attn_combine.
  int cluster;
  void* out;
  const float* gates;
};

// --- portable kernels (any storage type) ----------------------------------
// src: [rows][K] device table, src[r * K + k] = tap k of context row r.
void launch_tap_norm(DT dt, const void* const* src, int rows, const void* aux, void* u, int K, int Ht,
                     float eps, cudaStream_t st);
// out[j] = rmsnorm(in[map(j)]) * g, in rows taken from in0 for map < rows0 else in1.
// map(j) = (j / a) * b + (j % a) + c.   in_f32: inputs are fp32, else storage type.
void launch_rmsnorm(DT dt, bool in_f32, const void* in0, int rows0, const void* in1, int64_t ld_in,
                    const void* g, void* out, int64_t ld_out, int rows, int H, int a, int b, int c, float eps,
                    cudaStream_t st);
// current[sess_map[j]] is the anchor of compact session j; ids outside
// [0, V) set bit 1 of *err and read row 0.
void launch_embed(DT dt, const void* E, const int32_t* current, const int32_t* sess_map, int mask_token, int V,
                  int B, int nrows, int H, void* h, int32_t* err, cudaStream_t st);
// table[m] = cos / sin of pos(m) * theta^(-2j/d), j < d/2: pos(m) = meta[m].pos,
// or first + m when meta is NULL (the model's table indexed by position).
void launch_rope_table(const RowMeta* meta, int64_t first, int M, int d, float theta, float2* table,
                       cudaStream_t st);
// Context-only forward: K (k norm, RoPE from the position table) and V of
// every row into the session caches, 32 rows of one KV head of one layer per
// CTA; the same bits as k_qkv_post writes for a context row.  Layer layer0 + z
// (z < layers) reads qkv + z * layer_stride, rows ldq apart, K of head h at
// column kcol0 + h d and V at vcol0 + h d, with gain k_norms[z] (a device table).
void launch_kv_ctx(DT dt, const float* qkv, int64_t ldq, int64_t kcol0, int64_t vcol0, int64_t layer_stride,
                   const RowMeta* meta, int M, const float2* rope, const void* const* k_norms, int Hkv, int d,
                   float eps, SessTables tabs, int layer0, int layers, cudaStream_t st);
// Every layer's norm of the same rows: out + l * out_layer = rmsnorm(in; gains[l])
// (gains: a device table), the sums in launch_rmsnorm's order.
void launch_rmsnorm_layers(DT dt, const void* in, int64_t ld_in, const void* const* gains, void* out, int64_t ld_out,
                           int64_t out_layer, int rows, int layers, int H, float eps, cudaStream_t st);
// Returns the number of kernels launched (2 from kVApartRows rows on: the V
// rows go to the transposed cache planes 32 rows at a time).
constexpr int kVApartRows = 64;
// rope: the model's table indexed by position ([pos][d/2]).
// early: the kernel before this one (the QKV product) lets dependants start
// only after its own wait, so the row and session tables are read before this
// kernel's wait
int launch_qkv_post(DT dt, const float* qkv, int64_t ldq, const RowMeta* meta, int M, const float2* rope,
                    const void* q_norm, const void* k_norm, int Hq, int Hkv, int d, int gated, float eps,
                    SessTables tabs, int L, int layer, void* Q, float* G, cudaStream_t st, int early = 0);
void launch_attention_simt(DT dt, const void* Q, const AttnItem* items, int n_items, SessTables tabs,
                           AttnParams p, float* part, cudaStream_t st);
// bf16 block attention on tcgen05 tensor cores (key ranges must start on a
// multiple of 64); false if the shape is not supported (head_dim other than
// 128, more than 128 query rows per KV head, no tensor maps).
// Largest cluster of key ranges merged in-kernel (non-portable size).
constexpr int kAttnMaxCluster = 16;
// Returns 0 if the shapes need the CUDA-core path, 1 if partials were written
// for k_attn_combine, 2 if the output was merged in-kernel (p.cluster > 1).
int launch_attention_tc(const void* Q, const AttnItem* items, int n_items, SessTables tabs, AttnParams p, float* part,
                        int* err, cudaStream_t st);
// max_splits: the largest item count of a session (0: not known); up to 32
// the merge runs in one pass for d = 128.  early: the partials come from
// k_attn_tc, which lets this kernel start only after its own wait, so the
// item tables and gates are read before this kernel's wait.
void launch_attention_combine(DT dt, const float* part, const int32_t* item_first, const int32_t* item_count,
                              int B, AttnParams p, const float* G, void* O, cudaStream_t st, int max_splits = 0,
                              int early = 0);
void launch_residual(DT dt, void* h, const float* delta, int64_t ld_delta, int rows, int H, cudaStream_t st);
void launch_swiglu(DT dt, const float* gu, int64_t ld, int rows, int I, int up_offset, void* a,
                   cudaStream_t st);
void launch_gemm_simt(DT dt, const void* X, int64_t ldx, const void* W, int64_t ldw, float* Y, int64_t ldy,
                      int M, int N, int K, cudaStream_t st);
// Rows between a cache plane set and a flat [Hkv][n][d] buffer.  to_cache:
// flat -> cache.  transposed: the cache planes are V^T ([d][cap]).
void launch_kv_copy(DT dt, void* cache, int64_t cap, int64_t first, void* flat, int n_rows, int Hkv, int d,
                    bool to_cache, bool transposed, cudaStream_t st);

// Sampling: per (row, chunk) partials over a row of logits, then a merge.
struct SampleArgs {
  const void* logits;      // [rows][V] fp32 or bf16 (in_bf16)
  int64_t ld;
  int rows, V;
  int in_bf16;
  float temperature;       // 0: argmax
  int gumbel;              // add the draft's Gumbel noise (T > 0)
  uint64_t seed;
  uint32_t rnd;
  int rows_per_seq;        // rows of one session (seq id = row / rows_per_seq)
  int row_offset;          // Philox row of a session's first row
  const int32_t* seq_ids;  // [B] seq id per session
  const int32_t* out_map;  // [B] output row block of each session (NULL: identity)
  int32_t* err;            // bit 16: a row had no comparable score (non-finite logits)
  // optional per-session rows (fp32 logits only): row r of session b = r / rows_per_seq
  const float* const* seq_logits;  // [B] logits of the session's rows (NULL: logits + row * ld)
  int32_t* const* sess_tok;        // [B] also write the token of each row here
  float* const* sess_lse;          // [B] also write the log-sum-exp of each row here
  // truncated distributions: row r keeps entry v iff order_key(l_v / T, v) >= cut[r]
  // (NULL: every entry); the statistics and the draw then run over the kept entries
  const uint64_t* cut;
};

// The sampler's truncation of one session's distributions: top_k (0: none,
// else at most kTruncMaxK), then top_p and min_p inside the top_k.
struct Trunc {
  int32_t top_k;
  float top_p, min_p;
  int32_t pad;
};
constexpr int kTruncMaxK = 1024;
// cut[row] for the rows of a.rows (session of a row: row / a.rows_per_seq,
// with its Trunc in tr[]); sessions with top_k == 0 get cut 0.  Also into
// sess_cut[b][row % rows_per_seq] when given.
void launch_trunc_cut(const SampleArgs& a, const Trunc* tr, uint64_t* cut, uint64_t* const* sess_cut,
                      cudaStream_t st);
// Vocabulary entries per CTA of the sampling partials: 16384 when the rows
// give every SM at least eight such CTAs (the per-CTA merge then costs less
// next to the entries), else 4096 so that a few rows still spread over the
// SMs.  Both are multiples of 1024.
constexpr int kSampleChunkSmall = 4096, kSampleChunkLarge = 16384;
inline int sample_chunk(int64_t rows, int V, int num_sms) {
  const int64_t big = rows * ((V + kSampleChunkLarge - 1) / kSampleChunkLarge);
  return big >= 8 * (int64_t)num_sms ? kSampleChunkLarge : kSampleChunkSmall;
}
void launch_sample_partials(const SampleArgs& a, int chunk, float4* part, cudaStream_t st);
// Writes tok[row], q[row] (probability of the token at T), lse[row] (log-sum-exp of logits/T).
void launch_sample_combine(const SampleArgs& a, int chunks, const float4* part, int32_t* tok, float* qtok,
                           float* lse, cudaStream_t st);

struct VerifyArgs {
  const void* target;      // [B][n+1][V]
  int in_bf16;
  int B, n, V;
  float temperature;
  uint64_t seed;
  uint32_t rnd;
  const int32_t* seq_ids;  // [B]
  const int32_t* draft;    // [B][n] tokens under test
  const float* lse_t;      // [B][n+1] target log-sum-exp of logits/T
  const int32_t* amax_t;   // [B][n+1] target argmax
  const float* const* dlogits;  // [B] -> [n][V] fp32 draft logits of the last proposal
  const float* const* dlse;     // [B] -> [n]
  const int32_t* const* dtok;   // [B] -> [n] proposed tokens
  const float* dtemp;           // [B] temperature of that proposal
  int32_t* accept;              // [B]
  int32_t* bonus;               // [B]
  long long* const* accepted_total;  // [B] -> running counter of each session
  int32_t* err;                 // bit 2: a draft token id outside [0, V)
  int32_t* rej;                 // [B] scratch: first rejected position (0: none)
  // truncated distributions (NULL: full): the cut of each target row, and of
  // each session's proposal rows (dcut[b] NULL: that proposal was not truncated)
  const uint64_t* cut_t;        // [B][n+1]
  const uint64_t* const* dcut;  // [B] -> [n]
  // DFlash2 proposals (NULL, or cand_ids[b] NULL: q from the draft logits):
  // q_i is the candidate distribution of position i, ncand ids and probabilities
  const int32_t* const* cand_ids;   // [B] -> [n][ncand]
  const float* const* cand_probs;   // [B] -> [n][ncand]
  int ncand;
};
// Bonus-draw partial of one vocabulary chunk of one session.
struct VerifyPart {
  float rsum;      // sum of max(0, p - q)
  float rv;        // best log(max(0, p - q)) + Gumbel
  int32_t ri;
  float pv;        // best log p + Gumbel
  int32_t pi;
};
// T > 0: one grid of (session, vocabulary chunk) CTAs for the bonus draw,
// then the per-session finish; T == 0: the finish alone.  part holds
// B * verify_bonus_chunks(V) entries.
constexpr int kVerifyBonusChunk = 1024;
inline int verify_bonus_chunks(int V) { return (V + kVerifyBonusChunk - 1) / kVerifyBonusChunk; }
void launch_verify_accept(const VerifyArgs& a, VerifyPart* part, cudaStream_t st);

// The sampler's penalties of one session over a committed token history:
// an id seen c > 0 times has a positive logit divided by `repeat` and a
// non-positive one multiplied by it, then loses `presence` once and
// `frequency` c times.  n_hist == 0: no penalties for this session.
struct Penalty {
  float repeat, presence, frequency;
  int32_t n_hist;
  const int32_t* hist;  // device [n_hist] token ids
};
constexpr int kMaxPenaltyHistory = 4096;
// Draft rows, in place: rows_per_seq rows of session b (rows[b] + i * ld)
// get b's penalties; every row of a block sees the same history.  One CTA per
// session.  Ids outside [0, V) are ignored.
void launch_penalize_rows(const Penalty* pen, float* const* rows, int rows_per_seq, int64_t ld, int V, int B,
                          cudaStream_t st);
// Target rows of verify: out [B][n+1][V] fp32 = target (fp32, or bf16 when
// in_bf16) with row r of session b penalised over b's history plus the draft
// tokens draft[b][0..r).  One CTA per row.
void launch_penalize_target(const Penalty* pen, const void* target, int in_bf16, float* out, const int32_t* draft,
                            int B, int n, int V, cudaStream_t st);

// --- DFlash2 ---------------------------------------------------------------
constexpr int kMaxConvTaps = 8;
constexpr int kMaxCandidates = 32;
constexpr int kDflash2Depth = 7;  // dflash.go dflash2Depth: a DFlash2 session's fixed draft length
// h[row] += sum over taps j <= row % nrows of softmax_j(a[row][g][.]) * x[row - j],
// channel c in group g = c / (H / G); a: [rows][G * taps] fp32, x: the
// normalised rows in the storage type.  One CTA per row.
void launch_dynconv(DT dt, void* h, const void* x, const float* a, int rows, int nrows, int H, int G, int taps,
                    cudaStream_t st);
// The kc largest logits of each of n_rows rows (row r: rows[r / rows_per_seq]
// + (r % rows_per_seq) * ld) in the sampler's order: ids and logits
// [n_rows][kc]; part holds n_rows * topk_chunks(V) * kc keys.
int topk_chunks(int V);
void launch_topk_candidates(const float* const* rows, int rows_per_seq, int64_t ld, int V, int kc, int n_rows,
                            uint64_t* part, int32_t* ids, float* logit, cudaStream_t st);
struct SelectArgs {
  int B, n, kc, rank, V;
  float temperature;
  uint64_t seed;
  uint32_t rnd;
  const int32_t* current;    // [caller batch] anchors
  const int32_t* sess_map;   // [B] caller index of each session
  const int32_t* seq_ids;    // [B]
  const void* sel_prev;      // [V][rank] A, storage type
  const void* sel_next;      // [V][rank] B
  const int32_t* cand_ids;   // [B * n][kc]
  const float* cand_logit;   // [B * n][kc]
  int32_t* const* sess_tok;  // [B] -> [n]
  int32_t* const* sess_ids;  // [B] -> [n][kc]
  float* const* sess_probs;  // [B] -> [n][kc]
  int32_t* out_tokens;       // [caller batch][n]
  float* out_q;              // [caller batch][n]
  int32_t* err;              // bit 1: an anchor outside [0, V)
};
void launch_select(DT dt, const SelectArgs& a, cudaStream_t st);

// --- tensor-core path (bf16, sm_103a) --------------------------------------
struct TcGemmPlan;  // opaque, defined in gemm_tc.cu

// Largest per-call table that travels as a kernel parameter.
constexpr int kTableParamMax = 31744;
// Writes bytes (<= kTableParamMax) of host data to dst with a one-CTA kernel
// in the launch chain; returns -1 if the table is too large.
int launch_table_write(void* dst, const void* src, size_t bytes, cudaStream_t st);

// The target's taps of one committed run: K separate buffers (passed by value).
constexpr int kMaxTaps = 8;
struct TapSrc {
  const char* p[kMaxTaps];
};
// Row r of tap k (src.p[k] + r * src_ld bytes, tap_bytes long) to dst + r * dst_ld + k * tap_bytes.
void launch_copy_taps(void* dst, int64_t dst_ld, const TapSrc& src, int K, int64_t src_ld, int64_t tap_bytes, int rows,
                      cudaStream_t st);
// rows x row_bytes from src (row stride src_ld bytes) to dst (dst_ld bytes), as a kernel.
// Several row copies in one launch: copy i moves rows[i] rows of row_bytes
// bytes from src[i] (rows src_ld[i] bytes apart) to dst[i] (rows packed).
// The table travels as the kernel's parameter.
constexpr int kMaxRowCopies = 128;
struct RowCopies {
  char* dst[kMaxRowCopies];
  const char* src[kMaxRowCopies];
  int64_t src_ld[kMaxRowCopies];
  int32_t rows[kMaxRowCopies];
  int32_t n;
  int64_t row_bytes;
};
void launch_copy_rows_batch(const RowCopies& t, cudaStream_t st);
void launch_copy_rows(void* dst, int64_t dst_ld, const void* src, int64_t src_ld, int64_t row_bytes, int rows,
                      cudaStream_t st);

}  // namespace dfl
