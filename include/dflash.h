/*
 * dflash.h — C ABI of the GB300-native DFlash block-diffusion draft round.
 *
 * One draft round has four parts, each an entry point below:
 *   1. committed / flush:  buffered target feature rows (the concatenated
 *      hidden taps of the target's layers) pass aux_hidden_norms, fc and
 *      hidden_norm, then each layer's input norm and a K/V-only projection,
 *      and land in the draft K/V cache at their own slots.
 *   2. propose:  one forward of [anchor, mask x n] against that cache; the
 *      anchor row is dropped, rows 1..n are unembedded and sampled from one
 *      batched distribution.
 *   3. commit_block:  the block's rows are rewound out of the cache before
 *      any write; a committed run that starts past the buffered frontier is
 *      refused as a context gap.
 *   4. verify:  accepted prefix plus a bonus token from the target logits
 *      and the proposal probabilities.
 *
 * Sources (web pages): "Ollama DFlash block-diffusion draft model in
 * mlxrunner" (Facts); ollama mlxrunner/dflash.go (gitea mirror: committed,
 * settle, close, takePending, commitBlock, flush, propose, selectBlock, and
 * the DFlash2 commit note); mlxcel PR #1771 "feat(speculative): add the
 * Laguna DFlash drafter" (summary, review commits, "Where the landed code
 * and the issue text disagree").
 *
 * Conventions
 *   - Every call returns DFLASH_OK (0) or a negative status.  On error no
 *     session or model state changes, and dflash_last_error() returns a
 *     message for the calling thread.  Nothing aborts the process (the
 *     pages panic on a context gap; here it is a status).
 *   - Pointers are DEVICE pointers unless marked (host).  Device work is
 *     enqueued on the session's stream (batched calls: the stream of the
 *     first session) and is asynchronous unless stated otherwise.
 *   - Matrices are row-major [out, in]; activations are row-major
 *     [rows, width].  Storage type is fp32 or bf16 per the model config.
 *   - A batched call takes a HOST array of sessions of one model.  The
 *     random streams use the session's index in that array as its seq id.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define DFLASH_OK 0
#define DFLASH_ERR_INVALID_ARG (-1) /* null pointer, negative size, bad enum */
#define DFLASH_ERR_SHAPE (-2)       /* config or weight geometry inconsistent / unsupported */
#define DFLASH_ERR_CONTEXT_GAP (-3) /* committed run starts past the buffered frontier */
#define DFLASH_ERR_CAPACITY (-4)    /* would exceed the session's max_ctx */
#define DFLASH_ERR_CUDA (-5)        /* a CUDA runtime call or launch failed */
#define DFLASH_ERR_OOM (-6)         /* device allocation failed */
#define DFLASH_ERR_STATE (-7)       /* call not valid in this state (e.g. verify without propose) */
#define DFLASH_ERR_DEVICE (-8)      /* a kernel reported a bad input (see dflash_device_status) */

#define DFLASH_DTYPE_F32 0
#define DFLASH_DTYPE_BF16 1

/* Feature rows held between flushes (dflash.go dflashPendingFlushTokens). */
#define DFLASH_PENDING_FLUSH_TOKENS 256

/* dflash_config.flags */
#define DFLASH_FLAG_SIMT_GEMM 1u /* bf16 models: use the CUDA-core GEMM instead of tcgen05 (testing) */

typedef struct dflash_model dflash_model;
typedef struct dflash_session dflash_session;

/* Draft geometry and block parameters.  Bounds checked by dflash_model_create
 * (the Laguna PR treats the drafter config as untrusted): block_size in
 * 2..512, window 0 (full attention) or 2..2^20, head_dim 64 or 128,
 * n_q_heads a multiple of n_kv_heads, bf16 widths multiples of 64, n_taps
 * at most 8. */
typedef struct dflash_config {
  int32_t dtype;           /* DFLASH_DTYPE_F32 or DFLASH_DTYPE_BF16 */
  int32_t n_taps;          /* K: tapped target layers */
  int32_t target_hidden;   /* H_t: width of one tap; a feature row is K*H_t wide */
  int32_t hidden;          /* H */
  int32_t n_layers;        /* L */
  int32_t n_q_heads;       /* Hq */
  int32_t n_kv_heads;      /* Hkv */
  int32_t head_dim;        /* d */
  int32_t intermediate;    /* I, SwiGLU width */
  int32_t vocab;           /* V */
  int32_t block_size;      /* B_s; draft limit is B_s - 1 */
  int32_t mask_token;      /* m */
  int32_t window;          /* W: a query at p sees keys r with p - r < W; 0 = unlimited */
  int32_t causal_block;    /* 1: causal inside the block; 0: bidirectional */
  int32_t gated_attention; /* 1: per-head sigmoid gate from g_proj on the attention output */
  uint32_t flags;          /* DFLASH_FLAG_* */
  float rope_theta;        /* RoPE base (rotate-half pairs j, j + d/2) */
  float rms_eps;           /* RMSNorm epsilon */
  /* DFlash2 (ollama dflash.go, the DFlash2 commit note): block-local dynamic
   * convolutions and a candidate selector.  variant DFLASH_VARIANT_DFLASH (0)
   * ignores the three fields after it.  For DFLASH_VARIANT_DFLASH2:
   * conv_taps in 1..8 (the convolution's width), sel_rank in 1..256 (the
   * selector tables' rank), sel_candidates in 1..32 (candidates per
   * position, at most vocab); the pages give none of the three. */
  int32_t variant;
  int32_t conv_taps;
  int32_t sel_rank;
  int32_t sel_candidates;
} dflash_config;

#define DFLASH_VARIANT_DFLASH 0
#define DFLASH_VARIANT_DFLASH2 1
#define DFLASH2_DEPTH 7 /* dflash.go dflash2Depth: a DFlash2 proposal's fixed length */

/* Per-layer weights, device pointers in the storage type.  Borrowed: they
 * must stay valid until dflash_model_destroy. */
typedef struct dflash_layer_weights {
  const void* in_norm;   /* [H] input_layernorm, applied to context and block rows */
  const void* w_qkv;     /* [(Hq + 2 Hkv) d, H] fused projection, rows q | k | v */
  const void* q_norm;    /* [d] per-head RMSNorm of q */
  const void* k_norm;    /* [d] per-head RMSNorm of k */
  const void* w_g;       /* [Hq, H] g_proj (gated_attention) or NULL */
  const void* w_o;       /* [H, Hq d] */
  const void* post_norm; /* [H] */
  const void* w_gate;    /* [I, H] */
  const void* w_up;      /* [I, H] */
  const void* w_down;    /* [H, I] */
  /* DFlash2 only (NULL otherwise): the layer's dynamic convolution, after the
   * attention residual.  x = RMSNorm(h; conv_norm); row i of the block adds
   * sum_j w_ij * x_{i-j} over j < conv_taps (rows before the anchor's count
   * as zero), w_i = softmax over the taps of (w_dc x_i) taken per channel
   * group, one group of H / Hq channels per query head. */
  const void* conv_norm; /* [H] */
  const void* w_dc;      /* [Hq conv_taps, H]: row g * conv_taps + j is tap j of group g */
} dflash_layer_weights;

typedef struct dflash_weights {
  const void* aux_norms;   /* [K, H_t] one RMSNorm gain per tap (aux_hidden_norms) */
  const void* w_fc;        /* [H, K H_t] */
  const void* hidden_norm; /* [H] */
  const void* final_norm;  /* [H] */
  const void* embed;       /* [V, H] token embeddings of the block */
  const void* unembed;     /* [V, H] */
  const dflash_layer_weights* layers; /* (host) array of n_layers */
  /* DFlash2 only (NULL otherwise): the selector's tables.  The candidates of
   * position i are the sel_candidates largest logits of block row i (value
   * descending, then id), scored logit + <sel_prev[prev], sel_next[c]> with
   * prev the token chosen at position i - 1 (the anchor for the first). */
  const void* sel_prev;  /* [V, sel_rank] */
  const void* sel_next;  /* [V, sel_rank] */
} dflash_weights;

typedef struct dflash_counters {
  int64_t rounds;       /* proposals made */
  int64_t proposed;     /* tokens proposed */
  int64_t accepted;     /* tokens accepted by dflash_verify (reads device memory: synchronises) */
  int64_t flushes;      /* context-only forwards */
  int64_t flushed_rows; /* feature rows written to the cache */
} dflash_counters;

/* Message of the calling thread's last failed call ("" if none). */
DFLASH_API const char* dflash_last_error(void);
/* ABI version (major * 100 + minor). */
DFLASH_API int dflash_version(void);

/* Validates the config and weight geometry and builds the model.  *out is
 * owned by the caller and released with dflash_model_destroy.
 * Errors: INVALID_ARG, SHAPE (out-of-bounds config, e.g. block_size outside
 * 2..512 or a head geometry that does not divide), OOM, CUDA. */
DFLASH_API int dflash_model_create(const dflash_config* cfg /*host*/, const dflash_weights* w /*host*/,
                        dflash_model** out /*host*/);
DFLASH_API int dflash_model_destroy(dflash_model* m);

/* blockSize - 1 (dflash.go draftLimit); negative status on a null model. */
DFLASH_API int dflash_draft_limit(const dflash_model* m);

/* Reads (synchronously) and clears the model's device error word: 0 if no
 * kernel saw a bad input since the last call, else DFLASH_ERR_DEVICE with
 * the reason in dflash_last_error (token id out of range, ...). */
DFLASH_API int dflash_device_status(dflash_model* m);

/* Opens a session whose cache already holds `restored_offset` context rows
 * (dflash.go open: ctxOffset = the caches' restored offset; the rows are
 * supplied with dflash_kv_import).  max_ctx bounds the context rows the
 * session may ever hold (its cache holds max_ctx + block_size slots, or a
 * ring of window + block_size slots when the draft has a window).
 * stream: a cudaStream_t (NULL = legacy default stream). */
DFLASH_API int dflash_open(dflash_model* m, int64_t restored_offset, int64_t max_ctx, void* stream,
                dflash_session** out /*host*/);

/* dflash.go committed: `features` holds n_rows target feature rows
 * [n_rows, K*H_t] (row_stride elements apart) for tokens at positions
 * position..position+n_rows-1.  Rows the session already holds (a
 * restored prefix) are skipped; start = F + P - position < 0 is a context
 * gap (DFLASH_ERR_CONTEXT_GAP, nothing changes).  New rows are staged (a
 * device copy made on the stream, so `features` may be reused once the
 * stream reaches this call); when the held rows reach
 * DFLASH_PENDING_FLUSH_TOKENS they are flushed in one context-only forward.
 * Errors: INVALID_ARG, CONTEXT_GAP, CAPACITY (F + P + new rows > max_ctx). */
DFLASH_API int dflash_committed(dflash_session* s, const void* features, int64_t row_stride, int32_t n_rows,
                     int64_t position);
/* The same run given as the target's n_taps hidden states in separate
 * buffers: taps is a host array of n_taps device pointers, tap k being
 * [n_rows, H_t] with rows row_stride elements apart.  The rows are read where
 * they are (a flush reads them in place; staged rows are copied once, tap by
 * tap), so a target that keeps its captured hidden states apart needs no
 * concatenation (the Laguna PR paid a copy of [1, T, 5 * hidden] per round).
 * Same state changes and errors as dflash_committed; a null tap pointer is
 * INVALID_ARG. */
DFLASH_API int dflash_committed_taps(dflash_session* s, const void* const* taps /*host [n_taps]*/, int64_t row_stride,
                                     int32_t n_rows, int64_t position);

/* dflash_committed for a batch of sessions of one model in one call: session
 * b receives n_rows[b] rows at features[b] (a device pointer; rows
 * row_stride elements apart, the same stride for all) for the committed run
 * at position[b].  Each session's run is taken as dflash_committed takes it
 * (gap check, a restored prefix skipped, rows held below the threshold);
 * every session whose held rows reach DFLASH_PENDING_FLUSH_TOKENS flushes,
 * and those flushes run together as one batched context-only forward (dflash.go
 * committed and flush: the held rows flush in one context-only forward).  The
 * work runs on the first session's stream.  Every check runs before any state
 * changes, so an error leaves every session as it was.  Errors: INVALID_ARG,
 * CONTEXT_GAP, CAPACITY, with the session's index in the message. */
DFLASH_API int dflash_committed_batch(dflash_session* const* s /*host [batch]*/, int32_t batch,
                                      const void* const* features /*host [batch]*/, int64_t row_stride,
                                      const int32_t* n_rows /*host [batch]*/, const int64_t* position /*host [batch]*/);

/* dflash.go flush: rewinds each session's outstanding block, then writes all
 * held rows in one batched context-only forward.  When the draft has a
 * window, rows that no later query can see (slot <= F_new - W) are dropped
 * before aux_hidden_norms and fc (Laguna PR), while F still advances past
 * them. */
DFLASH_API int dflash_flush(dflash_session* const* s /*host [batch]*/, int32_t batch);
/* dflash.go settle: the same as flushing the one session. */
DFLASH_API int dflash_settle(dflash_session* s);

/* dflash.go commitBlock: if a block is outstanding, rewind it (the cache
 * keeps only context rows; the block's K/V slots become free).  Every write
 * path (committed, flush, propose) runs this first. */
DFLASH_API int dflash_commit_block(dflash_session* const* s /*host [batch]*/, int32_t batch);

/* dflash.go propose + selectBlock, batched.  n = min(max_tokens, B_s - 1);
 * a DFlash2 model drafts n = min(DFLASH2_DEPTH, B_s - 1) whenever
 * max_tokens > 0 (dflash2Depth replaces the depth controller's pick), so the
 * outputs must hold that many rows, and draws them with its candidate
 * selector at the request temperature only (no truncation, no penalties):
 * position i's token comes from the sel_candidates largest logits of row i,
 * scored logit + <sel_prev[prev], sel_next[c]>, by Gumbel-max at T > 0
 * (stream 0, keyed by the candidate's id) or argmax at T = 0, and the
 * position's candidate distribution softmax(score / T) is kept for verify
 * (dflash_candidates reads it).
 * A session gets out_n[b] = 0 (the pages' nil) when n <= 0 or it has no
 * context yet (F + P == 0); the others draft n tokens:
 *   commitBlock; the held rows become context (written first, at slots
 *   F..F+P-1); the block [current[b], mask x n] runs at positions F..F+n;
 *   rows 1..n are unembedded; temperature 0 takes the argmax, T > 0 draws
 *   argmax(l/T + Gumbel) with Philox4x32-10 keyed by `seed` at counter
 *   (v, row | 0 << 16, b, round).
 * current: [batch] int32.  Outputs (device): out_tokens [batch, n] int32,
 * out_q [batch, n] fp32 (probability of each token under softmax(l/T); 1 at
 * T = 0), out_logits [batch, n, V] fp32 or NULL.  out_n: (host) [batch].
 * The session keeps the logits, log-sum-exp and tokens for dflash_verify. */
DFLASH_API int dflash_propose(dflash_session* const* s /*host [batch]*/, int32_t batch, const int32_t* current,
                   int32_t max_tokens, float temperature, uint64_t seed, uint64_t round, int32_t* out_tokens,
                   float* out_q, float* out_logits, int32_t* out_n /*host*/);

/* The session's sampler truncation (dflash.go selectBlock draws from the
 * sampler's Distribution, whose IDs are the kept tokens).  At T > 0 the
 * draft's draw and q, and verify's target p, use the truncated distribution:
 * order a row of l/T by value (descending), then id; keep the first top_k;
 * over those, keep an entry while the probability mass strictly before it is
 * below top_p, and while its probability is at least min_p times the largest;
 * renormalise over what is kept.  top_k in [0, 1024] (0: no truncation),
 * top_p in (0, 1], min_p in [0, 1]; top_p < 1 or min_p > 0 need top_k >= 1.
 * Else DFLASH_ERR_INVALID_ARG and nothing changes.  Takes effect at the next
 * propose and verify; verify's q stays the one the proposal was drawn with. */
DFLASH_API int dflash_set_sampler(dflash_session* s, int32_t top_k, float top_p, float min_p);

/* The session's sampler penalties over the committed token history
 * ("Ollama DFlash block-diffusion draft model in mlxrunner", Facts: penalties
 * see only committed history, not other rows of the block; dflash.go
 * selectBlock).  The form is the sampler's repetition, presence and frequency
 * penalties (the pages do not state it): an id that occurs c > 0 times in the
 * history has a positive logit divided by repeat_penalty and a non-positive
 * one multiplied by it, then loses presence_penalty once and
 * frequency_penalty c times; penalties act on the raw logits, before the
 * temperature and any truncation.
 *   propose: every row of the block is penalised over the same history, so
 *   no row of the block counts toward another's penalties; out_logits and the
 *   logits the session keeps for verify are the penalised ones (the
 *   distribution the proposal was drawn from).
 *   verify: target row r is penalised over the history plus the draft tokens
 *   d_1..d_r in front of it, the history classic decoding would have had, so
 *   the output keeps the target sampler's law.  The penalised rows go to a
 *   workspace copy; the caller's target logits are never written.
 * history: device [n_history] token ids, n_history <= 4096 (the caller's
 * window, oldest first); copied in stream order into the session, so the
 * buffer must stay valid until the stream reaches this call.  Call again with
 * the new window as tokens are committed.  repeat 1, presence 0 and frequency
 * 0 turn the penalties off.  Errors: INVALID_ARG (repeat <= 0 or not finite,
 * a non-finite penalty, n_history outside [0, 4096], a null history).
 * Sessions with penalties on are verified by dflash_verify only:
 * dflash_verify_noalloc refuses them (INVALID_ARG). */
/* A DFlash2 session's candidate distributions from its last proposal (the
 * DFlash2 commit note: the selector returns each position's candidate
 * distribution, which verification uses): out_ids [n, sel_candidates] int32
 * and out_probs [n, sel_candidates] fp32, device, in candidate order (logit
 * descending, then id); at T = 0 the probabilities are one-hot on the token.
 * Copied in stream order.  Errors: STATE if the model is not DFlash2 or the
 * session has no proposal. */
DFLASH_API int dflash_candidates(const dflash_session* s, int32_t* out_ids, float* out_probs);

DFLASH_API int dflash_set_penalties(dflash_session* s, float repeat_penalty, float presence_penalty,
                                    float frequency_penalty, const int32_t* history /*device [n_history]*/,
                                    int32_t n_history);

/* Speculative verification of each session's last proposal.
 * target_logits [batch, n+1, V] (fp32 or bf16 per logits_dtype): row r
 * scores the token after [current, d_1..d_r].  draft_tokens [batch, n]: the
 * tokens under test (normally the proposal; tests may force others).
 * T == 0: accept while argmax(row i-1) == d_i; bonus = argmax(row a).
 * T > 0: accept d_i iff u_i * q_i(d_i) < p_i(d_i), u_i uniform from stream 1;
 * at the first rejection the bonus is drawn from max(0, p_i - q_i) (from p_i
 * if that is all zero), after n acceptances from p of row n (stream 2).
 * q_i is the proposal's distribution softmax(l_i / T_propose) (one-hot of
 * the proposed token if that proposal was greedy); with a truncating sampler
 * (dflash_set_sampler) p and q are the truncated distributions; for a
 * DFlash2 proposal q_i is position i's candidate distribution (zero outside
 * the candidates).
 * Outputs: out_accept [batch] int32 in 0..n, out_bonus [batch] int32.
 * Errors: STATE if a session has no proposal with this n. */
DFLASH_API int dflash_verify(dflash_session* const* s /*host [batch]*/, int32_t batch, const void* target_logits,
                  int32_t logits_dtype, const int32_t* draft_tokens, int32_t n, float temperature, uint64_t seed,
                  uint64_t round, int32_t* out_accept, int32_t* out_bonus);

/* The same verification as dflash_verify, for callers that may not allocate
 * device memory: a serving runtime that hands out all GPU memory up front
 * under a fixed budget, or a decode loop that cannot take cudaMalloc's
 * implicit device synchronisation between rounds.  (The pages have no
 * counterpart; this is a property of this library.)  dflash_verify grows a
 * model workspace with cudaMalloc on demand; this call never calls cudaMalloc,
 * cudaFree or an allocating routine.  Its scratch is a 4 MiB array inside the
 * library image, present on every GPU that loads the library until the
 * process exits.  Limits: at most 128 sessions per call, and
 * batch * (n + 1) * ceil(V / chunk) 16-byte row partials (chunk = 16384 when
 * the call's target rows give every SM of the device eight such chunks, else
 * 4096) plus the bonus partials must fit the 4 MiB (about 200k partials);
 * larger calls return DFLASH_ERR_CAPACITY and change nothing.  The call runs
 * on the device the sessions were opened on: it makes that device current for
 * its duration and restores the caller's afterwards.  The first call on a
 * device looks up the scratch's device address (cudaGetSymbolAddress) with
 * that device current.  The per-session tables
 * travel as a kernel parameter, so the call does not wait for the stream.
 * Every call shares the one scratch area and leaves its contents there, so
 * calls that overlap on the GPU (different streams, no ordering between
 * them) race; issue them in stream order.  With timing on
 * (dflash_timing_enable) the call is timed and counted as dflash_verify is.
 * Arguments, outputs and errors otherwise as dflash_verify. */
DFLASH_API int dflash_verify_noalloc(dflash_session* const* s /*host [batch]*/, int32_t batch,
                                     const void* target_logits, int32_t logits_dtype, const int32_t* draft_tokens,
                                     int32_t n, float temperature, uint64_t seed, uint64_t round,
                                     int32_t* out_accept, int32_t* out_bonus);

/* dflash.go close: flush, then release the session (synchronises its stream). */
DFLASH_API int dflash_close(dflash_session* s);

DFLASH_API int dflash_stats(const dflash_session* s, dflash_counters* out /*host*/);

/* Host view of the cursors: F (ctxOffset), P (pendingCount), outstanding block. */
DFLASH_API int dflash_session_state(const dflash_session* s, int64_t* ctx_offset /*host*/, int32_t* pending /*host*/,
                         int32_t* block_outstanding /*host*/);

/* Copies context rows [first_slot, first_slot + n_rows) of one layer out of
 * / into the session cache.  k, v: [Hkv, n_rows, d] in the storage type.
 * Rows must lie below F + block_size (and, with a window, inside the ring).
 * Used for checkpoint / resume (restored prefixes) and inspection. */
DFLASH_API int dflash_kv_export(const dflash_session* s, int32_t layer, int64_t first_slot, int32_t n_rows, void* k_out,
                     void* v_out);
DFLASH_API int dflash_kv_import(dflash_session* s, int32_t layer, int64_t first_slot, int32_t n_rows, const void* k_in,
                     const void* v_in);

/* ---- measurement ---------------------------------------------------------
 * Not part of the round.  While timing is on, the runtime brackets every
 * launch of the matrix-product, attention, sampling and verify kernels with
 * CUDA events on the launching stream and records the launch's algorithmic
 * bytes (each operand read once, each output written once) and flops; every
 * kernel launch of the model is also counted. */
typedef struct dflash_kernel_time {
  char name[24];     /* kernel class: "gemm_tc", "gemm_simt", "attention", "sample", "verify", "all" */
  int64_t launches;  /* kernel launches of this class */
  double total_ms;   /* sum of event-measured durations (0 for "all") */
  double bytes;      /* algorithmic bytes of those launches */
  double flops;      /* algorithmic flops of those launches */
} dflash_kernel_time;

/* on != 0 clears the records and starts recording; on == 0 stops. */
DFLASH_API int dflash_timing_enable(dflash_model* m, int32_t on);
/* Synchronises the device, then writes up to max_entries classes to out
 * (host) and their number to *n_entries (host). */
DFLASH_API int dflash_timing_read(dflash_model* m, dflash_kernel_time* out, int32_t max_entries, int32_t* n_entries);

/* ---------------------------------------------------------------------------
 * Synthetic target (the model the draft speculates for).
 *
 * ollama mlxrunner/dflash.go and the mlxcel PR #1771 ("add the Laguna DFlash
 * drafter": the verify forward with its 5-tap capture and rollback trim) run
 * the draft against a real target.  No target checkpoint exists here: a small
 * fp32 dense decoder stands in (RMSNorm, rotate-half RoPE, causal multi-head
 * attention over its own cache, SwiGLU MLP).  Per position it gives what
 * dflash_committed consumes, the taps (the embedding output and the residual
 * stream after each attention and each MLP, [rows][(2 * n_layers + 1) *
 * hidden]), and what dflash_verify consumes, raw next-token logits
 * [rows][vocab].  Every row is computed against the cache and the earlier
 * rows of the call, so a multi-row verify forward equals token-by-token
 * decoding.
 * ------------------------------------------------------------------------- */
typedef struct dflash_target dflash_target;

typedef struct dflash_target_config {
  int32_t hidden, n_heads, head_dim, intermediate, vocab, n_layers;
  float rope_theta, rms_eps;
} dflash_target_config;

/* fp32 device matrices, row-major [out][in]; borrowed (must outlive the target) */
typedef struct dflash_target_layer {
  const void *n1, *wq, *wk, *wv, *wo, *n2, *wg, *wu, *wd;
} dflash_target_layer;

typedef struct dflash_target_weights {
  const void* embed;         /* [vocab][hidden] */
  const void* unembed;       /* [vocab][hidden] */
  const void* final_norm;    /* [hidden] */
  const dflash_target_layer* layers;  /* host array of n_layers */
} dflash_target_weights;

/* Validates the shapes (hidden and n_heads * head_dim at most 4096, hidden and
 * intermediate multiples of 4, head_dim a multiple of 4 and at most 128, else
 * DFLASH_ERR_SHAPE) and the weights (non-NULL; wo, wd and unembed 16-byte
 * aligned, else DFLASH_ERR_INVALID_ARG); allocates
 * a cache of max_ctx positions; every call enqueues on `stream`. */
DFLASH_API int dflash_target_create(const dflash_target_config* cfg, const dflash_target_weights* w, int64_t max_ctx,
                                    void* stream, dflash_target** out);
DFLASH_API int dflash_target_destroy(dflash_target* t);
/* Forward of `rows` tokens (device int32) at positions start.. , which must
 * equal the cached length (else DFLASH_ERR_CONTEXT_GAP); writes logits (device
 * fp32 [rows][vocab]) and, when taps is not NULL, the taps (device fp32).  The
 * rows join the cache. */
DFLASH_API int dflash_target_forward(dflash_target* t, const int32_t* tokens, int32_t rows, int64_t start,
                                     float* logits, float* taps);
/* Rolls the cache back to `length` rows (a rejected verify tail). */
DFLASH_API int dflash_target_trim(dflash_target* t, int64_t length);
DFLASH_API int dflash_target_length(const dflash_target* t, int64_t* length);
/* Greedy token of each logits row (device int32 [rows]), lowest id on a tie. */
DFLASH_API int dflash_target_argmax(dflash_target* t, const float* logits, int32_t rows, int32_t* out);
/* Synchronises the target's stream and reports a device-side error (a token
 * id outside [0, vocab)) as DFLASH_ERR_DEVICE. */
DFLASH_API int dflash_target_device_status(dflash_target* t);

/* ---- block-versus-chain exactness ----------------------------------------
 * Greedy speculative output equals plain greedy decoding only if the target's
 * multi-row verify forward gives the same logits as one-token decoding.  The
 * mlxcel Laguna PR (the real-checkpoint probe commit and the report commits)
 * compares a block_size-wide verify block with single-token decode on the
 * target alone, counts the logit bytes that differ at the first verify
 * position (its gate declines the pairing when any do) and reports the top-2
 * logits of both arms at every argmax disagreement, whose chain-arm margin
 * (0.0 or 0.125 there) shows a bf16 tie.  Logits here are fp32; bytes are
 * counted over their fp32 encodings. */
typedef struct {
  int32_t differing_bytes; /* bytes of the row's fp32 logits that differ between the arms */
  int32_t block_top[2];    /* the block arm's best and second token (value desc, then id asc) */
  int32_t chain_top[2];    /* the chain arm's */
  float block_val[2];      /* their logits */
  float chain_val[2];
} dflash_exactness_row;

typedef struct {
  int64_t rows;
  int64_t differing_bytes;           /* over all rows */
  int64_t first_row_differing_bytes; /* at the first verify position */
  int32_t disagreements;             /* rows whose block and chain argmax differ */
  int32_t allows;                    /* 1 when no logit byte differs at the first position */
} dflash_exactness_summary;

/* Row records of two device fp32 logit arrays [rows][vocab] (block arm,
 * chain arm) into device out[rows], on `stream`.  NaN entries are never
 * chosen as a top token.  Any [rows][vocab] pair can be compared, e.g. the
 * logits of an external target.  Bad sizes or null pointers:
 * DFLASH_ERR_INVALID_ARG. */
DFLASH_API int dflash_logits_compare(const float* block, const float* chain, int32_t rows, int32_t vocab,
                                     dflash_exactness_row* out, void* stream);
/* Host reduction of `rows` row records (host memory) into *out. */
DFLASH_API int dflash_exactness_summarize(const dflash_exactness_row* rows_host, int32_t rows,
                                          dflash_exactness_summary* out);
/* The probe on a dflash_target: `rows` tokens at start (= the cached length,
 * else DFLASH_ERR_CONTEXT_GAP) as one block forward into block_logits, then
 * as `rows` one-token forwards into chain_logits (both device fp32
 * [rows][vocab], caller-owned), then the comparison into device out_rows.
 * The cache is trimmed back to `start`, so the probe leaves the target as it
 * found it.  When summary is not NULL the call synchronises the stream and
 * fills it. */
DFLASH_API int dflash_target_exactness_probe(dflash_target* t, const int32_t* tokens, int32_t rows, int64_t start,
                                             float* block_logits, float* chain_logits,
                                             dflash_exactness_row* out_rows, dflash_exactness_summary* summary);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H */
