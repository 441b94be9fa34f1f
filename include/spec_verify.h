/*
 * spec_verify.h -- C ABI of the target-verification round of speculative
 * decoding on one GB300 (sm_103a).
 *
 * The round (sources, by page title and section):
 *  - "Model-neutral Speculative Decoding", section "The exactness
 *    transaction": evaluate the anchor and the proposal block in one target
 *    pass; sample target rows only through the first mismatch; commit the
 *    accepted prefix; emit exactly one correction or bonus token; for greedy
 *    decoding the speculative and autoregressive token ids match exactly; for
 *    stochastic decoding the target sampler advances once per emitted sample
 *    and never for a rejected suffix.
 *  - "Speculative Decoding (D5-R) -- Plan", section 3 "Mechanism -- one
 *    round": one nt = d+1 forward whose rows are the next token plus the d
 *    drafted candidates at contiguous positions; greedy argmax per verify row,
 *    accept while equal to the drafted token, always emit at least one token;
 *    the target writes d+1 KV rows in place and rejected slots are simply
 *    overwritten next round ("positions are data"); and the status notes on
 *    the weights-once batched verify and bitwise position-invariant verify
 *    attention.
 *  - "DFlash and DSpark Speculative Decoding", "How DSpark Works" and
 *    "Notes": lossless output under the strict rejection sampler (accept with
 *    min(1, p/q), else resample from norm(max(0, p - q))).
 *
 * Conventions for every function below:
 *  - Return value: SPEC_OK (0) or a negative SPEC_E_* code; the message of
 *    the last failure on the calling thread is in spec_last_error().
 *  - Pointers are DEVICE pointers owned by the caller unless a parameter says
 *    "host".  fp16 data is passed as uint16_t (IEEE binary16 bits).  Device
 *    arrays must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued on it asynchronously, except for create/destroy/state calls,
 *    which synchronise.
 *  - On an error return nothing has been enqueued and no state has changed.
 *    Errors that can only be seen on the device (a token id out of range, a
 *    position past max_ctx, a non-finite logit) set the model's device error
 *    word: the round then commits nothing, writes -1 to its n_acc and emitted
 *    outputs, and spec_error_check() reports SPEC_E_INVALID.
 *  - A model or packed matrix is used from one stream at a time.
 *  - The library allocates device memory only in *_create, and, for the
 *    standalone entry points that need scratch, on first use per device
 *    (a cached, growing workspace).
 *  - Two environment variables, read once (at matrix / model creation for
 *    the first, at the first launch for the second), change how kernels are
 *    launched but never what they compute beyond the summation order of
 *    one GEMM's K split:
 *      SPEC_VERIFY_LINEAR_SPLIT  "KW:S" (every matrix) or "N:K:KW:S" entries,
 *        comma-separated: the K split of the verify GEMM (KW warps of a CTA
 *        and S CTAs share a tile's K range) instead of the library's choice.
 *        The split is fixed per matrix, so rows stay bitwise equal across nt
 *        under any setting; results under two settings may differ in the
 *        last bits.  Meant for tests and tuning.
 *      SPEC_VERIFY_PDL=0  launch every kernel as a plain stream-ordered
 *        launch (no programmatic dependent launch).  Results are unchanged.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_OK 0
#define SPEC_E_INVALID (-1)     /* bad argument, token id, non-finite value */
#define SPEC_E_SHAPE (-2)       /* size or alignment precondition violated */
#define SPEC_E_CUDA (-3)        /* a CUDA runtime call failed */
#define SPEC_E_OOM (-4)         /* device allocation failed */
#define SPEC_E_UNSUPPORTED (-5) /* mode not supported: fails closed */
#define SPEC_E_TIMEOUT (-6)     /* a bounded device wait ran out */

#define SPEC_Q4 4 /* 4-bit signed ints in [-8, 7], blocks of 32, fp16 scale */
#define SPEC_Q6 6 /* 6-bit signed ints in [-32, 31], blocks of 32, fp16 scale */
#define SPEC_Q8 8 /* 8-bit signed ints in [-128, 127], blocks of 32, fp16 scale */

#define SPEC_MAX_NT 16 /* rows per sequence in one round: anchor + up to 15 drafts */

/* Copies the last error message of the calling thread into buf. */
void spec_last_error(char* buf, size_t len);

/* ------------------------------------------------------------------------
 * Block-quantised matrix W[N][K] in canonical planes (device, caller-owned):
 *   qs     Q4 / Q6: [N][K/32][16] bytes.  Byte j of block b holds element
 *          32b+j in its low nibble and element 32b+j+16 in its high nibble.
 *          Q4 stores u = q + 8 (the q4_0 element order); Q6 stores the low 4
 *          bits of u = q + 32.
 *          Q8: [N][K/32][32] bytes, byte j of block b = element 32b+j as a
 *          two's-complement int8 (the q8_0 element order).
 *   qh     [N][K/32][8] bytes, Q6 only (NULL for Q4 and Q8): the high 2 bits
 *          of u, element j of the block at bits 2*(j%4) of byte j/4.
 *   scales [N][K/32] fp16.  W[n][k] = scale[n][k/32] * q[n][k].
 * The q4_0 / q8_0 weights of the pages' targets ("Speculative Decoding
 * (D5-R) -- Plan", status notes: the verify machinery extended to q8_0/q4_0)
 * are these planes with each block's scale split out of its bytes.
 * Preconditions: K % 32 == 0, N % 16 == 0.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t qtype; /* SPEC_Q4, SPEC_Q6 or SPEC_Q8 */
  int32_t N, K;
  const void* qs;
  const void* qh;
  const void* scales;
} spec_qweight;

/* A matrix repacked into the streaming layout of the verify GEMM. */
typedef struct spec_qmat spec_qmat;

/* Repacks `w` into a new device-resident matrix (the caller may free the
 * canonical planes after return).  max_rows bounds the nt of later
 * spec_linear_q calls (1..16*1024).  Synchronises `stream`. */
int spec_qmat_create(const spec_qweight* w, int max_rows, void* stream,
                     spec_qmat** out);
int spec_qmat_destroy(spec_qmat* m);

/* Weights-once multi-row dequant GEMM ("Speculative Decoding (D5-R) --
 * Plan", section 1: the batched verify is a weights-once round, not a
 * per-row restream):
 *   y[r][n] = sum_k W[n][k] * x[r][k],  r < nt,
 * x fp16 [nt][K] row-major, y fp32 [nt][N] row-major.  Every row is computed
 * by the same instruction sequence whatever nt is, so row r is bitwise equal
 * to the nt = 1 result for the same x row.  1 <= nt <= max_rows. */
int spec_linear_q(const spec_qmat* w, const uint16_t* x, int nt, float* y,
                  void* stream);

/* The same product on the tensor cores, as multi-sequence rounds run it
 * (tcgen05.mma with tensor-memory accumulators; rows are the N dimension):
 * each weight q * scale enters as an exact pair of fp16 numbers, hi =
 * fp16(q * scale) and lo = q * scale - hi (two MMAs per 16-k step), so every
 * product is exact and only the fp32 accumulation over K rounds.  Every row
 * is computed by the same instructions whatever R is, so a row's result does
 * not depend on the other rows; it differs from spec_linear_q's in the last
 * bits (that kernel accumulates each 32-block's integer sum and applies the
 * scale in fp32).  The matrix's (tile, 64-k chunk) work is cut once, at
 * creation, from N, K and the SM count (never from R): one CTA per tile, a
 * K split, or one run per SM that may cross a tile boundary; a tile cut
 * across CTAs is summed in k order, its CTAs launched cooperatively (all
 * resident).  1 <= R <= max_rows (launched in blocks of 192 rows). */
int spec_linear_q_tc(const spec_qmat* w, const uint16_t* x, int R, float* y,
                     void* stream);

/* ------------------------------------------------------------------------
 * Decoder model: RMSNorm -> QKV + rotate-half RoPE -> causal GQA attention
 * over the KV cache -> O + residual -> RMSNorm -> gate/up + SwiGLU -> down +
 * residual, n_layers times; final RMSNorm; LM head over the full vocabulary.
 * Every linear is a block-quantised matrix of any of the formats above
 * (SPEC_Q4, SPEC_Q6, SPEC_Q8).  Residual stream fp32, activations fp16, KV
 * cache fp16.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t n_layers; /* 0 allowed: LM head only (spec_lm_head) */
  int32_t hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  int32_t max_ctx;  /* KV positions per sequence (at most 786432) */
  int32_t max_nt;   /* rows per sequence per round, <= SPEC_MAX_NT */
  int32_t max_seqs; /* sequence slots */
  float rms_eps;    /* e.g. 1e-6 */
  float rope_theta; /* e.g. 10000 */
  int32_t use_rope; /* 1: rotate q and new k at their absolute positions */
} spec_model_desc;

typedef struct {
  const uint16_t* embed;      /* fp16 [vocab][hidden] (NULL if n_layers == 0) */
  const float* norm_w;        /* fp32 [2*n_layers+1][hidden]: attn_l, ffn_l ..., final */
  const spec_qweight* wqkv;   /* HOST array [n_layers]; rows [q heads | k heads | v heads] */
  const spec_qweight* wo;     /* HOST array [n_layers]; [hidden][n_q_heads*head_dim] */
  const spec_qweight* wgu;    /* HOST array [n_layers]; rows [gate (ffn) ; up (ffn)] */
  const spec_qweight* wd;     /* HOST array [n_layers]; [hidden][ffn] */
  spec_qweight lm_head;       /* [vocab][hidden] */
} spec_model_weights;

typedef struct spec_model spec_model;

/* Creates a model: repacks all weights, allocates the fp16 KV cache
 * [n_layers][max_seqs][n_kv_heads][max_ctx][head_dim] (zeroed), activation
 * buffers for max_seqs*max_nt rows and the per-sequence state
 * (n_past = 0, emit_idx = 0, anchor = 0).  Synchronises `stream`. */
int spec_model_create(const spec_model_desc* desc, const spec_model_weights* w,
                      void* stream, spec_model** out);
int spec_model_destroy(spec_model* m);

/* Device pointers of layer `layer`'s K and V caches, each
 * [max_seqs][n_kv_heads][max_ctx][head_dim] fp16, for filling a context. */
int spec_model_kv_cache(spec_model* m, int layer, uint16_t** k, uint16_t** v);

/* Copies a context into the cache of slot `seq`, layer `layer`, positions
 * [pos0, pos0 + n_pos): k and v are fp16 [n_kv_heads][n_pos][head_dim]
 * (device or host memory).  Asynchronous on `stream`. */
int spec_kv_fill(spec_model* m, int layer, int seq, int pos0, int n_pos,
                 const uint16_t* k, const uint16_t* v, void* stream);

/* The reverse of spec_kv_fill: copies positions [pos0, pos0 + n_pos) of slot
 * `seq`, layer `layer` out to k and v, fp16 [n_kv_heads][n_pos][head_dim]
 * (device or host memory).  Asynchronous on `stream`. */
int spec_kv_read(spec_model* m, int layer, int seq, int pos0, int n_pos, uint16_t* k,
                 uint16_t* v, void* stream);

/* Diagnostics: copies up to `bytes` of an internal activation buffer of the
 * last target pass to dst (device or host).  which: 0 residual h fp32
 * [R][hidden], 1 normed input fp16 [R][hidden] (after the final norm: the LM
 * head input), 2 SwiGLU output fp16 [R][ffn], 3 attention output fp16
 * [R][n_q_heads*head_dim], 4 rotated q fp16 [R][n_q_heads][head_dim] (the
 * last layer's), 5 logits fp32 [R][vocab].  Asynchronous on `stream`. */
int spec_model_debug_read(spec_model* m, int which, void* dst, size_t bytes, void* stream);

/* Per-sequence transaction state, HOST arrays of n entries for the slots
 * seq_ids[0..n): n_past (committed positions), emit_idx (sampler slot of the
 * next emitted token), anchor (last committed token, row 0 of the next
 * round).  NULL arrays are skipped.  Synchronous. */
int spec_state_set(spec_model* m, int n, const int32_t* seq_ids,
                   const int32_t* n_past, const uint64_t* emit_idx,
                   const int32_t* anchor);
int spec_state_get(spec_model* m, int n, const int32_t* seq_ids, int32_t* n_past,
                   uint64_t* emit_idx, int32_t* anchor);

/* Synchronises `stream`, reads and clears a device error word: the model's
 * (m != NULL), else the one word this device's standalone entry points share
 * (spec_linear_q, spec_accept_*): bit 0x10 there is a weight or activation
 * copy that did not arrive within about a second.
 * Returns SPEC_OK or SPEC_E_INVALID (the bits are stored in *bits if not NULL). */
int spec_error_check(spec_model* m, void* stream, uint32_t* bits);

/* 1 (default): spec_verify_round replays one captured CUDA graph per
 * (n_seq, d, mode) shape -- for a greedy round the whole round, target pass,
 * accept and commit; the caller's arrays are kernel arguments of the graph,
 * updated in place when they change from one call to the next.  0: launches
 * kernels one by one. */
int spec_model_set_graphs(spec_model* m, int enable);

/* Which GEMM a round's linear layers (and LM head) run on is chosen by the
 * round's number of sequences, never by d: rounds of at least `min_seqs`
 * sequences use the tensor-core GEMM of spec_linear_q_tc, the others the
 * GEMM of spec_linear_q.  So a sequence's rows are bitwise the same at every
 * depth d for a given batch size, and greedy speculative decoding of a batch
 * is byte-identical to plain decoding of the same batch.  Default 2; 0 turns
 * the tensor-core GEMM off.  Synchronises the device and drops captured
 * graphs. */
int spec_model_set_tc_min_seqs(spec_model* m, int min_seqs);

/* In-round kernel timing.  enable = 1: the model's later rounds launch their
 * kernels one by one (no graph), with a CUDA event recorded before and after
 * each verify-GEMM launch and each attention launch (chunk + merge kernels);
 * the events see each kernel inside a real round (its inputs written by the
 * kernel before it, the caches as the round leaves them), at the price of
 * the serialisation an event imposes between neighbouring kernels.  Calling
 * it (enable 0 or 1) synchronises the device and clears the totals. */
int spec_model_profile(spec_model* m, int enable);

/* Kernel classes of spec_model_profile_read. */
#define SPEC_PROF_QKV 0       /* QKV GEMM + RoPE + KV write */
#define SPEC_PROF_O 1         /* O GEMM + residual */
#define SPEC_PROF_GATE_UP 2   /* gate/up GEMM + SwiGLU */
#define SPEC_PROF_DOWN 3      /* down GEMM + residual */
#define SPEC_PROF_LM_HEAD 4   /* LM head (+ logits) + argmax */
#define SPEC_PROF_ALL_GEMMS 5 /* classes 0-4 together */
#define SPEC_PROF_ATTN 6      /* verify attention (chunk + merge kernels) */

/* Totals since the last spec_model_profile call for one kernel class (HOST
 * outputs, each may be NULL): summed event-to-event seconds, launches, and
 * the algorithmic bytes (packed weights once, activations in, outputs out;
 * 0 for attention, whose bytes depend on positions held on the device) and
 * flops (2 * rows * N * K) of those launches.  Synchronises the device. */
int spec_model_profile_read(spec_model* m, int kind, double* seconds, int64_t* launches,
                            double* bytes, double* flops);

/* Test hook for the fail-closed path of the verify GEMM's bounded waits.
 * Every wait of a GEMM CTA on its copies (weights and activations, TMA bulk
 * copies completing on an mbarrier) gives up after about a second (131072
 * suspended tries of about 10 us), sets ERR_TIMEOUT (0x10) in the model's
 * error word, waits with the full budget for the copies it issued and
 * finishes without using them, so the round commits nothing and writes -1
 * outputs.  This call sets the try budget of the FIRST wait of each GEMM CTA
 * on its copies (the activation slice of the spec_linear_q kernel, the first
 * weight records of the tensor-core kernel) for the model's later rounds; 0
 * makes that wait give up at once.  Drains always keep the full budget.
 * 0 <= tries <= 131072; synchronises the device and drops captured graphs. */
int spec_model_set_wait_budget(spec_model* m, int tries);

/* Causal GQA attention of nt query rows per sequence over the KV cache of
 * `layer`, bitwise position-invariant: row i of sequence s (absolute
 * position n_past[s] + i) is computed exactly as it would be at nt = 1
 * ("Speculative Decoding (D5-R) -- Plan", status notes: batched verify
 * attention made bitwise position-invariant).  First writes k_new/v_new
 * [n_seq*nt][n_kv_heads][head_dim] at positions n_past..n_past+nt-1 of each
 * sequence; n_past itself is not changed.
 *   seq_ids  device int32 [n_seq] slots;  q fp16 [n_seq*nt][n_q_heads][head_dim]
 *   out      fp16 [n_seq*nt][n_q_heads*head_dim] */
int spec_verify_attn(spec_model* m, int layer, int n_seq, const int32_t* seq_ids,
                     int nt, const uint16_t* q, const uint16_t* k_new,
                     const uint16_t* v_new, uint16_t* out, void* stream);

/* Full-vocabulary LM head: logits[r][v] = sum_k W_lm[v][k] x[r][k] (fp32),
 * with a fused per-row argmax (ties to the lowest id).  x fp16 [R][hidden],
 * R <= max_seqs*max_nt; logits [R][vocab] or NULL; argmax int32 [R] or NULL.
 * A NaN logit sets the device error word. */
int spec_lm_head(spec_model* m, const uint16_t* x, int R, float* logits,
                 int32_t* argmax, void* stream);

/* Greedy accept ("Speculative Decoding (D5-R) -- Plan", section 3):
 *   a = number of leading i < d with argmax[s][i] == draft[s][i];
 *   emitted[s] = draft[s][0..a-1], argmax[s][a], then -1 padding;
 *   n_acc[s] = a.
 * argmax [n_seq][d+1], draft [n_seq][d], emitted [n_seq][d+1]. */
int spec_accept_greedy(const int32_t* argmax, const int32_t* draft, int n_seq,
                       int d, int32_t* n_acc, int32_t* emitted, void* stream);

/* Strict rejection sampling ("DFlash and DSpark Speculative Decoding",
 * "Notes"; sampler-advance rule of "Model-neutral Speculative Decoding", "The
 * exactness transaction").  For each sequence s, slot i < d, draft x:
 *   z = logits / temperature (fp32, round to nearest);
 *   W_v = floor(exp(z_v - max z) * 2^32) (own fp32 exp, identical on every
 *   platform), S = sum W_v; Wq, Sq likewise from q_logits;
 *   U = Philox4x32-10(key = seed, counter = (j lo, j hi, seq_ids[s], 0)) for
 *   the emitted slot j = emit_idx[s] + i;
 *   accept iff U[0] * Wq_x * S < 2^32 * W_x * Sq  (u < p_x / q_x, exact);
 *   on the first rejection resample from R_v = max(0, W_v*Sq - Wq_v*S) with
 *   threshold floor(U[1] * sum R / 2^32) and stop; after d accepts sample the
 *   bonus from row d with floor(U[1] * S / 2^32).
 * emit_idx[s] += n_acc[s] + 1: one sampler slot per emitted token, none for
 * the rejected suffix.
 *   p_logits fp32 [n_seq][d+1][V]; q_logits fp32 [n_seq][d][V] (may be NULL
 *   when d == 0); draft int32 [n_seq][d]; seq_ids int32 [n_seq];
 *   emit_idx uint64 [n_seq] (in/out); n_acc [n_seq]; emitted [n_seq][d+1].
 * Decisions are bit-identical to any correct implementation of the same
 * integer rules on the same fp32 logits. */
int spec_accept_stochastic(const float* p_logits, const float* q_logits,
                           const int32_t* draft, int n_seq, int d, int V,
                           float temperature, uint64_t seed,
                           const int32_t* seq_ids, uint64_t* emit_idx,
                           int32_t* n_acc, int32_t* emitted, void* stream);

/* Same computation, arguments and results as spec_accept_stochastic, but
 * this entry point allocates no memory at all.  It is for callers that cannot
 * call cudaMalloc: code whose device memory is owned by a custom allocator
 * or a fixed arena that forbids outside allocations, and latency-critical
 * loops that must not risk the implicit device synchronisation an
 * allocation can cause.  (The pages have no counterpart for this entry
 * point; it is an addition of this library.)
 *  - Scratch is one fixed array in the library's device globals (about 64 KB
 *    per GPU that loads the library, held until the process exits), so the
 *    batch is limited: n_seq <= 1024 and n_seq * (2d + 1) <= 4096; larger
 *    batches return SPEC_E_SHAPE with a message.  V is limited as for
 *    spec_accept_stochastic.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls share the one array: calls whose work overlaps on the GPU
 *    (different streams, or different host threads) race and must be ordered
 *    by the caller.  Each call clears the array's error word itself.
 *  - Errors seen on the device (non-finite logit, bad draft id) make the
 *    affected outputs -1 and leave emit_idx unchanged, as in
 *    spec_accept_stochastic; spec_error_check does not report them. */
int spec_accept_stochastic_noalloc(const float* p_logits, const float* q_logits,
                                   const int32_t* draft, int n_seq, int d, int V,
                                   float temperature, uint64_t seed,
                                   const int32_t* seq_ids, uint64_t* emit_idx,
                                   int32_t* n_acc, int32_t* emitted, void* stream);

typedef struct {
  int32_t greedy;      /* 1: greedy argmax accept; 0: strict rejection sampling */
  float temperature;   /* stochastic only, > 0 */
  uint64_t seed;       /* stochastic only: Philox key */
} spec_sampling;

/* One verify round ("Model-neutral Speculative Decoding", "The exactness
 * transaction", steps 3-6): rows [anchor, draft[s][0..d-1]] of each sequence
 * at positions n_past..n_past+d in one weights-once target pass (all layers
 * and the LM head), then the accept step, then the commit:
 *   n_past += n_acc + 1, emit_idx += n_acc + 1, anchor = last emitted token.
 * The new KV rows are written in place; rejected rows are overwritten later.
 *   seq_ids int32 [n_seq] (distinct slots < max_seqs: a slot named twice, or
 *   out of range, sets the device error word and the round commits nothing);
 *   draft int32 [n_seq][d];
 *   q_logits fp32 [n_seq][d][vocab] (draft distributions; NULL iff greedy);
 *   sampling: HOST pointer;  n_acc int32 [n_seq]; emitted int32 [n_seq][d+1];
 *   logits_out fp32 [n_seq*(d+1)][vocab] or NULL.
 * 1 <= n_seq <= max_seqs, 0 <= d < max_nt.  All arrays are device memory,
 * read and written in place on `stream`; n_acc and emitted must overlap
 * neither each other nor seq_ids / draft (SPEC_E_INVALID otherwise). */
int spec_verify_round(spec_model* m, int n_seq, const int32_t* seq_ids,
                      const int32_t* draft, int d, const float* q_logits,
                      const spec_sampling* sampling, int32_t* n_acc,
                      int32_t* emitted, float* logits_out, void* stream);

/* The same verify round with seq_ids, draft, n_acc and emitted in HOST
 * memory (any host memory; shapes as for spec_verify_round).  q_logits may
 * be device memory or host memory; host q_logits (pinned for full copy
 * bandwidth) are copied into a buffer the model allocated at creation, on a
 * stream of the model's own, while the round's target pass (which does not
 * read them) runs; the accept waits for the copy.
 * The small inputs are copied into the model's mapped pinned staging, which
 * the kernels read and write in place (no copy engine steps; a greedy round
 * with graphs on is one graph launch); the
 * call synchronises `stream` before it copies the outputs out, so they are
 * valid on return.  Calls on one model must not overlap (the staging is the
 * model's).  Errors: as spec_verify_round, plus SPEC_E_CUDA from the
 * synchronisation. */
int spec_verify_round_host(spec_model* m, int n_seq, const int32_t* seq_ids,
                           const int32_t* draft, int d, const float* q_logits,
                           const spec_sampling* sampling, int32_t* n_acc,
                           int32_t* emitted, void* stream);

/* ---------------------------------------------------------------------------
 * Adaptive draft depth: a host controller that picks the depth d of the next
 * verify round ("Speculative Decoding (D5-R) -- Plan", status notes, which
 * list the ingredients: smoothed acceptance estimates, a window of measured
 * round costs, hysteresis, trying unmeasured depths first, a cap on d; the
 * rules below are this library's reading).  Host only: no GPU work, no
 * stream, no model.
 *  - Position i = 1..d_max keeps decayed Beta counts (a_i, b_i).  A round at
 *    depth d in which a sequence accepted n drafts adds 1 to a_i for
 *    i <= min(n, d) and, if n < d, 1 to b_{n+1}; a negative n (a failed
 *    sequence) adds nothing.  All counts are first multiplied by `decay`.
 *  - p_i = (a_i + prior_accept) / (a_i + b_i + prior_accept + prior_reject)
 *    (prior_reject = 0: a position never observed has p_i = 1).
 *  - E(d) = sum_{k=0..d} prod_{i<=k} p_i tokens per round; c(d) = the
 *    minimum of the depth's last `cost_window` round times; r(d) = E / c.
 *  - While some depth in [d_min, d_max] has no round time, the deepest such
 *    depth is next (its r counts as +infinity).  Otherwise the smallest
 *    depth of maximal r replaces the current depth when its r exceeds the
 *    current r by the factor (1 + hysteresis).  The first depth is d_max.
 * Every double is rounded operation by operation, as written above. */
typedef struct {
  int32_t d_min, d_max;       /* 0 <= d_min <= d_max <= SPEC_MAX_NT - 1 */
  double prior_accept;        /* >= 0 */
  double prior_reject;        /* >= 0; prior_accept + prior_reject > 0 */
  double decay;               /* (0, 1] */
  double hysteresis;          /* >= 0 */
  int32_t cost_window;        /* 1..64 round times per depth */
} spec_depth_params;
typedef struct spec_depth_ctl spec_depth_ctl;

/* Defaults: d in [1, 7], prior (1, 0), decay 0.95, hysteresis 0.10, window 4. */
void spec_depth_params_default(spec_depth_params* p);
/* params NULL = the defaults.  SPEC_E_INVALID on a parameter out of range. */
int spec_depth_ctl_create(const spec_depth_params* params, spec_depth_ctl** out);
int spec_depth_ctl_destroy(spec_depth_ctl* c);
/* The depth of the next round. */
int spec_depth_ctl_next(const spec_depth_ctl* c, int32_t* d);
/* A finished round: its depth d (in [d_min, d_max]), the n_seq accepted
 * counts (HOST int32, e.g. spec_verify_round's n_acc copied back) and its
 * time in seconds (finite, > 0).  *next_d (may be NULL) gets the next depth.
 * SPEC_E_SHAPE / SPEC_E_INVALID leave the controller unchanged. */
int spec_depth_ctl_observe(spec_depth_ctl* c, int32_t d, int32_t n_seq, const int32_t* n_acc,
                           double round_seconds, int32_t* next_d);
/* Diagnostics: p[0..d_max] (p[0] = 1) and r[0..d_max] (0 below d_min,
 * +infinity for depths without a round time); either may be NULL. */
int spec_depth_ctl_estimates(const spec_depth_ctl* c, double* p, double* r);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
