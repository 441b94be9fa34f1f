// common.cuh -- internal declarations shared by the CUDA translation units of
// the verify-round library (sm_103a).  Not part of the public ABI.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/spec_verify.h"

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------
// Device error-word bits (atomicOr'd by kernels; never trap).
enum : uint32_t {
  ERR_TOKEN = 1u << 0,     // token id outside [0, vocab)
  ERR_POS = 1u << 1,       // n_past + nt > max_ctx
  ERR_NONFINITE = 1u << 2, // NaN/Inf logit
  ERR_SEQ = 1u << 3,       // sequence slot outside [0, max_seqs), or named twice in a round
  ERR_TIMEOUT = 1u << 4,   // a bounded wait gave up
};

void set_error(const std::string& msg);
int fail(int code, const std::string& msg);
#define CUDA_TRY(expr)                                                       \
  do {                                                                       \
    cudaError_t e_ = (expr);                                                 \
    if (e_ != cudaSuccess)                                                   \
      return fail(SPEC_E_CUDA, std::string(#expr ": ") + cudaGetErrorString(e_)); \
  } while (0)

// ---------------------------------------------------------------------------
// packed (streaming) layout of a block-quantised matrix
// ---------------------------------------------------------------------------
// The matrix is cut into tiles of 16 output rows, grouped in pairs of two
// tiles (one warp's work), and chunks of 64 along K (two quantisation
// blocks).  Each (pair, chunk) is one contiguous record:
//   [2 x 512 B nibble words][2 x 64 B fp16 scales][Q6: 2 x 256 B high fields]
// For tile i of the quad and lane l = 4g + t, the 16-byte nibble vector at
// i*512 + 16l holds the four k16 steps' mma.m16n8k16 A-fragment words of rows
// g / g+8 (k order inside each 32-block permuted so that lane t reads 8
// consecutive activations); the scales at 1024 + i*64 + 8g are (row g, blk0),
// (row g+8, blk0), (g, blk1), (g+8, blk1); the Q6 high fields at
// 1152 + i*256 + 8l are one word per block, pre-positioned for the
// magic-number merge.  K is zero-padded to a multiple of 64 and N to a
// multiple of 32 rows (padding weights have q = 0, scale 0).
struct QMat {
  int qtype = 0;
  int N = 0, K = 0, Kp = 0;
  int nch = 0;       // Kp / 64
  int n_tiles = 0;   // N / 16
  int n_pairs = 0;   // ceil(n_tiles / 2): one warp's tiles
  int n_grp = 0;     // CTA tile groups (8 / kw pairs each)
  int rec_bytes = 0; // 1152 (Q4) or 1664 (Q6)
  int kw = 1;        // warps sharing one pair's K range inside a CTA
  int S = 1;         // K segments across CTAs
  int nc_cta = 0;    // chunks of one CTA's K range (at most)
                     // (kw, S) are fixed per matrix: independent of nt
  int tc_P = 1;      // CTAs (runs of work) of the tensor-core GEMM (multi-sequence rounds)
  int tc_H = 2;      // 128-row halves of a tensor-core GEMM CTA (1 or 2)
  uint8_t* rec = nullptr;  // [n_pairs][nch][rec_bytes]
  void* base = nullptr;    // single allocation
  size_t bytes = 0;        // streamed bytes
};

// Row permutation applied at repack: packed row p <- canonical row perm(p).
enum PermKind { PERM_IDENTITY = 0, PERM_ROPE_PAIRS = 1, PERM_GATE_UP = 2 };

// sms: SM count of the device (sets the stream-K worker count).
int qmat_pack(const spec_qweight* w, PermKind perm, int head_dim, int sms, cudaStream_t st,
              QMat* out);
void qmat_free(QMat* q);

// Epilogue kinds of the verify GEMM.
enum EpiKind {
  EPI_STORE = 0,   // y[r][n] = acc (fp32)
  EPI_RESID = 1,   // y[r][n] += acc (fp32 residual stream)
  EPI_SWIGLU = 2,  // out16[r][j] = silu(gate) * up (gate/up interleaved by 8 rows)
  EPI_QKV = 3,     // RoPE on q/k pairs, q -> fp16 buffer, k/v -> KV cache
  EPI_LMHEAD = 4,  // optional fp32 logits + fused per-row argmax
};

struct RowInfo {  // per verify row: sequence slot and absolute position
  int slot;
  int pos;
};

struct LinEpi {
  EpiKind kind = EPI_STORE;
  float* y = nullptr;        // STORE/RESID/LMHEAD logits (may be null for LMHEAD)
  int ldy = 0;               // row stride of y (elements)
  __half* out16 = nullptr;   // SWIGLU output [R][ldo] / QKV q output [R][nq*hd]
  int ldo = 0;
  // QKV
  __half* kcache = nullptr;  // layer base [max_seqs][nkv][max_ctx][hd]
  __half* vcache = nullptr;
  const RowInfo* rows = nullptr;
  const float2* rope = nullptr;  // [max_ctx][hd/2] (cos, sin), null = no rope
  int nq = 0, nkv = 0, hd = 0, max_ctx = 0;
  // LMHEAD
  int32_t* argmax = nullptr;
  uint32_t* err = nullptr;
  // LMHEAD of a stochastic round: each logits row's order key of its largest
  // logit (the sampler's maximum) goes to the accept's per-row keys, where
  // row r (sequence r / rk_nt, row r % rk_nt) is entry
  // (r / rk_nt) * rk_stride + r % rk_nt, and the same sequence's draft-row
  // entries rk_nt .. rk_stride - 1 are zeroed for the accept's max pass;
  // rk_row0 is the global index of this launch's row 0
  uint32_t* row_key = nullptr;
  int rk_row0 = 0, rk_nt = 1, rk_stride = 1;
};

// Order-preserving 32-bit key of a float (-0 taken as +0): the key of the
// largest logit of a row, shared by the LM head's argmax and the sampler.
__device__ __forceinline__ uint32_t logit_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// The LM head's sampler outputs for one of its rows (see LinEpi::row_key).
__device__ __forceinline__ void write_row_key(const LinEpi& e, int r, uint32_t key) {
  const int g = e.rk_row0 + r, s = g / e.rk_nt, i = g - s * e.rk_nt;
  uint32_t* k = e.row_key + (size_t)s * e.rk_stride;
  k[i] = key;
  if (i < e.rk_stride - e.rk_nt) k[e.rk_nt + i] = 0u;  // draft row i of the sequence
}

// Tries of a bounded mbarrier wait (each suspends for at most ~10 us):
// about a second in all.
constexpr int LIN_WAIT_TRIES = 1 << 17;

struct LinScratch {
  int wait_tries = LIN_WAIT_TRIES;  // budget of a GEMM's first copy wait
  float* part = nullptr;         // K-split partials
  size_t part_floats = 0;
  unsigned* tickets = nullptr;   // zero-initialised, reset by their last user
  size_t n_tickets = 0;
  float2* amax_part = nullptr;   // LM-head argmax partials (value, index bits)
  size_t amax_entries = 0;
  unsigned long long* amax_keys = nullptr;  // [256] packed maxima of the tensor-core LM head (zeroed)
  uint32_t* err = nullptr;       // device error word
};

size_t lin_part_floats(const QMat& w, int R);
size_t lin_tickets_needed(const QMat& w, int R);
size_t lin_amax_entries(const QMat& w, int R);
int linear_launch(const QMat& w, const __half* x, int R, const LinEpi& epi,
                  const LinScratch& scr, cudaStream_t st);

// The tensor-core (tcgen05) verify GEMM of multi-sequence rounds (tcgemm.cu):
// 1 <= R <= 256 rows per launch, the same epilogues.
int tc_npad(int R);
int tc_choose_halves(int N, int nch, int sms);
int tc_choose_ctas(int N, int nch, int sms, int halves);
size_t tc_part_floats(const QMat& w, int R);
size_t tc_tickets_needed(const QMat& w);
int tc_linear_launch(const QMat& w, const __half* x, int R, const LinEpi& epi,
                     const LinScratch& scr, cudaStream_t st);

// ---------------------------------------------------------------------------
// small ops (ops.cu)
// ---------------------------------------------------------------------------
struct EmbedArgs {
  const __half* embed;
  const int32_t* anchor;   // [max_seqs]
  const int32_t* draft;    // [n_seq][nt - 1]
  const int32_t* seq_ids;  // [n_seq]
  const int32_t* n_past;   // [max_seqs]
  RowInfo* rows;           // [n_seq * nt]
  int32_t* tokens;         // [n_seq * nt]
  float* h;                // [n_seq * nt][H]
  uint32_t* err;
  const float* gamma;  // the first RMSNorm's gains [H]
  __half* xn;          // its output [n_seq * nt][H]
  float eps;
  int V, H, nt, max_seqs, max_ctx;
};
// Embedding rows into h and, fused, the first RMSNorm of h into xn.
void launch_embed_rows(const __half* embed, int V, int H, const int32_t* anchor,
                       const int32_t* draft, const int32_t* seq_ids, int n_seq,
                       int nt, const int32_t* n_past, int max_seqs, int max_ctx,
                       RowInfo* rows, int32_t* tokens, float* h, const float* gamma,
                       float eps, __half* xn, uint32_t* err, cudaStream_t st);
// Points the embedding node of an instantiated graph (captured from
// launch_embed_rows) at new draft and sequence-id arrays; the other arguments
// keep their captured values.
cudaError_t embed_node_retarget(cudaGraphExec_t ex, cudaGraphNode_t node, const int32_t* draft,
                                const int32_t* seq_ids);
void launch_rmsnorm(const float* h, const float* gamma, int R, int H, float eps,
                    __half* out, cudaStream_t st);
void launch_rope_table(float2* tab, int max_ctx, int hd, float theta, cudaStream_t st);
void launch_kv_write(const __half* k_new, const __half* v_new, const RowInfo* rows,
                     int R, int nkv, int hd, int max_ctx, __half* kcache,
                     __half* vcache, cudaStream_t st);
void launch_row_info(const int32_t* seq_ids, int n_seq, int nt,
                     const int32_t* n_past, int max_seqs, int max_ctx,
                     RowInfo* rows, uint32_t* err, cudaStream_t st);

// ---------------------------------------------------------------------------
// attention (attn.cu)
// ---------------------------------------------------------------------------
constexpr int ATTN_CHUNK = 128;  // positions per chunk, at absolute multiples
size_t attn_part_floats(int max_seqs, int nkv, int max_ctx, int max_nt, int group, int hd);
int attn_launch(const __half* q, const __half* kcache, const __half* vcache,
                const RowInfo* rows, int n_seq, int nt, int nq, int nkv, int hd,
                int max_ctx, float* part, __half* out, cudaStream_t st);

// ---------------------------------------------------------------------------
// accept (accept.cu)
// ---------------------------------------------------------------------------
struct StochScratch {
  uint32_t* row_key = nullptr;         // [n_seq][2d+1]: order key of the row's largest logit
  unsigned long long* row_sum = nullptr;  // [n_seq][2d+1]
  int4* decision = nullptr;            // [n_seq]: (a, row, U2, flags)
  size_t rows_cap = 0;
  size_t seq_cap = 0;
};
size_t stoch_rows_needed(int n_seq, int d);
void launch_accept_greedy(const int32_t* argmax, const int32_t* draft, int n_seq,
                          int d, int32_t* n_acc, int32_t* emitted, cudaStream_t st);
// p_keys_ready: the p rows' maximum keys are already in scr.row_key and the
// q rows' keys zeroed (written by the round's LM head, LinEpi::row_key), so
// only the q rows get a max pass.
int launch_accept_stochastic(const float* p, const float* q, const int32_t* draft,
                             int n_seq, int d, int V, float T, uint64_t seed,
                             const int32_t* seq_ids, uint64_t* emit_idx,
                             int emit_by_slot, int n_slots, int32_t* n_acc,
                             int32_t* emitted, const StochScratch& scr,
                             uint32_t* err, cudaStream_t st, bool p_keys_ready = false);
void launch_commit(const int32_t* seq_ids, int n_seq, int d, int n_slots, const int32_t* n_acc_in,
                   int32_t* n_acc, int32_t* emitted, int32_t* n_past,
                   uint64_t* emit_idx, int32_t* anchor, const uint32_t* err,
                   cudaStream_t st);

// Greedy accept fused with the commit (the verify round's tail).
struct GreedyRoundArgs {
  const int32_t* argmax;   // [n_seq][d + 1]
  const int32_t* draft;    // [n_seq][d]
  const int32_t* seq_ids;  // [n_seq]
  int32_t* n_acc;          // [n_seq]
  int32_t* emitted;        // [n_seq][d + 1]
  int32_t* n_past;         // [n_slots]
  uint64_t* emit_idx;      // [n_slots]
  int32_t* anchor;         // [n_slots]
  const uint32_t* err;
  int n_seq, d, n_slots;
};
void launch_accept_commit_greedy(const GreedyRoundArgs& a, cudaStream_t st);
// Points the tail node of an instantiated round graph (captured from
// launch_accept_commit_greedy) at new input and output arrays.
cudaError_t accept_commit_node_retarget(cudaGraphExec_t ex, cudaGraphNode_t node,
                                        const int32_t* draft, const int32_t* seq_ids,
                                        int32_t* n_acc, int32_t* emitted);

// Whether kernels that can overlap their predecessor's tail are launched as
// programmatic dependents (default on; SPEC_VERIFY_PDL=0 in the environment
// turns it off).
bool programmatic_launch();

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;  // (a & b) | c
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4],
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_16816_c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                            uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ void mma_16816_zero(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// Programmatic dependent launch.  grid_dep_wait blocks until the grids this
// one depends on have completed and their writes are visible (it returns at
// once for a plain launch); grid_dep_launch lets the stream's next kernel,
// if it was launched programmatically, start before this grid completes.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_stream2(const uint2* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
#endif
