// api.cu -- the C ABI of the verify-round library: packed matrices, the
// decoder model object, per-sequence transaction state, the verify round
// (one weights-once target pass, accept, commit) and CUDA-graph replay.
//
// The round follows "Model-neutral Speculative Decoding", section "The
// exactness transaction", steps 3-6, and "Speculative Decoding (D5-R) --
// Plan", section 3 "Mechanism -- one round".  Step 1 (checkpoint) and step 7
// (restore) reduce to the per-sequence triple (n_past, emit_idx, anchor):
// the commit kernel is the only writer of that triple and it is skipped when
// the device error word is set, so a failed round leaves the last committed
// transaction in place; rejected KV rows need no restore because positions
// are data and are overwritten by the next round.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------
static thread_local std::string g_last_error;
void set_error(const std::string& msg) { g_last_error = msg; }
int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

extern "C" void spec_last_error(char* buf, size_t len) {
  if (buf == nullptr || len == 0) return;
  size_t n = std::min(len - 1, g_last_error.size());
  memcpy(buf, g_last_error.data(), n);
  buf[n] = '\0';
}

static cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Kernel attributes that must be set before any launch (and outside stream
// capture); once per device.
void attn_init_attrs();
void accept_init_attrs();
void linear_init_attrs();
void tc_init_attrs();
static std::mutex g_attr_mu;
static std::vector<int> g_attr_done;
static void init_attrs_once() {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (std::find(g_attr_done.begin(), g_attr_done.end(), dev) != g_attr_done.end()) return;
  attn_init_attrs();
  accept_init_attrs();
  linear_init_attrs();
  tc_init_attrs();
  g_attr_done.push_back(dev);
}

bool programmatic_launch() {
  static const bool on = [] {
    const char* e = std::getenv("SPEC_VERIFY_PDL");
    return !(e != nullptr && e[0] == '0');
  }();
  return on;
}

static int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// ---------------------------------------------------------------------------
// per-device workspace of the standalone entry points (grown on demand)
// ---------------------------------------------------------------------------
struct Workspace {
  StochScratch st;
  void* st_base = nullptr;
  uint32_t* err = nullptr;
};
static std::mutex g_ws_mu;
static std::map<int, Workspace> g_ws;

static int workspace_get(size_t rows, size_t seqs, Workspace** out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(g_ws_mu);
  Workspace& w = g_ws[dev];
  if (w.err == nullptr) {
    if (cudaMalloc(&w.err, sizeof(uint32_t)) != cudaSuccess) {
      cudaGetLastError();
      return fail(SPEC_E_OOM, "workspace error word");
    }
    CUDA_TRY(cudaMemset(w.err, 0, sizeof(uint32_t)));
  }
  if (rows > w.st.rows_cap || seqs > w.st.seq_cap) {
    rows = std::max(rows, w.st.rows_cap);
    seqs = std::max(seqs, w.st.seq_cap);
    if (w.st_base) {
      CUDA_TRY(cudaDeviceSynchronize());
      cudaFree(w.st_base);
      w.st_base = nullptr;
    }
    // each part starts on a 256-byte boundary (the decisions are 16-byte
    // int4 stores, whatever the row count)
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    const size_t sum_bytes = up(rows * sizeof(unsigned long long));
    const size_t dec_bytes = up(seqs * sizeof(int4));
    const size_t bytes = sum_bytes + dec_bytes + up(rows * sizeof(uint32_t));
    if (cudaMalloc(&w.st_base, bytes) != cudaSuccess) {
      cudaGetLastError();
      w.st = StochScratch();
      return fail(SPEC_E_OOM, "workspace");
    }
    char* p = (char*)w.st_base;
    w.st.row_sum = (unsigned long long*)p;
    w.st.decision = (int4*)(p + sum_bytes);
    w.st.row_key = (uint32_t*)(p + sum_bytes + dec_bytes);
    w.st.rows_cap = rows;
    w.st.seq_cap = seqs;
  }
  *out = &w;
  return SPEC_OK;
}

// ---------------------------------------------------------------------------
// packed matrices
// ---------------------------------------------------------------------------
struct spec_qmat {
  QMat w;
  int max_rows = 0;
  LinScratch scr;
  void* scr_base = nullptr;
};

static int alloc_lin_scratch(const std::vector<const QMat*>& mats, int R, LinScratch* scr,
                             void** base) {
  size_t part = 0, tick = 1, amax = 16;
  for (const QMat* q : mats) {
    part = std::max(part, lin_part_floats(*q, R));
    tick = std::max(tick, lin_tickets_needed(*q, R));
    amax = std::max(amax, lin_amax_entries(*q, R));
    part = std::max(part, tc_part_floats(*q, R));
    tick = std::max(tick, tc_tickets_needed(*q));
  }
  tick = std::max(tick, (size_t)64);
  const size_t keys = 256;  // packed argmax maxima of the tensor-core LM head
  const size_t bytes = keys * sizeof(unsigned long long) + part * sizeof(float) +
                       amax * sizeof(float2) + tick * sizeof(unsigned) + 16 + 256;
  if (cudaMalloc(base, bytes) != cudaSuccess) {
    cudaGetLastError();
    return fail(SPEC_E_OOM, "linear scratch");
  }
  char* p = (char*)*base;
  scr->amax_keys = (unsigned long long*)p;
  p += keys * sizeof(unsigned long long);
  scr->part = (float*)p;
  scr->part_floats = part;
  p += part * sizeof(float);
  scr->amax_part = (float2*)p;
  scr->amax_entries = amax;
  p += amax * sizeof(float2);
  scr->tickets = (unsigned*)p;
  scr->n_tickets = tick;
  p += tick * sizeof(unsigned);
  scr->err = (uint32_t*)p;  // the scratch's own error word (a model points it at its word)
  CUDA_TRY(cudaMemset(scr->tickets, 0, tick * sizeof(unsigned) + 16));
  CUDA_TRY(cudaMemset(scr->amax_keys, 0, keys * sizeof(unsigned long long)));
  return SPEC_OK;
}

extern "C" int spec_qmat_create(const spec_qweight* w, int max_rows, void* stream,
                                spec_qmat** out) {
  if (out == nullptr || w == nullptr) return fail(SPEC_E_INVALID, "null argument");
  *out = nullptr;
  if (max_rows < 1 || max_rows > 16 * 1024) return fail(SPEC_E_SHAPE, "max_rows out of range");
  init_attrs_once();
  cudaStream_t st = as_stream(stream);
  spec_qmat* m = new spec_qmat();
  int rc = qmat_pack(w, PERM_IDENTITY, 0, sm_count(), st, &m->w);
  if (rc != SPEC_OK) {
    delete m;
    return rc;
  }
  m->max_rows = max_rows;
  rc = alloc_lin_scratch({&m->w}, max_rows, &m->scr, &m->scr_base);
  if (rc == SPEC_OK) {
    // a copy that never arrives is reported through the standalone entry
    // points' error word (spec_error_check with no model)
    Workspace* ws = nullptr;
    rc = workspace_get(0, 0, &ws);
    if (rc == SPEC_OK) m->scr.err = ws->err;
  }
  if (rc == SPEC_OK && cudaStreamSynchronize(st) != cudaSuccess)
    rc = fail(SPEC_E_CUDA, std::string("repack: ") + cudaGetErrorString(cudaGetLastError()));
  if (rc != SPEC_OK) {
    qmat_free(&m->w);
    if (m->scr_base) cudaFree(m->scr_base);
    delete m;
    return rc;
  }
  *out = m;
  return SPEC_OK;
}

extern "C" int spec_qmat_destroy(spec_qmat* m) {
  if (m == nullptr) return SPEC_OK;
  cudaDeviceSynchronize();
  qmat_free(&m->w);
  if (m->scr_base) cudaFree(m->scr_base);
  delete m;
  return SPEC_OK;
}

extern "C" int spec_linear_q_tc(const spec_qmat* w, const uint16_t* x, int R, float* y,
                                void* stream) {
  if (w == nullptr || x == nullptr || y == nullptr) return fail(SPEC_E_INVALID, "null argument");
  if (R < 1 || R > w->max_rows) return fail(SPEC_E_SHAPE, "R outside [1, max_rows]");
  if (!aligned16(x)) return fail(SPEC_E_SHAPE, "x must be 16-byte aligned");
  LinEpi e;
  e.kind = EPI_STORE;
  e.y = y;
  e.ldy = w->w.N;
  return tc_linear_launch(w->w, reinterpret_cast<const __half*>(x), R, e, w->scr, as_stream(stream));
}

extern "C" int spec_linear_q(const spec_qmat* w, const uint16_t* x, int nt, float* y,
                             void* stream) {
  if (w == nullptr || x == nullptr || y == nullptr) return fail(SPEC_E_INVALID, "null argument");
  if (nt < 1 || nt > w->max_rows) return fail(SPEC_E_SHAPE, "nt outside [1, max_rows]");
  if (!aligned16(x)) return fail(SPEC_E_SHAPE, "x must be 16-byte aligned");
  LinEpi e;
  e.kind = EPI_STORE;
  e.y = y;
  e.ldy = w->w.N;
  return linear_launch(w->w, reinterpret_cast<const __half*>(x), nt, e, w->scr, as_stream(stream));
}

// ---------------------------------------------------------------------------
// model
// ---------------------------------------------------------------------------
// One instantiated verify graph.  The graph is kept beside its executable
// because the node handles belong to it; the caller's arrays are kernel
// arguments of the embedding node (draft, sequence ids) and, in a greedy
// round graph, of the accept + commit node, retargeted when they change.
struct RoundGraph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaGraphNode_t embed = nullptr;
  cudaGraphNode_t tail = nullptr;
  const int32_t* draft = nullptr;
  const int32_t* seq_ids = nullptr;
  int32_t* n_acc = nullptr;
  int32_t* emitted = nullptr;
};

static void round_graph_free(RoundGraph* g) {
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  *g = RoundGraph{};
}

struct spec_model {
  spec_model_desc d{};
  int device = 0, sms = 1;
  __half* embed = nullptr;
  float* norm_w = nullptr;
  std::vector<QMat> wqkv, wo, wgu, wd;
  QMat lm;
  __half* kc = nullptr;
  __half* vc = nullptr;
  size_t layer_elems = 0;  // per-layer cache elements
  float2* rope = nullptr;
  int32_t* n_past = nullptr;
  uint64_t* emit_idx = nullptr;
  int32_t* anchor = nullptr;
  uint32_t* err = nullptr;
  int Rmax = 0;
  float* h = nullptr;
  __half* xa = nullptr;   // norm output [R][H]
  __half* xs = nullptr;   // SwiGLU output [R][F]
  __half* qbuf = nullptr; // [R][nq][hd]
  __half* ao = nullptr;   // attention output [R][nq*hd]
  float* logits = nullptr;
  int32_t* argmax = nullptr;
  RowInfo* rows = nullptr;
  int32_t* tokens = nullptr;
  int32_t* seq_ids_buf = nullptr;
  int32_t* nacc_tmp = nullptr;
  // spec_verify_round_host: mapped pinned staging (the kernels read the
  // inputs and write the outputs there directly) and its device addresses,
  // each [max_seqs] sequence ids / accept counts then [max_seqs][max_nt] ids
  int32_t* io_host_in = nullptr;
  int32_t* io_host_out = nullptr;
  int32_t* io_dev_in = nullptr;
  int32_t* io_dev_out = nullptr;
  float* attn_part = nullptr;
  float* qhost_buf = nullptr;  // [max_seqs][max_nt - 1][vocab]: host q_logits of the host entry
  cudaStream_t q_stream = nullptr;  // their copy, beside the round's target pass
  cudaEvent_t q_done = nullptr;
  LinScratch lscr;
  StochScratch sscr;
  std::vector<void*> allocs;
  bool use_graphs = true;
  int tc_min_seqs = 2;  // rounds of at least this many sequences use the tensor-core GEMM
  // in-round kernel timing (spec_model_profile): events around each GEMM and
  // attention launch of raw-launched rounds
  struct ProfRec {
    cudaEvent_t a, b;
    int kind;
    double bytes, flops;
  };
  bool prof = false;
  std::vector<ProfRec> prof_recs;
  std::vector<cudaEvent_t> prof_pool;
  cudaStream_t cap_stream = nullptr;
  std::map<long long, RoundGraph> graphs;
  size_t weight_bytes = 0;
};

static int dalloc(spec_model* m, void** p, size_t bytes) {
  if (bytes == 0) bytes = 16;
  if (cudaMalloc(p, bytes) != cudaSuccess) {
    cudaGetLastError();
    return fail(SPEC_E_OOM, "cudaMalloc of " + std::to_string(bytes) + " bytes failed");
  }
  m->allocs.push_back(*p);
  return SPEC_OK;
}
template <typename T>
static int dalloc_t(spec_model* m, T** p, size_t count) {
  return dalloc(m, reinterpret_cast<void**>(p), count * sizeof(T));
}

static void model_free(spec_model* m) {
  cudaDeviceSynchronize();
  for (auto& r : m->prof_recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (cudaEvent_t e : m->prof_pool) cudaEventDestroy(e);
  for (auto& kv : m->graphs) round_graph_free(&kv.second);
  m->graphs.clear();
  for (auto* v : {&m->wqkv, &m->wo, &m->wgu, &m->wd})
    for (auto& q : *v) qmat_free(&q);
  qmat_free(&m->lm);
  for (void* p : m->allocs) cudaFree(p);
  m->allocs.clear();
  if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
  if (m->q_stream) cudaStreamDestroy(m->q_stream);
  if (m->q_done) cudaEventDestroy(m->q_done);
  if (m->io_host_in) cudaFreeHost(m->io_host_in);
  if (m->io_host_out) cudaFreeHost(m->io_host_out);
  delete m;
}

static int check_desc(const spec_model_desc* D, const spec_model_weights* W) {
  if (D == nullptr || W == nullptr) return fail(SPEC_E_INVALID, "null desc or weights");
  if (D->n_layers < 0 || D->hidden <= 0 || D->vocab <= 0 || D->max_nt < 1 ||
      D->max_nt > SPEC_MAX_NT || D->max_seqs < 1 || D->max_ctx < 1)
    return fail(SPEC_E_SHAPE, "bad model dimensions");
  if (D->max_ctx > 786432) return fail(SPEC_E_SHAPE, "max_ctx above 786432 is not supported");
  if (D->hidden % 64 != 0) return fail(SPEC_E_SHAPE, "hidden must be a multiple of 64");
  if (D->vocab % 16 != 0) return fail(SPEC_E_SHAPE, "vocab must be a multiple of 16");
  if (!(D->rms_eps >= 0.0f)) return fail(SPEC_E_INVALID, "rms_eps must be >= 0");
  if (D->n_layers > 0) {
    if (D->head_dim != 64 && D->head_dim != 128)
      return fail(SPEC_E_UNSUPPORTED, "head_dim must be 64 or 128");
    if (D->n_q_heads <= 0 || D->n_kv_heads <= 0 || D->n_q_heads % D->n_kv_heads != 0)
      return fail(SPEC_E_SHAPE, "n_q_heads must be a positive multiple of n_kv_heads");
    if (D->ffn <= 0 || D->ffn % 32 != 0) return fail(SPEC_E_SHAPE, "ffn must be a multiple of 32");
    if ((D->n_q_heads * D->head_dim) % 32 != 0) return fail(SPEC_E_SHAPE, "bad attention width");
    if (W->embed == nullptr || W->wqkv == nullptr || W->wo == nullptr || W->wgu == nullptr ||
        W->wd == nullptr)
      return fail(SPEC_E_INVALID, "missing layer weights");
    if (D->use_rope && !(D->rope_theta > 0.0f)) return fail(SPEC_E_INVALID, "rope_theta must be > 0");
    const int H = D->hidden, hd = D->head_dim, nq = D->n_q_heads, nkv = D->n_kv_heads, F = D->ffn;
    for (int l = 0; l < D->n_layers; l++) {
      if (W->wqkv[l].N != (nq + 2 * nkv) * hd || W->wqkv[l].K != H)
        return fail(SPEC_E_SHAPE, "wqkv shape");
      if (W->wo[l].N != H || W->wo[l].K != nq * hd) return fail(SPEC_E_SHAPE, "wo shape");
      if (W->wgu[l].N != 2 * F || W->wgu[l].K != H) return fail(SPEC_E_SHAPE, "wgu shape");
      if (W->wd[l].N != H || W->wd[l].K != F) return fail(SPEC_E_SHAPE, "wd shape");
    }
  }
  if (W->lm_head.N != D->vocab || W->lm_head.K != D->hidden) return fail(SPEC_E_SHAPE, "lm_head shape");
  if (W->norm_w == nullptr) return fail(SPEC_E_INVALID, "missing norm weights");
  return SPEC_OK;
}

extern "C" int spec_model_create(const spec_model_desc* desc, const spec_model_weights* w,
                                 void* stream, spec_model** out) {
  if (out == nullptr) return fail(SPEC_E_INVALID, "null out");
  *out = nullptr;
  int rc = check_desc(desc, w);
  if (rc != SPEC_OK) return rc;
  init_attrs_once();
  cudaStream_t st = as_stream(stream);
  spec_model* m = new spec_model();
  m->d = *desc;
  cudaGetDevice(&m->device);
  m->sms = sm_count();
  const spec_model_desc& D = m->d;
  const int L = D.n_layers, H = D.hidden, V = D.vocab, hd = D.head_dim, nq = D.n_q_heads,
            nkv = D.n_kv_heads, F = D.ffn;
  m->Rmax = D.max_seqs * D.max_nt;
  const int R = m->Rmax;
#define TRY(x)                 \
  do {                         \
    int rc_ = (x);             \
    if (rc_ != SPEC_OK) {      \
      model_free(m);           \
      return rc_;              \
    }                          \
  } while (0)
  // weights
  m->wqkv.resize(L);
  m->wo.resize(L);
  m->wgu.resize(L);
  m->wd.resize(L);
  for (int l = 0; l < L; l++) {
    TRY(qmat_pack(&w->wqkv[l], PERM_ROPE_PAIRS, hd, m->sms, st, &m->wqkv[l]));
    TRY(qmat_pack(&w->wo[l], PERM_IDENTITY, 0, m->sms, st, &m->wo[l]));
    TRY(qmat_pack(&w->wgu[l], PERM_GATE_UP, 0, m->sms, st, &m->wgu[l]));
    TRY(qmat_pack(&w->wd[l], PERM_IDENTITY, 0, m->sms, st, &m->wd[l]));
    m->weight_bytes += m->wqkv[l].bytes + m->wo[l].bytes + m->wgu[l].bytes + m->wd[l].bytes;
  }
  TRY(qmat_pack(&w->lm_head, PERM_IDENTITY, 0, m->sms, st, &m->lm));
  m->weight_bytes += m->lm.bytes;
  TRY(dalloc_t(m, &m->norm_w, (size_t)(2 * L + 1) * H));
  if (cudaMemcpyAsync(m->norm_w, w->norm_w, sizeof(float) * (2 * L + 1) * H,
                      cudaMemcpyDefault, st) != cudaSuccess)
    TRY(fail(SPEC_E_CUDA, "copy norm weights"));
  if (L > 0) {
    TRY(dalloc_t(m, &m->embed, (size_t)V * H));
    if (cudaMemcpyAsync(m->embed, w->embed, sizeof(__half) * V * H, cudaMemcpyDefault, st) !=
        cudaSuccess)
      TRY(fail(SPEC_E_CUDA, "copy embedding"));
    m->layer_elems = (size_t)D.max_seqs * nkv * D.max_ctx * hd;
    TRY(dalloc_t(m, &m->kc, m->layer_elems * L));
    TRY(dalloc_t(m, &m->vc, m->layer_elems * L));
    if (cudaMemsetAsync(m->kc, 0, sizeof(__half) * m->layer_elems * L, st) != cudaSuccess ||
        cudaMemsetAsync(m->vc, 0, sizeof(__half) * m->layer_elems * L, st) != cudaSuccess)
      TRY(fail(SPEC_E_CUDA, "clear KV cache"));
    TRY(dalloc_t(m, &m->rope, (size_t)D.max_ctx * (hd / 2)));
    launch_rope_table(m->rope, D.max_ctx, hd, D.rope_theta > 0 ? D.rope_theta : 10000.0f, st);
    TRY(dalloc_t(m, &m->qbuf, (size_t)R * nq * hd));
    TRY(dalloc_t(m, &m->ao, (size_t)R * nq * hd));
    TRY(dalloc_t(m, &m->xs, (size_t)R * F));
    TRY(dalloc_t(m, &m->attn_part, attn_part_floats(D.max_seqs, nkv, D.max_ctx, D.max_nt,
                                                    nq / nkv, hd)));
  }
  TRY(dalloc_t(m, &m->n_past, D.max_seqs));
  TRY(dalloc_t(m, &m->emit_idx, D.max_seqs));
  TRY(dalloc_t(m, &m->anchor, D.max_seqs));
  TRY(dalloc_t(m, &m->err, 1));
  cudaMemsetAsync(m->n_past, 0, sizeof(int32_t) * D.max_seqs, st);
  cudaMemsetAsync(m->emit_idx, 0, sizeof(uint64_t) * D.max_seqs, st);
  cudaMemsetAsync(m->anchor, 0, sizeof(int32_t) * D.max_seqs, st);
  cudaMemsetAsync(m->err, 0, sizeof(uint32_t), st);
  TRY(dalloc_t(m, &m->h, (size_t)R * H));
  TRY(dalloc_t(m, &m->xa, (size_t)R * H));
  TRY(dalloc_t(m, &m->logits, (size_t)R * V));
  if (D.max_nt > 1 && L > 0)
    TRY(dalloc_t(m, &m->qhost_buf, (size_t)D.max_seqs * (D.max_nt - 1) * V));
  TRY(dalloc_t(m, &m->argmax, R));
  TRY(dalloc_t(m, &m->rows, R));
  TRY(dalloc_t(m, &m->tokens, R));
  TRY(dalloc_t(m, &m->seq_ids_buf, D.max_seqs));
  TRY(dalloc_t(m, &m->nacc_tmp, D.max_seqs));
  {
    const size_t io = (size_t)D.max_seqs * (1 + D.max_nt);
    if (cudaHostAlloc(reinterpret_cast<void**>(&m->io_host_in), io * sizeof(int32_t),
                      cudaHostAllocMapped) != cudaSuccess ||
        cudaHostAlloc(reinterpret_cast<void**>(&m->io_host_out), io * sizeof(int32_t),
                      cudaHostAllocMapped) != cudaSuccess ||
        cudaHostGetDevicePointer(reinterpret_cast<void**>(&m->io_dev_in), m->io_host_in, 0) !=
            cudaSuccess ||
        cudaHostGetDevicePointer(reinterpret_cast<void**>(&m->io_dev_out), m->io_host_out, 0) !=
            cudaSuccess) {
      cudaGetLastError();
      TRY(fail(SPEC_E_OOM, "mapped pinned host staging"));
    }
  }
  // scratch
  std::vector<const QMat*> mats{&m->lm};
  for (int l = 0; l < L; l++) {
    mats.push_back(&m->wqkv[l]);
    mats.push_back(&m->wo[l]);
    mats.push_back(&m->wgu[l]);
    mats.push_back(&m->wd[l]);
  }
  {
    void* base = nullptr;
    TRY(alloc_lin_scratch(mats, R, &m->lscr, &base));
    m->allocs.push_back(base);
    m->lscr.err = m->err;
  }
  m->sscr.rows_cap = stoch_rows_needed(D.max_seqs, D.max_nt - 1);
  m->sscr.seq_cap = D.max_seqs;
  TRY(dalloc_t(m, &m->sscr.row_key, m->sscr.rows_cap));
  TRY(dalloc_t(m, &m->sscr.row_sum, m->sscr.rows_cap));
  TRY(dalloc_t(m, &m->sscr.decision, m->sscr.seq_cap));
  if (m->qhost_buf != nullptr &&
      (cudaStreamCreateWithFlags(&m->q_stream, cudaStreamNonBlocking) != cudaSuccess ||
       cudaEventCreateWithFlags(&m->q_done, cudaEventDisableTiming) != cudaSuccess)) {
    cudaGetLastError();
    TRY(fail(SPEC_E_CUDA, "q_logits copy stream"));
  }
  if (cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking) != cudaSuccess)
    TRY(fail(SPEC_E_CUDA, "capture stream"));
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) TRY(fail(SPEC_E_CUDA, std::string("model create: ") + cudaGetErrorString(e)));
#undef TRY
  *out = m;
  return SPEC_OK;
}

extern "C" int spec_model_destroy(spec_model* m) {
  if (m) model_free(m);
  return SPEC_OK;
}

extern "C" int spec_model_kv_cache(spec_model* m, int layer, uint16_t** k, uint16_t** v) {
  if (m == nullptr) return fail(SPEC_E_INVALID, "null model");
  if (layer < 0 || layer >= m->d.n_layers) return fail(SPEC_E_SHAPE, "layer out of range");
  if (k) *k = reinterpret_cast<uint16_t*>(m->kc + m->layer_elems * layer);
  if (v) *v = reinterpret_cast<uint16_t*>(m->vc + m->layer_elems * layer);
  return SPEC_OK;
}

extern "C" int spec_kv_fill(spec_model* m, int layer, int seq, int pos0, int n_pos,
                            const uint16_t* k, const uint16_t* v, void* stream) {
  if (m == nullptr || k == nullptr || v == nullptr) return fail(SPEC_E_INVALID, "null argument");
  const spec_model_desc& D = m->d;
  if (layer < 0 || layer >= D.n_layers || seq < 0 || seq >= D.max_seqs)
    return fail(SPEC_E_SHAPE, "layer or slot out of range");
  if (pos0 < 0 || n_pos < 0 || pos0 + n_pos > D.max_ctx) return fail(SPEC_E_SHAPE, "positions out of range");
  if (n_pos == 0) return SPEC_OK;
  const size_t row = (size_t)D.head_dim * sizeof(__half);
  for (int which = 0; which < 2; which++) {
    __half* base = (which == 0 ? m->kc : m->vc) + m->layer_elems * layer +
                   ((size_t)seq * D.n_kv_heads * D.max_ctx + pos0) * D.head_dim;
    const uint16_t* src = which == 0 ? k : v;
    // n_kv_heads blocks of n_pos rows; destination pitch max_ctx rows
    CUDA_TRY(cudaMemcpy2DAsync(base, row * D.max_ctx, src, row * n_pos, row * n_pos, D.n_kv_heads,
                               cudaMemcpyDefault, as_stream(stream)));
  }
  return SPEC_OK;
}

extern "C" int spec_kv_read(spec_model* m, int layer, int seq, int pos0, int n_pos, uint16_t* k,
                            uint16_t* v, void* stream) {
  if (m == nullptr || k == nullptr || v == nullptr) return fail(SPEC_E_INVALID, "null argument");
  const spec_model_desc& D = m->d;
  if (layer < 0 || layer >= D.n_layers || seq < 0 || seq >= D.max_seqs)
    return fail(SPEC_E_SHAPE, "layer or slot out of range");
  if (pos0 < 0 || n_pos < 0 || pos0 + n_pos > D.max_ctx) return fail(SPEC_E_SHAPE, "positions out of range");
  if (n_pos == 0) return SPEC_OK;
  const size_t row = (size_t)D.head_dim * sizeof(__half);
  for (int which = 0; which < 2; which++) {
    const __half* base = (which == 0 ? m->kc : m->vc) + m->layer_elems * layer +
                         ((size_t)seq * D.n_kv_heads * D.max_ctx + pos0) * D.head_dim;
    uint16_t* dst = which == 0 ? k : v;
    CUDA_TRY(cudaMemcpy2DAsync(dst, row * n_pos, base, row * D.max_ctx, row * n_pos, D.n_kv_heads,
                               cudaMemcpyDefault, as_stream(stream)));
  }
  return SPEC_OK;
}

extern "C" int spec_model_debug_read(spec_model* m, int which, void* dst, size_t bytes,
                                     void* stream) {
  if (m == nullptr || dst == nullptr) return fail(SPEC_E_INVALID, "null argument");
  const spec_model_desc& D = m->d;
  const size_t R = (size_t)m->Rmax;
  const void* src = nullptr;
  size_t cap = 0;
  switch (which) {
    case 0: src = m->h; cap = R * D.hidden * 4; break;
    case 1: src = m->xa; cap = R * D.hidden * 2; break;
    case 2: src = m->xs; cap = R * D.ffn * 2; break;
    case 3: src = m->ao; cap = R * D.n_q_heads * D.head_dim * 2; break;
    case 4: src = m->qbuf; cap = R * D.n_q_heads * D.head_dim * 2; break;
    case 5: src = m->logits; cap = R * D.vocab * 4; break;
    default: return fail(SPEC_E_INVALID, "unknown buffer");
  }
  if (src == nullptr) return fail(SPEC_E_UNSUPPORTED, "buffer not allocated for this model");
  CUDA_TRY(cudaMemcpyAsync(dst, src, std::min(bytes, cap), cudaMemcpyDefault, as_stream(stream)));
  return SPEC_OK;
}

extern "C" int spec_model_set_graphs(spec_model* m, int enable) {
  if (m == nullptr) return fail(SPEC_E_INVALID, "null model");
  m->use_graphs = enable != 0;
  return SPEC_OK;
}

extern "C" int spec_model_set_tc_min_seqs(spec_model* m, int min_seqs) {
  if (m == nullptr) return fail(SPEC_E_INVALID, "null model");
  if (min_seqs < 0) return fail(SPEC_E_INVALID, "min_seqs must be >= 0");
  if (min_seqs == m->tc_min_seqs) return SPEC_OK;
  CUDA_TRY(cudaDeviceSynchronize());
  for (auto& kv : m->graphs) round_graph_free(&kv.second);
  m->graphs.clear();
  m->tc_min_seqs = min_seqs;
  return SPEC_OK;
}

extern "C" int spec_model_profile(spec_model* m, int enable) {
  if (m == nullptr) return fail(SPEC_E_INVALID, "null model");
  CUDA_TRY(cudaDeviceSynchronize());
  for (auto& r : m->prof_recs) {
    m->prof_pool.push_back(r.a);
    m->prof_pool.push_back(r.b);
  }
  m->prof_recs.clear();
  m->prof = enable != 0;
  return SPEC_OK;
}

extern "C" int spec_model_profile_read(spec_model* m, int kind, double* seconds,
                                       int64_t* launches, double* bytes, double* flops) {
  if (m == nullptr) return fail(SPEC_E_INVALID, "null model");
  if (kind < 0 || kind > SPEC_PROF_ATTN) return fail(SPEC_E_INVALID, "unknown kernel class");
  CUDA_TRY(cudaDeviceSynchronize());
  double t = 0.0, b = 0.0, f = 0.0;
  int64_t n = 0;
  for (const auto& r : m->prof_recs) {
    const bool gemm = r.kind != SPEC_PROF_ATTN;
    if (!(r.kind == kind || (kind == SPEC_PROF_ALL_GEMMS && gemm))) continue;
    float ms = 0.0f;
    CUDA_TRY(cudaEventElapsedTime(&ms, r.a, r.b));
    t += ms * 1e-3;
    b += r.bytes;
    f += r.flops;
    n++;
  }
  if (seconds) *seconds = t;
  if (launches) *launches = n;
  if (bytes) *bytes = b;
  if (flops) *flops = f;
  return SPEC_OK;
}

extern "C" int spec_model_set_wait_budget(spec_model* m, int tries) {
  if (m == nullptr) return fail(SPEC_E_INVALID, "null model");
  if (tries < 0 || tries > LIN_WAIT_TRIES) return fail(SPEC_E_INVALID, "tries outside [0, 131072]");
  if (tries == m->lscr.wait_tries) return SPEC_OK;
  // the budget is a kernel argument: graphs captured with the old one go
  CUDA_TRY(cudaDeviceSynchronize());
  for (auto& kv : m->graphs) round_graph_free(&kv.second);
  m->graphs.clear();
  m->lscr.wait_tries = tries;
  return SPEC_OK;
}

extern "C" int spec_state_set(spec_model* m, int n, const int32_t* seq_ids,
                              const int32_t* n_past, const uint64_t* emit_idx,
                              const int32_t* anchor) {
  if (m == nullptr || (n > 0 && seq_ids == nullptr)) return fail(SPEC_E_INVALID, "null argument");
  for (int i = 0; i < n; i++) {
    const int s = seq_ids[i];
    if (s < 0 || s >= m->d.max_seqs) return fail(SPEC_E_INVALID, "sequence slot out of range");
    if (n_past && (n_past[i] < 0 || n_past[i] > m->d.max_ctx))
      return fail(SPEC_E_INVALID, "n_past out of range");
    if (anchor && (anchor[i] < 0 || anchor[i] >= m->d.vocab))
      return fail(SPEC_E_INVALID, "anchor id out of range");
  }
  for (int i = 0; i < n; i++) {
    const int s = seq_ids[i];
    if (n_past) CUDA_TRY(cudaMemcpy(m->n_past + s, n_past + i, 4, cudaMemcpyHostToDevice));
    if (emit_idx) CUDA_TRY(cudaMemcpy(m->emit_idx + s, emit_idx + i, 8, cudaMemcpyHostToDevice));
    if (anchor) CUDA_TRY(cudaMemcpy(m->anchor + s, anchor + i, 4, cudaMemcpyHostToDevice));
  }
  return SPEC_OK;
}

extern "C" int spec_state_get(spec_model* m, int n, const int32_t* seq_ids, int32_t* n_past,
                              uint64_t* emit_idx, int32_t* anchor) {
  if (m == nullptr || (n > 0 && seq_ids == nullptr)) return fail(SPEC_E_INVALID, "null argument");
  CUDA_TRY(cudaDeviceSynchronize());
  for (int i = 0; i < n; i++) {
    const int s = seq_ids[i];
    if (s < 0 || s >= m->d.max_seqs) return fail(SPEC_E_INVALID, "sequence slot out of range");
    if (n_past) CUDA_TRY(cudaMemcpy(n_past + i, m->n_past + s, 4, cudaMemcpyDeviceToHost));
    if (emit_idx) CUDA_TRY(cudaMemcpy(emit_idx + i, m->emit_idx + s, 8, cudaMemcpyDeviceToHost));
    if (anchor) CUDA_TRY(cudaMemcpy(anchor + i, m->anchor + s, 4, cudaMemcpyDeviceToHost));
  }
  return SPEC_OK;
}

extern "C" int spec_error_check(spec_model* m, void* stream, uint32_t* bits) {
  CUDA_TRY(cudaStreamSynchronize(as_stream(stream)));
  uint32_t* dev_err = nullptr;
  if (m != nullptr) {
    dev_err = m->err;
  } else {
    Workspace* w = nullptr;
    int rc = workspace_get(0, 0, &w);
    if (rc != SPEC_OK) return rc;
    dev_err = w->err;
  }
  uint32_t v = 0;
  CUDA_TRY(cudaMemcpy(&v, dev_err, 4, cudaMemcpyDeviceToHost));
  CUDA_TRY(cudaMemset(dev_err, 0, 4));
  if (bits) *bits = v;
  if (v != 0) return fail(SPEC_E_INVALID, "device error word set: 0x" + std::to_string(v));
  return SPEC_OK;
}

// ---------------------------------------------------------------------------
// the target pass
// ---------------------------------------------------------------------------
// The node that the last launch on a capturing stream created.
static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

static int last_captured_node(cudaStream_t st, cudaGraphNode_t* node) {
  cudaStreamCaptureStatus cs;
  const cudaGraphNode_t* deps = nullptr;
  size_t n = 0;
  CUDA_TRY(cudaStreamGetCaptureInfo(st, &cs, nullptr, nullptr, &deps, nullptr, &n));
  if (cs != cudaStreamCaptureStatusActive || n != 1)
    return fail(SPEC_E_CUDA, "graph capture: no single last node");
  *node = deps[0];
  return SPEC_OK;
}

// In-round timing: an event pair around one launch (profiling rounds only).
static cudaEvent_t prof_event(spec_model* m) {
  if (!m->prof_pool.empty()) {
    cudaEvent_t e = m->prof_pool.back();
    m->prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return e;
}
template <typename F>
static int timed_launch(spec_model* m, cudaStream_t st, int kind, double bytes, double flops,
                        F&& launch) {
  if (!m->prof) return launch();
  spec_model::ProfRec r{prof_event(m), prof_event(m), kind, bytes, flops};
  if (r.a) cudaEventRecord(r.a, st);
  const int rc = launch();
  if (r.b) cudaEventRecord(r.b, st);
  if (r.a && r.b) {
    m->prof_recs.push_back(r);
  } else {
    if (r.a) m->prof_pool.push_back(r.a);
    if (r.b) m->prof_pool.push_back(r.b);
  }
  return rc;
}
// Algorithmic bytes of one GEMM launch: the packed weights once, the fp16
// activations in, the outputs (fp32 or fp16) out.
static double gemm_bytes(const QMat& w, int R, int out_bytes) {
  return (double)w.bytes + (double)R * w.K * 2 + (double)R * w.N * out_bytes;
}

// The target pass over rows [anchor, draft[s][0..nt-2]] of each sequence;
// embed_node (capture only) receives the embedding node.
static int enqueue_forward(spec_model* m, int n_seq, int nt, const int32_t* draft,
                           const int32_t* seq_ids, bool write_logits, bool sampler_keys,
                           cudaStream_t st, cudaGraphNode_t* embed_node) {
  const spec_model_desc& D = m->d;
  // the GEMM is chosen by the number of sequences, never by nt: a round's
  // rows are bitwise the same at every depth d
  const bool tc = m->tc_min_seqs > 0 && n_seq >= m->tc_min_seqs;
  auto linear_launch = [tc](const QMat& w, const __half* x, int R, const LinEpi& e,
                            const LinScratch& scr, cudaStream_t s) {
    return tc ? tc_linear_launch(w, x, R, e, scr, s) : ::linear_launch(w, x, R, e, scr, s);
  };
  const int R = n_seq * nt, H = D.hidden, F = D.ffn, hd = D.head_dim, nq = D.n_q_heads,
            nkv = D.n_kv_heads, V = D.vocab;
  // the first RMSNorm runs inside the embedding kernel, the others as
  // their own kernels
  launch_embed_rows(m->embed, V, H, m->anchor, draft, seq_ids, n_seq, nt, m->n_past, D.max_seqs,
                    D.max_ctx, m->rows, m->tokens, m->h, m->norm_w, D.rms_eps, m->xa, m->err, st);
  if (embed_node != nullptr) {
    const int rc = last_captured_node(st, embed_node);
    if (rc != SPEC_OK) return rc;
  }
  for (int l = 0; l < D.n_layers; l++) {
    __half* kc = m->kc + m->layer_elems * l;
    __half* vc = m->vc + m->layer_elems * l;
    if (l > 0)
      launch_rmsnorm(m->h, m->norm_w + (size_t)(2 * l) * H, R, H, D.rms_eps, m->xa, st);
    LinEpi eq;
    eq.kind = EPI_QKV;
    eq.out16 = m->qbuf;
    eq.kcache = kc;
    eq.vcache = vc;
    eq.rows = m->rows;
    eq.rope = D.use_rope ? m->rope : nullptr;
    eq.nq = nq;
    eq.nkv = nkv;
    eq.hd = hd;
    eq.max_ctx = D.max_ctx;
    const QMat &wq = m->wqkv[l], &wo = m->wo[l], &wg = m->wgu[l], &wd = m->wd[l];
    auto flops = [R](const QMat& w) { return 2.0 * R * w.N * (double)w.K; };
    int rc = timed_launch(m, st, SPEC_PROF_QKV, gemm_bytes(wq, R, 2), flops(wq),
                          [&] { return linear_launch(wq, m->xa, R, eq, m->lscr, st); });
    if (rc) return rc;
    // attention: its bytes depend on the sequences' positions, which only
    // the device holds; the caller accounts for them
    rc = timed_launch(m, st, SPEC_PROF_ATTN, 0.0, 0.0, [&] {
                        return attn_launch(m->qbuf, kc, vc, m->rows, n_seq, nt, nq, nkv, hd,
                                           D.max_ctx, m->attn_part, m->ao, st);
                      });
    if (rc) return rc;
    LinEpi er;
    er.kind = EPI_RESID;
    er.y = m->h;
    er.ldy = H;
    rc = timed_launch(m, st, SPEC_PROF_O, gemm_bytes(wo, R, 8), flops(wo),
                      [&] { return linear_launch(wo, m->ao, R, er, m->lscr, st); });
    if (rc) return rc;
    launch_rmsnorm(m->h, m->norm_w + (size_t)(2 * l + 1) * H, R, H, D.rms_eps, m->xa, st);
    LinEpi es;
    es.kind = EPI_SWIGLU;
    es.out16 = m->xs;
    es.ldo = F;
    rc = timed_launch(m, st, SPEC_PROF_GATE_UP, gemm_bytes(wg, R, 1), flops(wg),
                      [&] { return linear_launch(wg, m->xa, R, es, m->lscr, st); });
    if (rc) return rc;
    rc = timed_launch(m, st, SPEC_PROF_DOWN, gemm_bytes(wd, R, 8), flops(wd),
                      [&] { return linear_launch(wd, m->xs, R, er, m->lscr, st); });
    if (rc) return rc;
  }
  if (D.n_layers > 0)
    launch_rmsnorm(m->h, m->norm_w + (size_t)(2 * D.n_layers) * H, R, H, D.rms_eps, m->xa, st);
  LinEpi el;
  el.kind = EPI_LMHEAD;
  el.y = write_logits ? m->logits : nullptr;
  el.ldy = V;
  el.argmax = m->argmax;
  el.err = m->err;
  if (sampler_keys) {  // a stochastic round: the sampler's row maxima come from here
    el.row_key = m->sscr.row_key;
    el.rk_nt = nt;
    el.rk_stride = 2 * nt - 1;
  }
  return timed_launch(m, st, SPEC_PROF_LM_HEAD, gemm_bytes(m->lm, R, write_logits ? 4 : 0),
                      2.0 * R * m->lm.N * (double)m->lm.K,
                      [&] { return linear_launch(m->lm, m->xa, R, el, m->lscr, st); });
}

// The target pass and, for a greedy round (greedy_tail), the fused accept +
// commit; replayed from a captured graph per (n_seq, d, logits, tail) when
// graphs are on.
static int run_round(spec_model* m, int n_seq, int d, const int32_t* draft, const int32_t* seq_ids,
                     bool write_logits, bool greedy_tail, int32_t* n_acc, int32_t* emitted,
                     cudaStream_t st, bool host_io = false) {
  // host_io: the arrays are the mapped staging's (a graph of its own, so
  // that it never needs retargeting)
  auto enqueue = [&](cudaStream_t s, cudaGraphNode_t* embed_node,
                     cudaGraphNode_t* tail_node) -> int {
    int rc = enqueue_forward(m, n_seq, d + 1, draft, seq_ids, write_logits,
                             write_logits && !greedy_tail, s, embed_node);
    if (rc != SPEC_OK || !greedy_tail) return rc;
    GreedyRoundArgs a;
    a.argmax = m->argmax;
    a.draft = draft;
    a.seq_ids = seq_ids;
    a.n_acc = n_acc;
    a.emitted = emitted;
    a.n_past = m->n_past;
    a.emit_idx = m->emit_idx;
    a.anchor = m->anchor;
    a.err = m->err;
    a.n_seq = n_seq;
    a.d = d;
    a.n_slots = m->d.max_seqs;
    launch_accept_commit_greedy(a, s);
    return tail_node != nullptr ? last_captured_node(s, tail_node) : SPEC_OK;
  };
  if (!m->use_graphs || m->prof) return enqueue(st, nullptr, nullptr);
  const long long key = ((long long)(host_io ? 1 : 0) << 40) | ((long long)n_seq << 20) |
                        ((long long)(d + 1) << 2) | (write_logits ? 2 : 0) | (greedy_tail ? 1 : 0);
  auto it = m->graphs.find(key);
  if (it != m->graphs.end()) {
    RoundGraph& g = it->second;
    const bool moved_in = g.draft != draft || g.seq_ids != seq_ids;
    const bool moved_out = greedy_tail && (g.n_acc != n_acc || g.emitted != emitted);
    bool ok = true;
    if (moved_in || moved_out) {
      ok = embed_node_retarget(g.exec, g.embed, draft, seq_ids) == cudaSuccess;
      if (ok && greedy_tail)
        ok = accept_commit_node_retarget(g.exec, g.tail, draft, seq_ids, n_acc, emitted) ==
             cudaSuccess;
    }
    if (ok) {
      g.draft = draft;
      g.seq_ids = seq_ids;
      g.n_acc = n_acc;
      g.emitted = emitted;
    } else {  // a node that cannot be updated: capture the graph again
      cudaGetLastError();
      round_graph_free(&g);
      m->graphs.erase(it);
      it = m->graphs.end();
    }
  }
  if (it == m->graphs.end()) {
    RoundGraph g;
    CUDA_TRY(cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal));
    int rc = enqueue(m->cap_stream, &g.embed, greedy_tail ? &g.tail : nullptr);
    cudaError_t e = cudaStreamEndCapture(m->cap_stream, &g.graph);
    if (rc != SPEC_OK || e != cudaSuccess) {
      round_graph_free(&g);
      if (rc != SPEC_OK) return rc;
      return fail(SPEC_E_CUDA, std::string("graph capture: ") + cudaGetErrorString(e));
    }
    e = cudaGraphInstantiate(&g.exec, g.graph, 0);
    if (e != cudaSuccess) {
      round_graph_free(&g);
      return fail(SPEC_E_CUDA, std::string("graph instantiate: ") + cudaGetErrorString(e));
    }
    g.draft = draft;
    g.seq_ids = seq_ids;
    g.n_acc = n_acc;
    g.emitted = emitted;
    it = m->graphs.emplace(key, g).first;
  }
  CUDA_TRY(cudaGraphLaunch(it->second.exec, st));
  return SPEC_OK;
}

extern "C" int spec_verify_round(spec_model* m, int n_seq, const int32_t* seq_ids,
                                 const int32_t* draft, int d, const float* q_logits,
                                 const spec_sampling* sampling, int32_t* n_acc,
                                 int32_t* emitted, float* logits_out, void* stream) {
  if (m == nullptr || seq_ids == nullptr || sampling == nullptr || n_acc == nullptr ||
      emitted == nullptr)
    return fail(SPEC_E_INVALID, "null argument");
  const spec_model_desc& D = m->d;
  if (D.n_layers == 0) return fail(SPEC_E_UNSUPPORTED, "verify round needs a decoder (n_layers > 0)");
  if (n_seq < 1 || n_seq > D.max_seqs) return fail(SPEC_E_SHAPE, "n_seq outside [1, max_seqs]");
  if (d < 0 || d + 1 > D.max_nt) return fail(SPEC_E_SHAPE, "d + 1 outside [1, max_nt]");
  if (d > 0 && draft == nullptr) return fail(SPEC_E_INVALID, "null draft");
  const bool greedy = sampling->greedy != 0;
  if (!greedy) {
    if (!(sampling->temperature > 0.0f) || !std::isfinite(sampling->temperature))
      return fail(SPEC_E_INVALID, "temperature must be finite and > 0");
    if (d > 0 && q_logits == nullptr) return fail(SPEC_E_INVALID, "stochastic accept needs q_logits");
  } else if (q_logits != nullptr) {
    return fail(SPEC_E_INVALID, "q_logits must be NULL in greedy mode");
  }
  // the kernels read seq_ids and draft in place and write n_acc and emitted
  const size_t in_ids = sizeof(int32_t) * n_seq, in_draft = sizeof(int32_t) * n_seq * d,
               out_em = sizeof(int32_t) * n_seq * (d + 1);
  if (overlaps(emitted, out_em, seq_ids, in_ids) || overlaps(emitted, out_em, draft, in_draft) ||
      overlaps(n_acc, in_ids, seq_ids, in_ids) || overlaps(n_acc, in_ids, draft, in_draft) ||
      overlaps(n_acc, in_ids, emitted, out_em))
    return fail(SPEC_E_INVALID, "n_acc / emitted overlap each other or seq_ids / draft");
  cudaStream_t st = as_stream(stream);
  const int nt = d + 1;
  const bool write_logits = !greedy || logits_out != nullptr;
  int rc = run_round(m, n_seq, d, draft, seq_ids, write_logits, greedy, n_acc, emitted, st);
  if (rc != SPEC_OK) return rc;
  if (!greedy) {
    rc = launch_accept_stochastic(m->logits, q_logits, draft, n_seq, d, D.vocab,
                                  sampling->temperature, sampling->seed, seq_ids, m->emit_idx, 1,
                                  D.max_seqs, m->nacc_tmp, emitted, m->sscr, m->err, st, true);
    if (rc != SPEC_OK) return rc;
    launch_commit(seq_ids, n_seq, d, D.max_seqs, m->nacc_tmp, n_acc, emitted, m->n_past,
                  m->emit_idx, m->anchor, m->err, st);
  }
  if (logits_out != nullptr)
    CUDA_TRY(cudaMemcpyAsync(logits_out, m->logits, sizeof(float) * n_seq * nt * D.vocab,
                             cudaMemcpyDeviceToDevice, st));
  CUDA_TRY(cudaGetLastError());
  return SPEC_OK;
}

extern "C" int spec_verify_round_host(spec_model* m, int n_seq, const int32_t* seq_ids,
                                      const int32_t* draft, int d, const float* q_logits,
                                      const spec_sampling* sampling, int32_t* n_acc,
                                      int32_t* emitted, void* stream) {
  if (m == nullptr || seq_ids == nullptr || sampling == nullptr || n_acc == nullptr ||
      emitted == nullptr)
    return fail(SPEC_E_INVALID, "null argument");
  const spec_model_desc& D = m->d;
  if (D.n_layers == 0) return fail(SPEC_E_UNSUPPORTED, "verify round needs a decoder (n_layers > 0)");
  if (n_seq < 1 || n_seq > D.max_seqs) return fail(SPEC_E_SHAPE, "n_seq outside [1, max_seqs]");
  if (d < 0 || d + 1 > D.max_nt) return fail(SPEC_E_SHAPE, "d + 1 outside [1, max_nt]");
  if (d > 0 && draft == nullptr) return fail(SPEC_E_INVALID, "null draft");
  const bool greedy = sampling->greedy != 0;
  if (!greedy) {
    if (!(sampling->temperature > 0.0f) || !std::isfinite(sampling->temperature))
      return fail(SPEC_E_INVALID, "temperature must be finite and > 0");
    if (d > 0 && q_logits == nullptr) return fail(SPEC_E_INVALID, "stochastic accept needs q_logits");
  } else if (q_logits != nullptr) {
    return fail(SPEC_E_INVALID, "q_logits must be NULL in greedy mode");
  }
  cudaStream_t st = as_stream(stream);
  // q_logits in host memory are copied into the model's buffer first
  bool q_from_host = false;
  if (!greedy && d > 0) {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, q_logits) != cudaSuccess) {
      cudaGetLastError();
      pa.type = cudaMemoryTypeUnregistered;
    }
    if (pa.type != cudaMemoryTypeDevice && pa.type != cudaMemoryTypeManaged) {
      // on the model's copy stream, beside the target pass (which does not
      // read them); the accept waits for it.  The buffer is free: every call
      // has synchronised before returning.
      CUDA_TRY(cudaMemcpyAsync(m->qhost_buf, q_logits, sizeof(float) * n_seq * d * D.vocab,
                               cudaMemcpyHostToDevice, m->q_stream));
      CUDA_TRY(cudaEventRecord(m->q_done, m->q_stream));
      q_from_host = true;
      q_logits = m->qhost_buf;
    }
  }
  // the staging is free: every call has synchronised before returning
  std::memcpy(m->io_host_in, seq_ids, sizeof(int32_t) * n_seq);
  if (d > 0) std::memcpy(m->io_host_in + n_seq, draft, sizeof(int32_t) * n_seq * d);
  const int32_t* dseq = m->io_dev_in;
  const int32_t* ddraft = d > 0 ? m->io_dev_in + n_seq : nullptr;
  int32_t* dacc = m->io_dev_out;
  int32_t* dem = m->io_dev_out + n_seq;
  int rc = run_round(m, n_seq, d, ddraft, dseq, !greedy, greedy, dacc, dem, st, true);
  if (rc != SPEC_OK) {
    if (q_from_host) cudaStreamSynchronize(m->q_stream);
    return rc;
  }
  if (!greedy) {
    if (q_from_host) CUDA_TRY(cudaStreamWaitEvent(st, m->q_done, 0));
    rc = launch_accept_stochastic(m->logits, q_logits, ddraft, n_seq, d, D.vocab,
                                  sampling->temperature, sampling->seed, dseq, m->emit_idx, 1,
                                  D.max_seqs, m->nacc_tmp, dem, m->sscr, m->err, st, true);
    if (rc != SPEC_OK) {
      cudaStreamSynchronize(st);
      return rc;
    }
    launch_commit(dseq, n_seq, d, D.max_seqs, m->nacc_tmp, dacc, dem, m->n_past, m->emit_idx,
                  m->anchor, m->err, st);
  }
  CUDA_TRY(cudaStreamSynchronize(st));
  std::memcpy(n_acc, m->io_host_out, sizeof(int32_t) * n_seq);
  std::memcpy(emitted, m->io_host_out + n_seq, sizeof(int32_t) * n_seq * (d + 1));
  return SPEC_OK;
}

// ---------------------------------------------------------------------------
// standalone steps
// ---------------------------------------------------------------------------
extern "C" int spec_verify_attn(spec_model* m, int layer, int n_seq, const int32_t* seq_ids,
                                int nt, const uint16_t* q, const uint16_t* k_new,
                                const uint16_t* v_new, uint16_t* out, void* stream) {
  if (m == nullptr || seq_ids == nullptr || q == nullptr || k_new == nullptr ||
      v_new == nullptr || out == nullptr)
    return fail(SPEC_E_INVALID, "null argument");
  const spec_model_desc& D = m->d;
  if (layer < 0 || layer >= D.n_layers) return fail(SPEC_E_SHAPE, "layer out of range");
  if (n_seq < 1 || n_seq > D.max_seqs || nt < 1 || nt > D.max_nt)
    return fail(SPEC_E_SHAPE, "n_seq or nt out of range");
  if (!aligned16(q) || !aligned16(out)) return fail(SPEC_E_SHAPE, "q/out must be 16-byte aligned");
  cudaStream_t st = as_stream(stream);
  CUDA_TRY(cudaMemcpyAsync(m->seq_ids_buf, seq_ids, sizeof(int32_t) * n_seq,
                           cudaMemcpyDeviceToDevice, st));
  launch_row_info(m->seq_ids_buf, n_seq, nt, m->n_past, D.max_seqs, D.max_ctx, m->rows, m->err, st);
  __half* kc = m->kc + m->layer_elems * layer;
  __half* vc = m->vc + m->layer_elems * layer;
  launch_kv_write(reinterpret_cast<const __half*>(k_new), reinterpret_cast<const __half*>(v_new),
                  m->rows, n_seq * nt, D.n_kv_heads, D.head_dim, D.max_ctx, kc, vc, st);
  return attn_launch(reinterpret_cast<const __half*>(q), kc, vc, m->rows, n_seq, nt, D.n_q_heads,
                     D.n_kv_heads, D.head_dim, D.max_ctx, m->attn_part,
                     reinterpret_cast<__half*>(out), st);
}

extern "C" int spec_lm_head(spec_model* m, const uint16_t* x, int R, float* logits,
                            int32_t* argmax, void* stream) {
  if (m == nullptr || x == nullptr) return fail(SPEC_E_INVALID, "null argument");
  if (R < 1 || R > m->Rmax) return fail(SPEC_E_SHAPE, "R outside [1, max_seqs*max_nt]");
  if (!aligned16(x)) return fail(SPEC_E_SHAPE, "x must be 16-byte aligned");
  LinEpi e;
  e.kind = EPI_LMHEAD;
  e.y = logits;
  e.ldy = m->d.vocab;
  e.argmax = argmax != nullptr ? argmax : m->argmax;
  e.err = m->err;
  return linear_launch(m->lm, reinterpret_cast<const __half*>(x), R, e, m->lscr, as_stream(stream));
}

extern "C" int spec_accept_greedy(const int32_t* argmax, const int32_t* draft, int n_seq, int d,
                                  int32_t* n_acc, int32_t* emitted, void* stream) {
  if (argmax == nullptr || n_acc == nullptr || emitted == nullptr || (d > 0 && draft == nullptr))
    return fail(SPEC_E_INVALID, "null argument");
  if (n_seq < 1 || d < 0) return fail(SPEC_E_SHAPE, "n_seq >= 1 and d >= 0 required");
  launch_accept_greedy(argmax, draft, n_seq, d, n_acc, emitted, as_stream(stream));
  CUDA_TRY(cudaGetLastError());
  return SPEC_OK;
}

void stoch_finalize(int n_seq, int d, int32_t* n_acc, int32_t* emitted, uint64_t* emit_idx,
                    const uint32_t* err, cudaStream_t st);

extern "C" int spec_accept_stochastic(const float* p_logits, const float* q_logits,
                                      const int32_t* draft, int n_seq, int d, int V,
                                      float temperature, uint64_t seed, const int32_t* seq_ids,
                                      uint64_t* emit_idx, int32_t* n_acc, int32_t* emitted,
                                      void* stream) {
  if (p_logits == nullptr || seq_ids == nullptr || emit_idx == nullptr || n_acc == nullptr ||
      emitted == nullptr || (d > 0 && (draft == nullptr || q_logits == nullptr)))
    return fail(SPEC_E_INVALID, "null argument");
  if (n_seq < 1 || d < 0 || V < 1) return fail(SPEC_E_SHAPE, "n_seq >= 1, d >= 0, V >= 1 required");
  if (!(temperature > 0.0f) || !std::isfinite(temperature))
    return fail(SPEC_E_INVALID, "temperature must be finite and > 0");
  init_attrs_once();  // the row-statistics kernel's shared-memory limit
  Workspace* w = nullptr;
  int rc = workspace_get(stoch_rows_needed(n_seq, d), n_seq, &w);
  if (rc != SPEC_OK) return rc;
  cudaStream_t st = as_stream(stream);
  rc = launch_accept_stochastic(p_logits, q_logits, draft, n_seq, d, V, temperature, seed, seq_ids,
                                emit_idx, 0, 0, n_acc, emitted, w->st, w->err, st);
  if (rc != SPEC_OK) return rc;
  stoch_finalize(n_seq, d, n_acc, emitted, emit_idx, w->err, st);
  CUDA_TRY(cudaGetLastError());
  return SPEC_OK;
}
