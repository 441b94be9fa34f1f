// ops.cu -- small per-row kernels of the verify pass: row bookkeeping and
// embedding gather, RMSNorm to fp16, the RoPE table and the KV write of the
// standalone attention entry point.
//
// Row layout of one verify round ("Speculative Decoding (D5-R) -- Plan",
// section 3): sequence s contributes rows [anchor, x_1 .. x_d] at the
// contiguous absolute positions n_past[s] .. n_past[s] + d.
#include <math.h>

#include "common.cuh"

namespace {

// Rows of up to NORM_REG_VEC * 1024 values are normalised from registers.
constexpr int NORM_REG_VEC = 8;

// Row r = (sequence s, offset i): the sequence's slot (checked) and the
// row's absolute position n_past[slot] + i (checked against max_ctx; an
// invalid position becomes max_ctx, where consumers write nothing).
__device__ __forceinline__ RowInfo row_info(const int32_t* __restrict__ seq_ids, int r, int nt,
                                            const int32_t* __restrict__ n_past, int max_seqs,
                                            int max_ctx, uint32_t* __restrict__ err) {
  const int s = r / nt, i = r % nt;
  int slot = seq_ids[s];
  if (slot < 0 || slot >= max_seqs) {
    atomicOr(err, ERR_SEQ);
    slot = 0;
  }
  int pos = n_past[slot] + i;
  if (pos < 0 || pos >= max_ctx) {
    atomicOr(err, ERR_POS);
    pos = max_ctx;
  }
  return RowInfo{slot, pos};
}

// Two sequences of one round naming the same slot would race on its KV rows
// and commit twice ("Model-neutral Speculative Decoding", "Capabilities fail
// closed"): sequence s compares its slot with those of sequences 0..s-1 and
// flags ERR_SEQ on a repeat, which makes the round commit nothing.
__device__ __forceinline__ bool slot_repeats(const int32_t* __restrict__ seq_ids, int s,
                                             int raw, int t0, int step) {
  for (int j = t0; j < s; j += step)
    if (seq_ids[j] == raw) return true;
  return false;
}

__global__ void row_info_kernel(const int32_t* __restrict__ seq_ids, int n_seq, int nt,
                                const int32_t* __restrict__ n_past, int max_seqs,
                                int max_ctx, RowInfo* __restrict__ rows,
                                uint32_t* __restrict__ err) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n_seq * nt) return;
  rows[r] = row_info(seq_ids, r, nt, n_past, max_seqs, max_ctx, err);
  if (r % nt == 0 && slot_repeats(seq_ids, r / nt, seq_ids[r / nt], 0, 1))
    atomicOr(err, ERR_SEQ);
}

// One CTA (256 threads) per verify row: the row's (slot, position) record,
// token lookup (anchor for row 0, drafts after), id check, fp16 -> fp32 copy
// of the embedding row, and the first RMSNorm of the row.  The arguments
// travel as one struct so that a captured launch can be pointed at a new
// round's draft and sequence-id arrays.
__global__ void embed_kernel(const EmbedArgs a) {
  grid_dep_launch();  // a programmatically launched GEMM may prefetch its weights now
  const int r = blockIdx.x;
  const int s = r / a.nt, i = r % a.nt;
  __shared__ int s_tok, s_raw;
  // the same record as row_info, with the loads in two dependent levels:
  // (slot, draft token), then (position, anchor); the token is published
  // first so that the row copy does not wait for the record
  int slot = 0, raw = 0;
  if (threadIdx.x == 0) {
    raw = a.seq_ids[s];
    s_raw = raw;
    const int dtok = i > 0 ? a.draft[s * (a.nt - 1) + (i - 1)] : 0;
    slot = raw < 0 || raw >= a.max_seqs ? 0 : raw;
    int tok = i == 0 ? a.anchor[slot] : dtok;
    if (tok < 0 || tok >= a.V) {
      atomicOr(a.err, ERR_TOKEN);
      tok = 0;
    }
    s_tok = tok;
    a.tokens[r] = tok;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (slot != raw) atomicOr(a.err, ERR_SEQ);
    int pos = a.n_past[slot] + i;
    if (pos < 0 || pos >= a.max_ctx) {
      atomicOr(a.err, ERR_POS);
      pos = a.max_ctx;
    }
    a.rows[r] = RowInfo{slot, pos};
  }
  // the sequence's first row checks that no earlier sequence names its slot
  if (i == 0 && slot_repeats(a.seq_ids, s, s_raw, threadIdx.x, blockDim.x))
    atomicOr(a.err, ERR_SEQ);
  // the row into h, then the first RMSNorm of it into xn: the sum of squares
  // in rmsnorm_kernel's order (thread-strided float4 partials, warp
  // butterfly, warps in order), so the result is that kernel's, bit for bit;
  // a row of up to NORM_REG_VEC * 1024 values and its gains stay in registers
  const uint2* src = reinterpret_cast<const uint2*>(a.embed + (size_t)s_tok * a.H);
  float4* dst = reinterpret_cast<float4*>(a.h + (size_t)r * a.H);
  const float4* gm = reinterpret_cast<const float4*>(a.gamma);
  const int H4 = a.H / 4;
  const bool in_regs = H4 <= NORM_REG_VEC * 256;
  auto load = [&](int j) {
    const uint2 w = src[j];
    const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  };
  float4 v[NORM_REG_VEC], gg[NORM_REG_VEC];
  float ss = 0.0f;
  if (in_regs) {
#pragma unroll
    for (int u = 0; u < NORM_REG_VEC; u++) {
      const int j = threadIdx.x + 256 * u;
      if (j < H4) {
        v[u] = load(j);
        gg[u] = gm[j];
      }
    }
#pragma unroll
    for (int u = 0; u < NORM_REG_VEC; u++)
      if (threadIdx.x + 256 * u < H4) {
        dst[threadIdx.x + 256 * u] = v[u];
        ss = fmaf(v[u].x, v[u].x, ss);
        ss = fmaf(v[u].y, v[u].y, ss);
        ss = fmaf(v[u].z, v[u].z, ss);
        ss = fmaf(v[u].w, v[u].w, ss);
      }
  } else {
    for (int j = threadIdx.x; j < H4; j += 256) {
      const float4 b = load(j);
      dst[j] = b;
      ss = fmaf(b.x, b.x, ss);
      ss = fmaf(b.y, b.y, ss);
      ss = fmaf(b.z, b.z, ss);
      ss = fmaf(b.w, b.w, ss);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  __shared__ float s_part[8];
  __shared__ float s_inv;
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.0f;
    for (int w = 0; w < 8; w++) tot += s_part[w];
    s_inv = 1.0f / sqrtf(tot / (float)a.H + a.eps);
  }
  __syncthreads();
  const float inv = s_inv;
  __half2* o = reinterpret_cast<__half2*>(a.xn + (size_t)r * a.H);
  if (in_regs) {
#pragma unroll
    for (int u = 0; u < NORM_REG_VEC; u++) {
      const int j = threadIdx.x + 256 * u;
      if (j < H4) {
        o[2 * j] = __floats2half2_rn(v[u].x * inv * gg[u].x, v[u].y * inv * gg[u].y);
        o[2 * j + 1] = __floats2half2_rn(v[u].z * inv * gg[u].z, v[u].w * inv * gg[u].w);
      }
    }
  } else {
    for (int j = threadIdx.x; j < H4; j += 256) {
      const float4 b = load(j), c = gm[j];
      o[2 * j] = __floats2half2_rn(b.x * inv * c.x, b.y * inv * c.y);
      o[2 * j + 1] = __floats2half2_rn(b.z * inv * c.z, b.w * inv * c.w);
    }
  }
}

// One CTA (256 threads) per row.  The sum of squares is reduced in a fixed
// order (thread-strided partials, warp butterfly, then warps in order), so a
// row's result does not depend on the other rows in the batch.  A row of up
// to NORM_REG_VEC * 1024 values stays in registers between the two passes,
// its gains loaded before the reduction (one round trip to memory).
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ h,
                                                      const float* __restrict__ gamma,
                                                      int H, float eps,
                                                      __half* __restrict__ out) {
  grid_dep_launch();  // a programmatically launched GEMM may prefetch its weights now
  const int r = blockIdx.x;
  const int H4 = H / 4;
  const float4* x = reinterpret_cast<const float4*>(h + (size_t)r * H);
  const float4* gm = reinterpret_cast<const float4*>(gamma);
  const bool in_regs = H4 <= NORM_REG_VEC * 256;
  float4 v[NORM_REG_VEC], gg[NORM_REG_VEC];
  float ss = 0.0f;
  if (in_regs) {
#pragma unroll
    for (int u = 0; u < NORM_REG_VEC; u++) {
      const int j = threadIdx.x + 256 * u;
      v[u] = j < H4 ? x[j] : make_float4(0.f, 0.f, 0.f, 0.f);
      gg[u] = j < H4 ? gm[j] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < NORM_REG_VEC; u++)
      if (threadIdx.x + 256 * u < H4) {
        ss = fmaf(v[u].x, v[u].x, ss);
        ss = fmaf(v[u].y, v[u].y, ss);
        ss = fmaf(v[u].z, v[u].z, ss);
        ss = fmaf(v[u].w, v[u].w, ss);
      }
  } else {
    for (int j = threadIdx.x; j < H4; j += 256) {
      const float4 a = x[j];
      ss = fmaf(a.x, a.x, ss);
      ss = fmaf(a.y, a.y, ss);
      ss = fmaf(a.z, a.z, ss);
      ss = fmaf(a.w, a.w, ss);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  __shared__ float s_part[8];
  __shared__ float s_inv;
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.0f;
    for (int w = 0; w < 8; w++) tot += s_part[w];
    s_inv = 1.0f / sqrtf(tot / (float)H + eps);
  }
  __syncthreads();
  const float inv = s_inv;
  __half2* o = reinterpret_cast<__half2*>(out + (size_t)r * H);
  if (in_regs) {
#pragma unroll
    for (int u = 0; u < NORM_REG_VEC; u++) {
      const int j = threadIdx.x + 256 * u;
      if (j < H4) {
        o[2 * j] = __floats2half2_rn(v[u].x * inv * gg[u].x, v[u].y * inv * gg[u].y);
        o[2 * j + 1] = __floats2half2_rn(v[u].z * inv * gg[u].z, v[u].w * inv * gg[u].w);
      }
    }
  } else {
    for (int j = threadIdx.x; j < H4; j += 256) {
      const float4 a = x[j], b = gm[j];
      o[2 * j] = __floats2half2_rn(a.x * inv * b.x, a.y * inv * b.y);
      o[2 * j + 1] = __floats2half2_rn(a.z * inv * b.z, a.w * inv * b.w);
    }
  }
}

// cos/sin of pos * theta^(-2i/hd), evaluated in fp64 and rounded to fp32.
__global__ void rope_table_kernel(float2* tab, int max_ctx, int hd, double theta) {
  const int half = hd / 2;
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (size_t)max_ctx * half) return;
  const int pos = (int)(idx / half), i = (int)(idx % half);
  const double f = pow(theta, -2.0 * (double)i / (double)hd);
  double s, c;
  sincos((double)pos * f, &s, &c);
  tab[idx] = make_float2((float)c, (float)s);
}

__global__ void kv_write_kernel(const __half* __restrict__ k_new,
                                const __half* __restrict__ v_new,
                                const RowInfo* __restrict__ rows, int nkv, int hd,
                                int max_ctx, __half* __restrict__ kc,
                                __half* __restrict__ vc) {
  const int r = blockIdx.x;
  const RowInfo ri = rows[r];
  if (ri.pos >= max_ctx) return;
  for (int j = threadIdx.x; j < nkv * hd; j += blockDim.x) {
    const int kvh = j / hd, d = j % hd;
    const size_t dst = (((size_t)ri.slot * nkv + kvh) * max_ctx + ri.pos) * hd + d;
    kc[dst] = k_new[(size_t)r * nkv * hd + j];
    vc[dst] = v_new[(size_t)r * nkv * hd + j];
  }
}

}  // namespace

void launch_row_info(const int32_t* seq_ids, int n_seq, int nt, const int32_t* n_past,
                     int max_seqs, int max_ctx, RowInfo* rows, uint32_t* err,
                     cudaStream_t st) {
  const int R = n_seq * nt;
  row_info_kernel<<<(R + 127) / 128, 128, 0, st>>>(seq_ids, n_seq, nt, n_past, max_seqs,
                                                   max_ctx, rows, err);
}

void launch_embed_rows(const __half* embed, int V, int H, const int32_t* anchor,
                       const int32_t* draft, const int32_t* seq_ids, int n_seq, int nt,
                       const int32_t* n_past, int max_seqs, int max_ctx, RowInfo* rows,
                       int32_t* tokens, float* h, const float* gamma, float eps, __half* xn,
                       uint32_t* err, cudaStream_t st) {
  EmbedArgs a;
  a.embed = embed;
  a.anchor = anchor;
  a.draft = draft;
  a.seq_ids = seq_ids;
  a.n_past = n_past;
  a.rows = rows;
  a.tokens = tokens;
  a.h = h;
  a.err = err;
  a.gamma = gamma;
  a.xn = xn;
  a.eps = eps;
  a.V = V;
  a.H = H;
  a.nt = nt;
  a.max_seqs = max_seqs;
  a.max_ctx = max_ctx;
  embed_kernel<<<n_seq * nt, 256, 0, st>>>(a);
}

cudaError_t embed_node_retarget(cudaGraphExec_t ex, cudaGraphNode_t node, const int32_t* draft,
                                const int32_t* seq_ids) {
  cudaKernelNodeParams p;
  cudaError_t e = cudaGraphKernelNodeGetParams(node, &p);
  if (e != cudaSuccess) return e;
  if (p.func != reinterpret_cast<void*>(embed_kernel) || p.kernelParams == nullptr)
    return cudaErrorInvalidValue;
  EmbedArgs a = *static_cast<const EmbedArgs*>(p.kernelParams[0]);
  a.draft = draft;
  a.seq_ids = seq_ids;
  void* args[] = {&a};
  p.kernelParams = args;
  p.extra = nullptr;
  return cudaGraphExecKernelNodeSetParams(ex, node, &p);
}

void launch_rmsnorm(const float* h, const float* gamma, int R, int H, float eps,
                    __half* out, cudaStream_t st) {
  rmsnorm_kernel<<<R, 256, 0, st>>>(h, gamma, H, eps, out);
}

void launch_rope_table(float2* tab, int max_ctx, int hd, float theta, cudaStream_t st) {
  const size_t n = (size_t)max_ctx * (hd / 2);
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(tab, max_ctx, hd,
                                                                 (double)theta);
}

void launch_kv_write(const __half* k_new, const __half* v_new, const RowInfo* rows, int R,
                     int nkv, int hd, int max_ctx, __half* kcache, __half* vcache,
                     cudaStream_t st) {
  kv_write_kernel<<<R, 256, 0, st>>>(k_new, v_new, rows, nkv, hd, max_ctx, kcache, vcache);
}
