// attn.cu -- causal GQA verify attention over the KV cache, bitwise
// position-invariant ("Speculative Decoding (D5-R) -- Plan", status notes:
// the batched verify attention was made bitwise position-invariant so that
// speculative output is byte-identical to sequential decoding).
//
// A query row at absolute position P attends to positions 0..P.  The cache is
// cut into chunks of ATTN_CHUNK positions at absolute multiples; each chunk
// gives a partial (row max m, row sum l, unnormalised o) computed by an
// instruction sequence that depends only on the row's own q and P, and the
// partials of chunks 0..P/ATTN_CHUNK are merged in increasing chunk order.
// Neither step depends on nt or on the other rows of the batch, so row i of
// an nt-row round equals the nt = 1 result at the same position bit for bit.
//
// One CTA per (chunk, kv head, sequence) -- or, with five or more m tiles
// of query rows, per group of two m tiles of them: the chunk's K and V tiles
// are staged in shared memory (cp.async, XOR-swizzled 16-byte units) and
// shared by the CTA's query rows of that kv head (GQA, nt x group rows),
// which are processed as m16 tiles with mma.sync m16n8k16: S = Q K^T, softmax in fp32
// (log2 domain), O = P V with P as an exact hi + lo pair of fp16 operands.
// Each half of the chunk's keys is a separate warp's (max, sum, O); the two
// are rescaled to the common max in one fixed order inside the CTA, so the
// chunk partial is still one (m, l, o) per row.
#include <math.h>

#include "common.cuh"

namespace {

constexpr int CH = ATTN_CHUNK;
constexpr int KS = 2;  // key halves of a chunk (one warp each)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// byte offset of 16-byte unit u of cache row p inside a swizzled tile
template <int HD>
__device__ __forceinline__ uint32_t tile_off(int p, int u) {
  return (uint32_t)(p * (HD * 2) + ((u ^ (p & 7)) << 4));
}

// Shared memory of the chunk kernel: the K tile, the q rows of its m tiles,
// the V tile, then -- unless they fit over K and q, which no warp reads any
// more once every work item is in one round -- the key-half exchange slots
// of the NW / 2 warp pairs (O fragments and (m, l)).
struct ChunkSmem {
  size_t q_off, v_off, slot_off, bytes;
};
inline ChunkSmem chunk_smem(int hd, int ds, int nw, int n_mt) {
  ChunkSmem c;
  const size_t kbytes = (size_t)CH * hd * 2, qbytes = (size_t)n_mt * 16 * hd * 2;
  const size_t slots = (size_t)(nw / 2) * (hd / 8 / ds + 1) * 32 * 16;
  const bool one_round = n_mt * ds * KS <= nw;
  c.q_off = kbytes;
  c.v_off = kbytes + qbytes;
  const bool alias = one_round && slots <= kbytes + qbytes;
  c.slot_off = alias ? 0 : c.v_off + kbytes;
  c.bytes = c.v_off + kbytes + (alias ? 0 : slots);
  return c;
}

// Residency MINB CTAs per SM.  Two, as the shared memory holds (with 8 warps
// that caps the registers at 128, which the q fragments read from shared
// memory allow).  Three for the 4-warp CTA of whole head dimensions (up to
// two m tiles, 72 KB of shared memory at head_dim 128) when one chunk's
// CTAs alone fill the SMs: held to 168 registers, 12 warps an SM (batched
// round, 12 sequences: 41.5 -> 37.5 us per layer; one sequence over a long
// context, the 8-layer decoder at nt 8, is faster at two).  The register
// cap changes no arithmetic: the bits are those of the two-CTA build.
template <int HD, int DS, int NW, int MINB>
__global__ void __launch_bounds__(NW * 32, MINB)
attn_chunk_kernel(const __half* __restrict__ q, const __half* __restrict__ kcache,
                  const __half* __restrict__ vcache, const RowInfo* __restrict__ rows,
                  int nt, int nq, int nkv, int max_ctx, int nchunks, int mt_group,
                  ChunkSmem lay, float* __restrict__ part) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* Ks = smem;
  unsigned char* Qs = smem + lay.q_off;
  unsigned char* Vs = smem + lay.v_off;
  const int c = blockIdx.x, s = blockIdx.z;
  const int G = nq / nkv, M = nt * G, Mmax_stride = M;  // rows of this (seq, kv head)
  // the (seq, kv head)'s m tiles are cut into groups of mt_group, one CTA
  // each: this CTA's tiles are mt0 .. mt0 + n_mt - 1
  const int n_mt_all = (M + 15) / 16, n_grp = (n_mt_all + mt_group - 1) / mt_group;
  const int kvh = blockIdx.y / n_grp, mt0 = (blockIdx.y % n_grp) * mt_group;
  const int n_mt = min(mt_group, n_mt_all - mt0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  // the row table and the committed cache belong to kernels that completed
  // before the one this grid depends on; the new rows' K/V, q and the
  // partials are that kernel's (or later) business
  const RowInfo last = rows[s * nt + nt - 1];
  const int pos_last = last.pos < max_ctx ? last.pos : max_ctx - 1;
  if (c * CH > pos_last) {
    grid_dep_launch();
    return;  // no row of this sequence reaches this chunk
  }
  const int slot = last.slot;
  const int new0 = min(rows[s * nt].pos, max_ctx);  // positions >= new0 are this round's

  // ---- stage K and V of positions [c*CH, c*CH + CH): the committed part
  // ---- before the grid dependency resolves, the round's new rows after it;
  // ---- K and V in separate copy groups so that S = Q K^T can start first
  constexpr int UNITS = HD / 8;              // 16-byte units per row
  constexpr int RP = NW * 32 / UNITS;         // rows per pass of the CTA
  const int u = threadIdx.x % UNITS, p0 = threadIdx.x / UNITS;
  const size_t head_base = ((size_t)slot * nkv + kvh) * max_ctx;
  // a thread copies unit u of the rows p0, p0 + RP, ... below CH: its
  // swizzled column (u ^ (p & 7)) is the same for all of them (RP is a
  // multiple of 8; it need not divide CH)
  static_assert(RP % 8 == 0, "rows per pass must keep the swizzle column");
  auto stage = [&](unsigned char* tile, const __half* cache, bool committed) {
    const uint32_t s0 = smem_u32(tile) + tile_off<HD>(p0, u);
    const __half* g0 = cache + (head_base + (size_t)c * CH + p0) * HD + u * 8;
#pragma unroll 4
    for (int i = 0; i < (CH + RP - 1) / RP; i++) {
      if (p0 + RP * i >= CH) break;
      const int pg = c * CH + p0 + RP * i;
      if ((pg < new0) != committed) continue;
      const uint32_t so = s0 + (uint32_t)(i * RP * HD * 2);
      if (pg < max_ctx) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(so),
                     "l"(g0 + (size_t)i * RP * HD));
      } else {
        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(so), "r"(0));
      }
    }
    asm volatile("cp.async.commit_group;");
  };
  stage(Ks, kcache, true);
  stage(Vs, vcache, true);
  grid_dep_wait();
  stage(Ks, kcache, false);
  // the q rows of the CTA's m tiles (row m = query i * G + gh), swizzled like
  // the cache tiles; rows past M are zero
  {
    const uint32_t qs0 = smem_u32(Qs);
    for (int e = threadIdx.x; e < n_mt * 16 * UNITS; e += NW * 32) {
      const int ml = e / UNITS, uu = e % UNITS, m = mt0 * 16 + ml;
      const uint32_t so = qs0 + tile_off<HD>(ml, uu);
      if (m < M) {
        const __half* src = q + ((size_t)(s * nt + m / G) * nq + kvh * G + m % G) * HD + uu * 8;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(so), "l"(src));
      } else {
        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(so), "r"(0));
      }
    }
    asm volatile("cp.async.commit_group;");
  }
  stage(Vs, vcache, false);
  grid_dep_launch();

  const float sc_log2 = 1.4426950408889634f / sqrtf((float)HD);
  const uint32_t ks_base = smem_u32(Ks), vs_base = smem_u32(Vs), qs_base = smem_u32(Qs);
  // work items: (m tile, slice of the head dimensions, half of the chunk's
  // keys).  The two key halves of an (m tile, slice) are consecutive warps:
  // each computes S, its own row max and P over its 64 keys (the same
  // instruction sequence whatever nt is), and O for HD / DS dimensions; the
  // half-1 warp hands (m, l, O) to the half-0 warp through shared memory,
  // which rescales both to the common max in a fixed order.
  constexpr int CHK = CH / KS;
  constexpr int DN = HD / 8 / DS;  // n8 blocks of head dimensions of a warp
  float4* x_o = reinterpret_cast<float4*>(smem + lay.slot_off);  // [NW/2][DN][32]
  float4* x_ml = x_o + (NW / 2) * DN * 32;                        // [NW/2][32]
  const int n_items = n_mt * DS * KS;
  for (int it0 = 0; it0 < n_items; it0 += NW) {  // uniform trip count: the barriers below
    const int it = it0 + warp;
    const int kh = it % KS, dh = (it / KS) % DS, mtl = it / (KS * DS), mt = mt0 + mtl;
    const int key0 = kh * CHK;
    const int mA = mt * 16 + g, mB = mA + 8;
    const bool okA = it < n_items && mA < M, okB = it < n_items && mB < M;
    int posA = -1, posB = -1;
    if (okA) {
      const RowInfo ri = rows[s * nt + mA / G];
      posA = ri.pos < max_ctx ? ri.pos : max_ctx - 1;
    }
    if (okB) {
      const RowInfo ri = rows[s * nt + mB / G];
      posB = ri.pos < max_ctx ? ri.pos : max_ctx - 1;
    }
    if (it0 == 0) {
      asm volatile("cp.async.wait_group 1;" ::: "memory");  // K and q (V's last group may fly)
      __syncthreads();
    }
    // the q fragment rows of this m tile for ldmatrix: lanes 0-7 rows 0-7,
    // 8-15 rows 8-15 (first 8 dims of a k16 step), 16-31 the same rows for
    // its second 8 dims
    const int q_row = min(mtl, n_mt - 1) * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
    // ---- S = Q K^T over the half (16 rows x CHK keys)
    float sacc[CHK / 8][4];
#pragma unroll
    for (int nb = 0; nb < CHK / 8; nb++)
#pragma unroll
      for (int e = 0; e < 4; e++) sacc[nb][e] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; kk += 2) {
      uint32_t qa0[4], qa1[4];
      ldsm_x4(qs_base + tile_off<HD>(q_row, 2 * kk + (lane >> 4)), qa0[0], qa0[1], qa0[2], qa0[3]);
      ldsm_x4(qs_base + tile_off<HD>(q_row, 2 * kk + 2 + (lane >> 4)), qa1[0], qa1[1], qa1[2],
              qa1[3]);
#pragma unroll
      for (int nb = 0; nb < CHK / 8; nb++) {
        const int key = key0 + 8 * nb + (lane & 7);
        const int unit = 2 * kk + (lane >> 3);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(ks_base + tile_off<HD>(key, unit), b0, b1, b2, b3);
        mma_16816(sacc[nb], qa0, b0, b1);
        mma_16816(sacc[nb], qa1, b2, b3);
      }
    }
    // ---- mask, row max over the half (fixed butterfly over the 4 lanes of a row)
    float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < CHK / 8; nb++)
#pragma unroll
      for (int e = 0; e < 2; e++) {
        const int kg = c * CH + key0 + 8 * nb + 2 * t + e;
        float va = sacc[nb][e] * sc_log2, vb = sacc[nb][2 + e] * sc_log2;
        va = kg <= posA ? va : -INFINITY;
        vb = kg <= posB ? vb : -INFINITY;
        sacc[nb][e] = va;
        sacc[nb][2 + e] = vb;
        mxA = fmaxf(mxA, va);
        mxB = fmaxf(mxB, vb);
      }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, off));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, off));
    }
    const float uA = mxA == -INFINITY ? 0.0f : mxA;
    const float uB = mxB == -INFINITY ? 0.0f : mxB;
    // ---- p = exp2(s - m) in fp32; l = sum of p in a fixed order
    float lA = 0.0f, lB = 0.0f;
#pragma unroll
    for (int nb = 0; nb < CHK / 8; nb++) {
      sacc[nb][0] = exp2f(sacc[nb][0] - uA);
      sacc[nb][1] = exp2f(sacc[nb][1] - uA);
      sacc[nb][2] = exp2f(sacc[nb][2] - uB);
      sacc[nb][3] = exp2f(sacc[nb][3] - uB);
      lA += sacc[nb][0];
      lA += sacc[nb][1];
      lB += sacc[nb][2];
      lB += sacc[nb][3];
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      lA += __shfl_xor_sync(0xffffffffu, lA, off);
      lB += __shfl_xor_sync(0xffffffffu, lB, off);
    }
    // ---- O = P V over the half (16 rows x HD / DS dims).  P enters the fp16
    // ---- MMA as an exact two-term split p = hi + lo (hi = fp16(p), lo =
    // ---- fp16(p - hi)), so the product carries ~22 bits of p instead of 11.
    if (it0 == 0) {
      asm volatile("cp.async.wait_group 0;" ::: "memory");  // V
      __syncthreads();
    }
    const int dn0 = dh * DN;
    float oacc[DN][4];
#pragma unroll
    for (int dn = 0; dn < DN; dn++)
#pragma unroll
      for (int e = 0; e < 4; e++) oacc[dn][e] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < CHK / 16; kk++) {
      uint32_t phi[4], plo[4];
#pragma unroll
      for (int h = 0; h < 2; h++) {         // key tiles 2kk (h = 0) and 2kk+1 (h = 1)
#pragma unroll
        for (int rw = 0; rw < 2; rw++) {    // rows g (rw = 0) and g+8 (rw = 1)
          const float p0 = sacc[2 * kk + h][2 * rw], p1 = sacc[2 * kk + h][2 * rw + 1];
          const __half2 hi = __floats2half2_rn(p0, p1);
          const float2 hf = __half22float2(hi);
          const __half2 lo = __floats2half2_rn(p0 - hf.x, p1 - hf.y);
          phi[2 * h + rw] = *reinterpret_cast<const uint32_t*>(&hi);
          plo[2 * h + rw] = *reinterpret_cast<const uint32_t*>(&lo);
        }
      }
#pragma unroll
      for (int dn = 0; dn < DN; dn += 2) {
        const int mi = lane >> 3;
        const int key = key0 + 16 * kk + (lane & 7) + (mi & 1) * 8;
        const int unit = dn0 + dn + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vs_base + tile_off<HD>(key, unit), b0, b1, b2, b3);
        mma_16816(oacc[dn], phi, b0, b1);
        mma_16816(oacc[dn], plo, b0, b1);
        mma_16816(oacc[dn + 1], phi, b2, b3);
        mma_16816(oacc[dn + 1], plo, b2, b3);
      }
    }
    // ---- the two halves: half 1 hands over, half 0 combines
    const int pr = warp >> 1;  // the pair's exchange slot
    if (kh == 1 && it < n_items) {
#pragma unroll
      for (int dn = 0; dn < DN; dn++)
        x_o[(pr * DN + dn) * 32 + lane] = make_float4(oacc[dn][0], oacc[dn][1], oacc[dn][2], oacc[dn][3]);
      x_ml[pr * 32 + lane] = make_float4(mxA, mxB, lA, lB);
    }
    __syncthreads();
    if (kh == 0 && it < n_items) {
      const float4 ml = x_ml[pr * 32 + lane];
      const float mA2 = fmaxf(mxA, ml.x), mB2 = fmaxf(mxB, ml.y);
      const float vA = mA2 == -INFINITY ? 0.0f : mA2, vB = mB2 == -INFINITY ? 0.0f : mB2;
      const float wA0 = exp2f(mxA - vA), wA1 = exp2f(ml.x - vA);
      const float wB0 = exp2f(mxB - vB), wB1 = exp2f(ml.y - vB);
      const float lA2 = fmaf(ml.z, wA1, lA * wA0), lB2 = fmaf(ml.w, wB1, lB * wB0);
#pragma unroll
      for (int dn = 0; dn < DN; dn++) {
        const float4 o1 = x_o[(pr * DN + dn) * 32 + lane];
        oacc[dn][0] = fmaf(o1.x, wA1, oacc[dn][0] * wA0);
        oacc[dn][1] = fmaf(o1.y, wA1, oacc[dn][1] * wA0);
        oacc[dn][2] = fmaf(o1.z, wB1, oacc[dn][2] * wB0);
        oacc[dn][3] = fmaf(o1.w, wB1, oacc[dn][3] * wB0);
      }
      // ---- partials: part[s][kvh][c][m] = (o[HD], m, l)
      const size_t base = (((size_t)s * nkv + kvh) * nchunks + c) * (size_t)Mmax_stride;
      if (okA) {
        float* dst = part + (base + mA) * (HD + 2) + 8 * dn0;
#pragma unroll
        for (int dn = 0; dn < DN; dn++)
          *reinterpret_cast<float2*>(dst + 8 * dn + 2 * t) = make_float2(oacc[dn][0], oacc[dn][1]);
        if (t == 0 && dh == 0)
          *reinterpret_cast<float2*>(part + (base + mA) * (HD + 2) + HD) = make_float2(mA2, lA2);
      }
      if (okB) {
        float* dst = part + (base + mB) * (HD + 2) + 8 * dn0;
#pragma unroll
        for (int dn = 0; dn < DN; dn++)
          *reinterpret_cast<float2*>(dst + 8 * dn + 2 * t) = make_float2(oacc[dn][2], oacc[dn][3]);
        if (t == 0 && dh == 0)
          *reinterpret_cast<float2*>(part + (base + mB) * (HD + 2) + HD) = make_float2(mB2, lB2);
      }
    }
    __syncthreads();  // the exchange slots are reused by the next items
  }
}

// One warp per (row, q head), two per CTA: merge chunks 0..P/CH in
// increasing order.  The chunks' (m, l) are loaded 32 at a time (one per
// lane) and the global max (exact in any order) is a warp reduction; the
// weights w_c = exp2(m_c - max) are broadcast by shuffle, and each lane sums
// w_c * o_c[d] for its HD / 32 head dimensions and w_c * l_c over the
// chunks in order, MB chunks' o loads in flight at a time (the first batch
// issued together with the (m, l) loads).  MB is the smallest of 4, 8, 16
// that holds the model's chunk count: its registers set the residency
// (batched round: MB 8 instead of 16 took the merge 11.4 -> 9.7 us).  The
// arithmetic of a row depends neither on MB nor on the other rows.
constexpr int MERGE_WARPS = 2;
constexpr int MERGE_MAX = 16;  // chunks of the warp merge; the CTA merge beyond
template <int HD, int MB>
__global__ void __launch_bounds__(MERGE_WARPS * 32)
attn_merge_kernel(const float* __restrict__ part, const RowInfo* __restrict__ rows,
                  int R, int nt, int nq, int nkv, int max_ctx, int nchunks,
                  __half* __restrict__ out) {
  grid_dep_launch();  // a programmatically launched GEMM may prefetch its weights now
  constexpr int DPL = HD / 32;  // head dimensions of a lane (4 or 2)
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * MERGE_WARPS + (threadIdx.x >> 5);
  if (item >= R * nq) return;  // whole warps
  const int r = item / nq, h = item % nq;
  const int s = r / nt, i = r % nt;
  const int G = nq / nkv, kvh = h / G, gh = h % G;
  const int M = nt * G, m = i * G + gh;
  const RowInfo ri = rows[r];
  const int pos = ri.pos < max_ctx ? ri.pos : max_ctx - 1;
  const int nc = pos / CH + 1;
  const size_t stride = (size_t)M * (HD + 2);  // floats between consecutive chunks
  const float* p0 = part + ((((size_t)s * nkv + kvh) * nchunks) * M + m) * (HD + 2);
  // a partial row is HD + 2 floats: only 8-byte alignment holds, so a
  // lane's dimensions come as float2 pairs
  auto load_o = [&](int c, float (&o)[DPL]) {
    const float* src = p0 + (size_t)c * stride + lane * DPL;
#pragma unroll
    for (int k = 0; k < DPL; k += 2) {
      const float2 t = __ldcg(reinterpret_cast<const float2*>(src + k));
      o[k] = t.x;
      o[k + 1] = t.y;
    }
  };
  grid_dep_wait();  // the partials come from the chunk kernel
  float ov[MB][DPL];
#pragma unroll
  for (int u = 0; u < MB; u++)
    if (u < nc) load_o(u, ov[u]);
  float2 ml0 = make_float2(-INFINITY, 0.0f);
  if (lane < nc) ml0 = __ldcg(reinterpret_cast<const float2*>(p0 + (size_t)lane * stride + HD));
  float mx = ml0.x;
  for (int c = lane + 32; c < nc; c += 32) mx = fmaxf(mx, __ldcg(p0 + (size_t)c * stride + HD));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float o[DPL], l = 0.0f;
#pragma unroll
  for (int k = 0; k < DPL; k++) o[k] = 0.0f;
  for (int cb = 0; cb < nc; cb += 32) {
    const int c = cb + lane;
    float2 ml = ml0;
    if (cb > 0) {
      ml = make_float2(0.0f, 0.0f);
      if (c < nc) ml = __ldcg(reinterpret_cast<const float2*>(p0 + (size_t)c * stride + HD));
    }
    const float w = c < nc ? exp2f(ml.x - mx) : 0.0f;
    const int nb = min(32, nc - cb);
    for (int u0 = 0; u0 < nb; u0 += MB) {
      if (cb > 0 || u0 > 0) {
#pragma unroll
        for (int u = 0; u < MB; u++)
          if (u0 + u < nb) load_o(cb + u0 + u, ov[u]);
      }
#pragma unroll
      for (int u = 0; u < MB; u++) {
        const float wu = __shfl_sync(0xffffffffu, w, (u0 + u) & 31);
        const float lu = __shfl_sync(0xffffffffu, ml.y, (u0 + u) & 31);
        if (u0 + u < nb) {
          l = fmaf(lu, wu, l);
#pragma unroll
          for (int k = 0; k < DPL; k++) o[k] = fmaf(ov[u][k], wu, o[k]);
        }
      }
    }
  }
  const float inv = 1.0f / l;
  __half* dst = out + (size_t)r * nq * HD + (size_t)h * HD + lane * DPL;
#pragma unroll
  for (int k = 0; k < DPL; k++) dst[k] = __float2half_rn(o[k] * inv);
}

// The merge for long contexts (more than 16 chunks): one CTA per (row, q
// head), one thread per head dimension, the same arithmetic in the same
// order as attn_merge_kernel (results are bitwise the same): merge chunks
// 0..P/CH in increasing order.  The o loads of the first MB chunks go out
// together with every chunk's (m, l), so a context of up to MB chunks costs
// one round trip; the global max (exact in any order) is a block reduction,
// the thread owning chunk c stores w_c = exp2(m_c - max) in shared memory,
// and each thread sums w_c * o_c[d] and w_c * l_c over the chunks in order.
constexpr int MERGE_MB = 40;
template <int HD>
__global__ void __launch_bounds__(HD)
attn_merge_cta_kernel(const float* __restrict__ part, const RowInfo* __restrict__ rows,
                  int R, int nt, int nq, int nkv, int max_ctx, int nchunks,
                  __half* __restrict__ out) {
  grid_dep_launch();  // a programmatically launched GEMM may prefetch its weights now
  extern __shared__ float s_ml[];  // [nchunks] w, then [nchunks] l
  float* s_w = s_ml;
  float* s_l = s_ml + nchunks;
  __shared__ float s_red[HD / 32];
  const int r = blockIdx.x / nq, h = blockIdx.x % nq;
  const int d = threadIdx.x, lane = d & 31, warp = d >> 5;
  const int s = r / nt, i = r % nt;
  const int G = nq / nkv, kvh = h / G, gh = h % G;
  const int M = nt * G, m = i * G + gh;
  const RowInfo ri = rows[r];
  const int pos = ri.pos < max_ctx ? ri.pos : max_ctx - 1;
  const int nc = pos / CH + 1;
  const size_t stride = (size_t)M * (HD + 2);  // floats between consecutive chunks
  const float* p0 = part + ((((size_t)s * nkv + kvh) * nchunks) * M + m) * (HD + 2);
  grid_dep_wait();  // the partials come from the chunk kernel
  float v[MERGE_MB];
#pragma unroll
  for (int u = 0; u < MERGE_MB; u++) v[u] = u < nc ? __ldcg(p0 + (size_t)u * stride + d) : 0.0f;
  float mx = -INFINITY;
  for (int c = d; c < nc; c += HD) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(p0 + (size_t)c * stride + HD));
    s_w[c] = ml.x;  // m for now
    s_l[c] = ml.y;
    mx = fmaxf(mx, ml.x);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) s_red[warp] = mx;
  __syncthreads();
  mx = s_red[0];
#pragma unroll
  for (int w = 1; w < HD / 32; w++) mx = fmaxf(mx, s_red[w]);
  for (int c = d; c < nc; c += HD) s_w[c] = exp2f(s_w[c] - mx);
  __syncthreads();
  float o = 0.0f, l = 0.0f;
#pragma unroll
  for (int u = 0; u < MERGE_MB; u++)
    if (u < nc) {
      const float w = s_w[u];
      l = fmaf(s_l[u], w, l);
      o = fmaf(v[u], w, o);
    }
  for (int c = MERGE_MB; c < nc; c += 16) {  // long contexts: sixteen loads in flight
    float v2[16];
#pragma unroll
    for (int u = 0; u < 16; u++) v2[u] = c + u < nc ? __ldcg(p0 + (size_t)(c + u) * stride + d) : 0.0f;
#pragma unroll
    for (int u = 0; u < 16; u++)
      if (c + u < nc) {
        const float w = s_w[c + u];
        l = fmaf(s_l[c + u], w, l);
        o = fmaf(v2[u], w, o);
      }
  }
  out[(size_t)r * nq * HD + (size_t)h * HD + d] = __float2half_rn(o * (1.0f / l));
}


template <int HD>
int attn_launch_t(const __half* q, const __half* kcache, const __half* vcache,
                  const RowInfo* rows, int n_seq, int nt, int nq, int nkv, int max_ctx,
                  float* part, __half* out, cudaStream_t st) {
  const int nchunks = (max_ctx + CH - 1) / CH;
  const int R = n_seq * nt;
  // both launched as programmatic dependents of the previous kernel: the
  // chunk kernel stages the committed cache and the merge kernel starts up
  // while their predecessors finish
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = programmatic_launch() ? 1 : 0;
  // one m tile: warp pairs also split the head dimensions (4 warps); two m
  // tiles: 4 warps; three or four: 8 warps, so that they are one round of
  // work items; five or more: CTAs of two m tiles (4 warps, two CTAs per SM)
  // (the bits of every output depend on none of these choices)
  const int n_mt = (nt * (nq / nkv) + 15) / 16;
  const int mt_group = n_mt <= 4 ? n_mt : 2;
  const int n_grp = (n_mt + mt_group - 1) / mt_group;
  const int ds = n_mt == 1 ? 2 : 1;
  const int nw = mt_group <= 2 ? 4 : 8;
  static const int sms = [] {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
  }();
  const bool dense = (long long)n_seq * nkv * n_grp >= sms;
  auto chunk = n_mt == 1 ? attn_chunk_kernel<HD, 2, 4, 2>
               : nw == 4 ? (dense ? attn_chunk_kernel<HD, 1, 4, 3> : attn_chunk_kernel<HD, 1, 4, 2>)
                         : attn_chunk_kernel<HD, 1, 8, 2>;
  const ChunkSmem lay = chunk_smem(HD, ds, nw, mt_group);
  cfg.gridDim = dim3(nchunks, nkv * n_grp, n_seq);
  cfg.blockDim = dim3(nw * 32);
  cfg.dynamicSmemBytes = lay.bytes;
  cudaError_t e = cudaLaunchKernelEx(&cfg, chunk, q, kcache, vcache, rows, nt, nq, nkv, max_ctx,
                                     nchunks, mt_group, lay, part);
  if (e == cudaSuccess) {
    // the model's chunk count picks the merge (never nt): a warp per (row,
    // head) for short contexts, a CTA per (row, head) -- every chunk's loads
    // in flight at once -- for long ones; both compute the same bits
    if (nchunks <= MERGE_MAX) {
      cfg.gridDim = dim3((R * nq + MERGE_WARPS - 1) / MERGE_WARPS);
      cfg.blockDim = dim3(MERGE_WARPS * 32);
      cfg.dynamicSmemBytes = 0;
      auto merge = nchunks <= 4   ? attn_merge_kernel<HD, 4>
                   : nchunks <= 8 ? attn_merge_kernel<HD, 8>
                                  : attn_merge_kernel<HD, 16>;
      e = cudaLaunchKernelEx(&cfg, merge, (const float*)part, rows, R, nt, nq, nkv, max_ctx,
                             nchunks, out);
    } else {
      cfg.gridDim = dim3(R * nq);
      cfg.blockDim = dim3(HD);
      cfg.dynamicSmemBytes = 2 * sizeof(float) * (size_t)nchunks;
      e = cudaLaunchKernelEx(&cfg, attn_merge_cta_kernel<HD>, (const float*)part, rows, R, nt, nq,
                             nkv, max_ctx, nchunks, out);
    }
  }
  if (e != cudaSuccess) return fail(SPEC_E_CUDA, std::string("attention launch: ") + cudaGetErrorString(e));
  return SPEC_OK;
}

}  // namespace

size_t attn_part_floats(int max_seqs, int nkv, int max_ctx, int max_nt, int group, int hd) {
  const int nchunks = (max_ctx + CH - 1) / CH;
  return (size_t)max_seqs * nkv * nchunks * (size_t)max_nt * group * (hd + 2);
}

int attn_launch(const __half* q, const __half* kcache, const __half* vcache,
                const RowInfo* rows, int n_seq, int nt, int nq, int nkv, int hd, int max_ctx,
                float* part, __half* out, cudaStream_t st) {
  if (hd == 128)
    return attn_launch_t<128>(q, kcache, vcache, rows, n_seq, nt, nq, nkv, max_ctx, part, out, st);
  if (hd == 64)
    return attn_launch_t<64>(q, kcache, vcache, rows, n_seq, nt, nq, nkv, max_ctx, part, out, st);
  return fail(SPEC_E_UNSUPPORTED, "verify attention supports head_dim 64 or 128");
}

void attn_init_attrs() {
  int dev = 0, optin = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  for (auto k : {attn_chunk_kernel<128, 2, 4, 2>, attn_chunk_kernel<128, 1, 4, 2>,
                 attn_chunk_kernel<128, 1, 4, 3>, attn_chunk_kernel<128, 1, 8, 2>,
                 attn_chunk_kernel<64, 2, 4, 2>, attn_chunk_kernel<64, 1, 4, 2>,
                 attn_chunk_kernel<64, 1, 4, 3>, attn_chunk_kernel<64, 1, 8, 2>})
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
}
