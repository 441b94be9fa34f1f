// linear.cu -- weights-once multi-row dequant GEMM of the verify pass.
//
// "Speculative Decoding (D5-R) -- Plan", section 1: the batched verify is a
// weights-once round, not a per-row restream; its cost is the weights once
// plus nt times the per-token work.  Here every packed weight byte is read
// from HBM exactly once per call, whatever nt is, and is applied to all
// nt rows in registers:
//
//   * 16 output rows x 64 k per warp step; the 4-bit / 6-bit integers are
//     turned into exact fp16 values with the 0x6400 magic-number trick and
//     fed as the A operand of mma.sync m16n8k16 (f16 x f16 -> f32); the
//     activations (n8 column tiles of verify rows) are the B operand;
//   * each 32-block is accumulated in a fresh fp32 fragment and folded into
//     the running sum with one fp32 FMA by its fp16 scale;
//   * K is split into S segments fixed per matrix (never per nt); the last
//     CTA of a tile group sums the S partials in segment order;
//   * epilogues: store, residual add, SwiGLU, RoPE + KV-cache write, and the
//     LM head's fused per-row argmax.
// Every output element is produced by the same instruction sequence for any
// nt (zero-padded columns never feed real ones), so verify rows are bitwise
// equal across nt ("Speculative Decoding (D5-R) -- Plan", status notes:
// batched verify made bitwise position-invariant).
#include <algorithm>
#include <cmath>
#include <cstdio>

#include "common.cuh"

namespace {

constexpr int WARPS = 4;  // warps per CTA
constexpr int TPW = 2;    // tiles (of 16 rows) per warp
// Weight-stream ring per warp: NS stages of one 64-k chunk of TPW tiles,
// filled with cp.async (16-byte copies that bypass L1) and consumed from
// shared memory; NS - 1 chunks are in flight while one is computed.
template <int QT>
struct Ring {
  static constexpr int NS = QT == 4 ? 8 : 6;
  static constexpr int QS = TPW * 512;                  // nibble words
  static constexpr int SC = TPW * 64;                   // fp16 scales
  static constexpr int QH = QT == 6 ? TPW * 256 : 0;    // 6-bit high fields
  static constexpr int STAGE = QS + SC + QH;
  static constexpr int WARP_BYTES = NS * STAGE;
  static constexpr int CTA_BYTES = WARPS * WARP_BYTES;
};

// ---------------------------------------------------------------------------
// repack: canonical planes -> streaming layout
// ---------------------------------------------------------------------------
__device__ __forceinline__ int perm_row(int p, PermKind perm, int hd, int N) {
  if (perm == PERM_ROPE_PAIRS) {
    int h = p / hd, w = p % hd, j = w / 16, rho = w % 16;
    int dim = rho < 8 ? 8 * j + rho : hd / 2 + 8 * j + (rho - 8);
    return h * hd + dim;
  }
  if (perm == PERM_GATE_UP) {
    int F = N / 2, j = p / 16, rho = p % 16;
    return rho < 8 ? 8 * j + rho : F + 8 * j + (rho - 8);
  }
  return p;
}

// u = q + bias of canonical element (row n, column k); padding gives q = 0.
__device__ __forceinline__ uint32_t canon_u(int qtype, const uint8_t* qs,
                                            const uint8_t* qh, int n, int K, int k) {
  if (k >= K) return qtype == 4 ? 8u : 32u;
  int nb = K / 32, b = k / 32, j = k % 32;
  uint8_t byte = qs[((size_t)n * nb + b) * 16 + (j % 16)];
  uint32_t lo = j < 16 ? (byte & 0xF) : (byte >> 4);
  if (qtype == 4) return lo;
  uint32_t hi = (qh[((size_t)n * nb + b) * 8 + j / 4] >> (2 * (j % 4))) & 3u;
  return lo | (hi << 4);
}

__global__ void pack_kernel(int qtype, const uint8_t* __restrict__ qs,
                            const uint8_t* __restrict__ qh,
                            const uint16_t* __restrict__ scales, int N, int K,
                            int nch, PermKind perm, int hd, uint4* __restrict__ oqs,
                            uint2* __restrict__ oqh, uint2* __restrict__ osc) {
  const int n_tiles = N / 16;
  size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  size_t total = (size_t)n_tiles * nch * 32;
  if (idx >= total) return;
  const int lane = (int)(idx % 32);
  const int c = (int)((idx / 32) % nch);
  const int T = (int)(idx / 32 / nch);
  const int g = lane >> 2, t = lane & 3;
  const int row_g = perm_row(T * 16 + g, perm, hd, N);
  const int row_g8 = perm_row(T * 16 + g + 8, perm, hd, N);
  // nibble slot i -> (row, element e): i = 0,4,2,6 -> row g e = 0,1,2,3;
  //                                    i = 1,5,3,7 -> row g+8 e = 0,1,2,3.
  const int slot_row8[8] = {0, 1, 0, 1, 0, 1, 0, 1};
  const int slot_e[8] = {0, 0, 2, 2, 1, 1, 3, 3};
  // Q6 high-field bit positions of nibble slot i, step A / step B.
  const int posA[8] = {4, 8, 6, 10, 20, 24, 22, 26};
  uint32_t w[4], hw[2] = {0u, 0u};
  for (int j = 0; j < 4; j++) {
    const int b = j / 2, jj = j % 2;
    uint32_t word = 0;
    for (int i = 0; i < 8; i++) {
      int row = slot_row8[i] ? row_g8 : row_g;
      int k = 64 * c + 32 * b + 8 * t + 4 * jj + slot_e[i];
      uint32_t u = canon_u(qtype, qs, qh, row, K, k);
      word |= (u & 0xFu) << (4 * i);
      if (qtype == 6) {
        int pos = jj == 0 ? posA[i] : (posA[i] + 24) % 32;  // rotl by 8 restores posA
        hw[b] |= ((u >> 4) & 3u) << pos;
      }
    }
    w[j] = word;
  }
  size_t o = ((size_t)T * nch + c) * 32 + lane;
  oqs[o] = make_uint4(w[0], w[1], w[2], w[3]);
  if (qtype == 6) oqh[o] = make_uint2(hw[0], hw[1]);
  if (t == 0) {
    const int nb = K / 32;
    auto sc_of = [&](int row, int blk) -> uint32_t {
      return blk < nb ? (uint32_t)scales[(size_t)row * nb + blk] : 0u;
    };
    uint32_t s0 = sc_of(row_g, 2 * c) | (sc_of(row_g8, 2 * c) << 16);
    uint32_t s1 = sc_of(row_g, 2 * c + 1) | (sc_of(row_g8, 2 * c + 1) << 16);
    osc[((size_t)T * nch + c) * 8 + g] = make_uint2(s0, s1);
  }
}

// ---------------------------------------------------------------------------
// the verify GEMM
// ---------------------------------------------------------------------------
struct LinArgs {
  const uint4* qs;
  const uint2* qh;
  const uint2* sc;
  const __half* x;
  int N, K, nch, n_tiles, S, R, n_grp;
  LinEpi epi;
  float* part;
  unsigned* tickets;
  float2* amax_part;
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Issue the copies of chunk c of this warp's tiles into ring stage `st`.
template <int QT>
__device__ __forceinline__ void issue_chunk(const LinArgs& a, unsigned char* st, int tile0, int c,
                                            int lane) {
#pragma unroll
  for (int i = 0; i < TPW; i++) {
    const int T = tile0 + i;
    if (T >= a.n_tiles) continue;
    const size_t u = (size_t)T * a.nch + c;
    cp_async16(smem_addr(st + i * 512 + lane * 16), a.qs + u * 32 + lane);
    if (lane < 4) cp_async16(smem_addr(st + Ring<QT>::QS + i * 64 + lane * 16), a.sc + u * 8 + 2 * lane);
    if constexpr (QT == 6)
      if (lane < 16)
        cp_async16(smem_addr(st + Ring<QT>::QS + Ring<QT>::SC + i * 256 + lane * 16),
                   a.qh + u * 32 + 2 * lane);
  }
}

// Activations (B operand) of chunk c for this lane: rows zrow0 + ct*8 + g,
// k = 64c + 32b + 8t .. +7 (zero beyond R or K).
template <int NCT>
__device__ __forceinline__ void load_x(uint4 (&xb)[NCT][2], const LinArgs& a, int c, int zrow0,
                                       int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int ct = 0; ct < NCT; ct++) {
    const int r = zrow0 + ct * 8 + g;
#pragma unroll
    for (int b = 0; b < 2; b++) {
      const int k = 64 * c + 32 * b + 8 * t;
      if (r < a.R && k < a.K)
        xb[ct][b] = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)r * a.K + k));
      else
        xb[ct][b] = make_uint4(0, 0, 0, 0);
    }
  }
}

// A fragments of one k16 step from a packed nibble word (+ Q6 high fields).
template <int QT>
__device__ __forceinline__ void dequant_step(uint32_t w, uint32_t hx, uint32_t (&A)[4]) {
  const uint32_t MAG = 0x64006400u;
  uint32_t w8 = w >> 8;
  uint32_t r0 = lop3_and_or(w, 0x000F000Fu, MAG);
  uint32_t r1 = lop3_and_or(w, 0x00F000F0u, MAG);
  uint32_t r2 = lop3_and_or(w8, 0x000F000Fu, MAG);
  uint32_t r3 = lop3_and_or(w8, 0x00F000F0u, MAG);
  if constexpr (QT == 6) {
    uint32_t hx2 = hx >> 2;
    r0 = lop3_and_or(hx, 0x00300030u, r0);
    r1 = lop3_and_or(hx, 0x03000300u, r1);
    r2 = lop3_and_or(hx2, 0x00300030u, r2);
    r3 = lop3_and_or(hx2, 0x03000300u, r3);
  }
  // bits-0.. form: h = 1024 + u  -> q = h - (1024 + bias)
  // bits-4.. form: h = 1024 + 16u -> q = h/16 - (64 + bias)
  const __half2 sub = QT == 4 ? __half2half2(__ushort_as_half(0x6408))   // 1032
                              : __half2half2(__ushort_as_half(0x6420));  // 1056
  const __half2 sixteenth = __half2half2(__ushort_as_half(0x2C00));      // 1/16
  const __half2 off = QT == 4 ? __half2half2(__ushort_as_half(0xD480))   // -72
                              : __half2half2(__ushort_as_half(0xD600));  // -96
  __half2 h0 = __hsub2(*reinterpret_cast<__half2*>(&r0), sub);
  __half2 h1 = __hfma2(*reinterpret_cast<__half2*>(&r1), sixteenth, off);
  __half2 h2 = __hsub2(*reinterpret_cast<__half2*>(&r2), sub);
  __half2 h3 = __hfma2(*reinterpret_cast<__half2*>(&r3), sixteenth, off);
  A[0] = *reinterpret_cast<uint32_t*>(&h0);
  A[1] = *reinterpret_cast<uint32_t*>(&h1);
  A[2] = *reinterpret_cast<uint32_t*>(&h2);
  A[3] = *reinterpret_cast<uint32_t*>(&h3);
}

template <int QT, int NCT>
__device__ __forceinline__ void compute_chunk(const unsigned char* st, const uint4 (&xb)[NCT][2],
                                              int tile0, int n_tiles, int lane,
                                              float (&acc)[TPW][NCT][4]) {
  const int g = lane >> 2;
#pragma unroll
  for (int i = 0; i < TPW; i++) {
    if (tile0 + i >= n_tiles) continue;
    const uint4 aw = *reinterpret_cast<const uint4*>(st + i * 512 + lane * 16);
    const uint2 sw = *reinterpret_cast<const uint2*>(st + Ring<QT>::QS + i * 64 + g * 8);
    uint2 hw = make_uint2(0, 0);
    if constexpr (QT == 6)
      hw = *reinterpret_cast<const uint2*>(st + Ring<QT>::QS + Ring<QT>::SC + i * 256 + lane * 8);
    const uint32_t words[4] = {aw.x, aw.y, aw.z, aw.w};
    const float2 s0 = __half22float2(*reinterpret_cast<const __half2*>(&sw.x));
    const float2 s1 = __half22float2(*reinterpret_cast<const __half2*>(&sw.y));
#pragma unroll
    for (int b = 0; b < 2; b++) {
      uint32_t hA = 0, hB = 0;
      if constexpr (QT == 6) {
        hA = b == 0 ? hw.x : hw.y;
        hB = __funnelshift_l(hA, hA, 8);
      }
      uint32_t A0[4], A1[4];
      dequant_step<QT>(words[2 * b], hA, A0);
      dequant_step<QT>(words[2 * b + 1], hB, A1);
      const float sg = b == 0 ? s0.x : s1.x;   // row g
      const float sg8 = b == 0 ? s0.y : s1.y;  // row g+8
#pragma unroll
      for (int ct = 0; ct < NCT; ct++) {
        float blk[4];
        mma_16816_zero(blk, A0, xb[ct][b].x, xb[ct][b].y);
        mma_16816(blk, A1, xb[ct][b].z, xb[ct][b].w);
        acc[i][ct][0] = fmaf(sg, blk[0], acc[i][ct][0]);
        acc[i][ct][1] = fmaf(sg, blk[1], acc[i][ct][1]);
        acc[i][ct][2] = fmaf(sg8, blk[2], acc[i][ct][2]);
        acc[i][ct][3] = fmaf(sg8, blk[3], acc[i][ct][3]);
      }
    }
  }
}

__device__ __forceinline__ bool amax_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Epilogue for one tile/column-tile fragment of finished sums.
template <int NCT>
__device__ __forceinline__ void epilogue_frag(const LinArgs& a, int T, int ct,
                                              int zrow0, int lane, const float (&v)[4],
                                              float (&bestv)[NCT][2], int (&besti)[NCT][2]) {
  const int g = lane >> 2, t = lane & 3;
  const LinEpi& e = a.epi;
  const int n0 = T * 16 + g, n1 = n0 + 8;
#pragma unroll
  for (int c = 0; c < 2; c++) {
    const int r = zrow0 + ct * 8 + 2 * t + c;
    const bool ok = r < a.R;
    const float x0 = v[c], x1 = v[2 + c];  // rows g and g+8, column r
    switch (e.kind) {
      case EPI_STORE:
        if (ok) {
          e.y[(size_t)r * e.ldy + n0] = x0;
          e.y[(size_t)r * e.ldy + n1] = x1;
        }
        break;
      case EPI_RESID:
        if (ok) {
          e.y[(size_t)r * e.ldy + n0] += x0;
          e.y[(size_t)r * e.ldy + n1] += x1;
        }
        break;
      case EPI_SWIGLU:
        if (ok) {
          const float sil = x0 / (1.0f + expf(-x0));
          e.out16[(size_t)r * e.ldo + T * 8 + g] = __float2half_rn(sil * x1);
        }
        break;
      case EPI_QKV:
        if (ok) {
          const int per_head = e.hd / 16;
          const int hh = T / per_head, j = T % per_head;
          const int i0 = 8 * j + g, i1 = e.hd / 2 + 8 * j + g;
          const RowInfo ri = e.rows[r];
          float y0 = x0, y1 = x1;
          if (e.rope != nullptr && hh < e.nq + e.nkv) {
            const int rp = ri.pos < e.max_ctx ? ri.pos : e.max_ctx - 1;  // invalid rows are flagged
            const float2 cs = e.rope[(size_t)rp * (e.hd / 2) + i0];
            y0 = x0 * cs.x - x1 * cs.y;
            y1 = x1 * cs.x + x0 * cs.y;
          }
          __half* dst;
          if (hh < e.nq) {
            dst = e.out16 + ((size_t)r * e.nq + hh) * e.hd;
          } else {
            const bool isk = hh < e.nq + e.nkv;
            const int kvh = isk ? hh - e.nq : hh - e.nq - e.nkv;
            if (ri.pos >= e.max_ctx) break;  // flagged by the row-info kernel
            dst = (isk ? e.kcache : e.vcache) +
                  (((size_t)ri.slot * e.nkv + kvh) * e.max_ctx + ri.pos) * e.hd;
          }
          dst[i0] = __float2half_rn(y0);
          dst[i1] = __float2half_rn(y1);
        }
        break;
      case EPI_LMHEAD:
        if (ok) {
          if (e.y != nullptr) {
            e.y[(size_t)r * e.ldy + n0] = x0;
            e.y[(size_t)r * e.ldy + n1] = x1;
          }
          if (x0 != x0 || x1 != x1) atomicOr(e.err, ERR_NONFINITE);
          if (amax_better(x0, n0, bestv[ct][c], besti[ct][c])) {
            bestv[ct][c] = x0;
            besti[ct][c] = n0;
          }
          if (amax_better(x1, n1, bestv[ct][c], besti[ct][c])) {
            bestv[ct][c] = x1;
            besti[ct][c] = n1;
          }
        }
        break;
    }
  }
}

template <int QT, int NCT>
__global__ void __launch_bounds__(WARPS * 32)
linear_q_kernel(const LinArgs a) {
  extern __shared__ __align__(128) unsigned char ring_smem[];
  constexpr int NS = Ring<QT>::NS;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int z = blockIdx.x, grp = blockIdx.y, seg = blockIdx.z;
  const int tile0 = (grp * WARPS + warp) * TPW;
  const int zrow0 = z * 8 * NCT;
  const int c_begin = (int)((long long)seg * a.nch / a.S);
  const int c_end = (int)((long long)(seg + 1) * a.nch / a.S);
  unsigned char* ring = ring_smem + warp * Ring<QT>::WARP_BYTES;

  float acc[TPW][NCT][4];
#pragma unroll
  for (int i = 0; i < TPW; i++)
#pragma unroll
    for (int ct = 0; ct < NCT; ct++)
#pragma unroll
      for (int q = 0; q < 4; q++) acc[i][ct][q] = 0.0f;

  if (tile0 < a.n_tiles) {
    const int nc = c_end - c_begin;
#pragma unroll
    for (int j = 0; j < NS - 1; j++) {
      if (j < nc) issue_chunk<QT>(a, ring + j * Ring<QT>::STAGE, tile0, c_begin + j, lane);
      cp_async_commit();
    }
    uint4 xb[NCT][2], xn[NCT][2];
    load_x<NCT>(xb, a, c_begin, zrow0, lane);
    for (int j = 0; j < nc; j++) {
      cp_async_wait<NS - 2>();  // chunk j has landed (this lane's copies)
      __syncwarp();             // ... and every lane's
      const int jn = j + NS - 1;
      if (jn < nc) issue_chunk<QT>(a, ring + (jn % NS) * Ring<QT>::STAGE, tile0, c_begin + jn, lane);
      cp_async_commit();
      if (j + 1 < nc) load_x<NCT>(xn, a, c_begin + j + 1, zrow0, lane);
      compute_chunk<QT, NCT>(ring + (j % NS) * Ring<QT>::STAGE, xb, tile0, a.n_tiles, lane, acc);
#pragma unroll
      for (int ct = 0; ct < NCT; ct++) {
        xb[ct][0] = xn[ct][0];
        xb[ct][1] = xn[ct][1];
      }
    }
    cp_async_wait<0>();
  }

  // ---- K-split: the last CTA of this (column group, tile group) sums the
  // ---- S partials in segment order.
  if (a.S > 1) {
    __shared__ int s_last;
    const int ZG = gridDim.x;
    if (tile0 < a.n_tiles) {
#pragma unroll
      for (int i = 0; i < TPW; i++) {
        const int T = tile0 + i;
        if (T >= a.n_tiles) continue;
#pragma unroll
        for (int ct = 0; ct < NCT; ct++) {
          size_t o = ((((size_t)seg * ZG + z) * a.n_tiles + T) * NCT + ct) * 32 + lane;
          reinterpret_cast<float4*>(a.part)[o] =
              make_float4(acc[i][ct][0], acc[i][ct][1], acc[i][ct][2], acc[i][ct][3]);
        }
      }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned prev = atomicAdd(&a.tickets[z * a.n_grp + grp], 1u);
      s_last = (prev == (unsigned)(a.S - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tile0 < a.n_tiles) {
#pragma unroll
      for (int i = 0; i < TPW; i++) {
        const int T = tile0 + i;
        if (T >= a.n_tiles) continue;
#pragma unroll
        for (int ct = 0; ct < NCT; ct++) {
          float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int s = 0; s < a.S; s++) {
            size_t o = ((((size_t)s * ZG + z) * a.n_tiles + T) * NCT + ct) * 32 + lane;
            float4 p = __ldcg(reinterpret_cast<const float4*>(a.part) + o);
            if (s == 0) {
              sum = p;
            } else {
              sum.x += p.x; sum.y += p.y; sum.z += p.z; sum.w += p.w;
            }
          }
          acc[i][ct][0] = sum.x; acc[i][ct][1] = sum.y;
          acc[i][ct][2] = sum.z; acc[i][ct][3] = sum.w;
        }
      }
    }
    if (threadIdx.x == 0) a.tickets[z * a.n_grp + grp] = 0u;  // ready for the next launch
  }

  // ---- epilogue
  float bestv[NCT][2];
  int besti[NCT][2];
#pragma unroll
  for (int ct = 0; ct < NCT; ct++)
#pragma unroll
    for (int c = 0; c < 2; c++) { bestv[ct][c] = -INFINITY; besti[ct][c] = 0x7fffffff; }
  if (tile0 < a.n_tiles) {
#pragma unroll
    for (int i = 0; i < TPW; i++) {
      const int T = tile0 + i;
      if (T >= a.n_tiles) continue;
#pragma unroll
      for (int ct = 0; ct < NCT; ct++) epilogue_frag<NCT>(a, T, ct, zrow0, lane, acc[i][ct], bestv, besti);
    }
  }
  if (a.epi.kind != EPI_LMHEAD) return;

  // ---- fused argmax: warp (over the 8 row lanes g) -> CTA -> grid.
  __shared__ float s_v[WARPS][8 * NCT];
  __shared__ int s_i[WARPS][8 * NCT];
  __shared__ int s_last_am;
#pragma unroll
  for (int ct = 0; ct < NCT; ct++)
#pragma unroll
    for (int c = 0; c < 2; c++) {
      float v = bestv[ct][c];
      int id = besti[ct][c];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, v, off);
        int oi = __shfl_xor_sync(0xffffffffu, id, off);
        if (amax_better(ov, oi, v, id)) { v = ov; id = oi; }
      }
      if ((lane >> 2) == 0) {
        s_v[warp][ct * 8 + 2 * (lane & 3) + c] = v;
        s_i[warp][ct * 8 + 2 * (lane & 3) + c] = id;
      }
    }
  __syncthreads();
  if (threadIdx.x < 8 * NCT) {
    const int col = threadIdx.x;
    float v = s_v[0][col];
    int id = s_i[0][col];
    for (int w = 1; w < WARPS; w++)
      if (amax_better(s_v[w][col], s_i[w][col], v, id)) { v = s_v[w][col]; id = s_i[w][col]; }
    a.amax_part[((size_t)z * a.n_grp + grp) * 16 + col] = make_float2(v, __int_as_float(id));
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned prev = atomicAdd(&a.tickets[gridDim.x * a.n_grp + z], 1u);
    s_last_am = (prev == (unsigned)(a.n_grp - 1));
  }
  __syncthreads();
  if (!s_last_am) return;
  __threadfence();
  if (threadIdx.x < 8 * NCT) {
    const int col = threadIdx.x;
    const int r = zrow0 + col;
    float v = -INFINITY;
    int id = 0x7fffffff;
    for (int gi = 0; gi < a.n_grp; gi++) {
      float2 p = __ldcg(a.amax_part + ((size_t)z * a.n_grp + gi) * 16 + col);
      int pi = __float_as_int(p.y);
      if (amax_better(p.x, pi, v, id)) { v = p.x; id = pi; }
    }
    if (r < a.R && a.epi.argmax != nullptr) a.epi.argmax[r] = id == 0x7fffffff ? 0 : id;
  }
  if (threadIdx.x == 0) a.tickets[gridDim.x * a.n_grp + z] = 0u;
}

// K-split for a matrix: fixed by its shape and the device only (never by
// nt, so rows stay bitwise nt-invariant).  Cost model: the launch runs
// ceil(CTAs / resident slots) waves, each as long as one segment (nch / S
// chunks) plus a start-up latency worth ~2 chunks and the partial-sum write
// (~0.5 chunk); the last CTA of a group reads S partials (~0.45 chunk each).
int choose_split(int n_tiles, int nch, int slots) {
  const int n_grp = (n_tiles + WARPS * TPW - 1) / (WARPS * TPW);
  const int s_max = std::max(1, nch / 2);
  int best = 1;
  double best_cost = 1e30;
  for (int S = 1; S <= s_max; S++) {
    const double waves = std::ceil((double)n_grp * S / slots);
    const double cost = waves * ((double)nch / S + 2.0 + (S > 1 ? 0.5 : 0.0)) +
                        (S > 1 ? 0.45 * S : 0.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

template <int QT, int NCT>
void launch_typed(const LinArgs& a, int ZG, cudaStream_t st) {
  dim3 grid(ZG, a.n_grp, a.S);
  linear_q_kernel<QT, NCT><<<grid, WARPS * 32, Ring<QT>::CTA_BYTES, st>>>(a);
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
int qmat_pack(const spec_qweight* w, PermKind perm, int head_dim, int split_sms,
              cudaStream_t st, QMat* out) {
  if (w == nullptr || out == nullptr) return fail(SPEC_E_INVALID, "null qweight");
  if (w->qtype != SPEC_Q4 && w->qtype != SPEC_Q6)
    return fail(SPEC_E_UNSUPPORTED, "qtype must be SPEC_Q4 or SPEC_Q6");
  if (w->N <= 0 || w->K <= 0 || w->N % 16 != 0 || w->K % 32 != 0)
    return fail(SPEC_E_SHAPE, "need N % 16 == 0 and K % 32 == 0");
  if (w->qs == nullptr || w->scales == nullptr || (w->qtype == SPEC_Q6 && w->qh == nullptr))
    return fail(SPEC_E_INVALID, "missing weight plane");
  if (perm == PERM_ROPE_PAIRS && (head_dim % 16 != 0 || w->N % head_dim != 0))
    return fail(SPEC_E_SHAPE, "head_dim must be a multiple of 16 dividing N");
  if (perm == PERM_GATE_UP && w->N % 32 != 0)
    return fail(SPEC_E_SHAPE, "gate/up rows must be a multiple of 32");
  QMat q;
  q.qtype = w->qtype;
  q.N = w->N;
  q.K = w->K;
  q.Kp = (w->K + 63) / 64 * 64;
  q.nch = q.Kp / 64;
  q.n_tiles = q.N / 16;
  if (split_sms > 0) {
    // resident CTAs per SM of the nt <= 8 variant (the split must not depend on nt)
    int per_sm = 0;
    if (q.qtype == 4)
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, linear_q_kernel<4, 1>, WARPS * 32,
                                                    Ring<4>::CTA_BYTES);
    else
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, linear_q_kernel<6, 1>, WARPS * 32,
                                                    Ring<6>::CTA_BYTES);
    cudaGetLastError();
    q.S = choose_split(q.n_tiles, q.nch, split_sms * std::max(per_sm, 1));
  } else {
    q.S = 1;
  }
  const size_t units = (size_t)q.n_tiles * q.nch;
  const size_t b_qs = units * 32 * sizeof(uint4);
  const size_t b_qh = q.qtype == 6 ? units * 32 * sizeof(uint2) : 0;
  const size_t b_sc = units * 8 * sizeof(uint2);
  q.bytes = b_qs + b_qh + b_sc;
  if (cudaMalloc(&q.base, q.bytes) != cudaSuccess) {
    cudaGetLastError();
    return fail(SPEC_E_OOM, "cudaMalloc of packed weights failed");
  }
  q.qs = reinterpret_cast<uint4*>(q.base);
  q.qh = q.qtype == 6 ? reinterpret_cast<uint2*>((char*)q.base + b_qs) : nullptr;
  q.sc = reinterpret_cast<uint2*>((char*)q.base + b_qs + b_qh);
  const size_t total = units * 32;
  const int threads = 256;
  pack_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, st>>>(
      q.qtype, (const uint8_t*)w->qs, (const uint8_t*)w->qh,
      (const uint16_t*)w->scales, q.N, q.K, q.nch, perm, head_dim, q.qs, q.qh, q.sc);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    cudaFree(q.base);
    return fail(SPEC_E_CUDA, std::string("pack kernel: ") + cudaGetErrorString(e));
  }
  *out = q;
  return SPEC_OK;
}

void qmat_free(QMat* q) {
  if (q->base) cudaFree(q->base);
  *q = QMat();
}

static int col_tiles(int R) { return R <= 8 ? 1 : 2; }
static int col_groups(int R) { return (R + 8 * col_tiles(R) - 1) / (8 * col_tiles(R)); }
static int tile_groups(const QMat& w) { return (w.n_tiles + WARPS * TPW - 1) / (WARPS * TPW); }

size_t lin_part_floats(const QMat& w, int R) {
  if (w.S <= 1) return 0;
  return (size_t)w.S * col_groups(R) * w.n_tiles * col_tiles(R) * 32 * 4;
}
size_t lin_tickets_needed(const QMat& w, int R) {
  return (size_t)col_groups(R) * tile_groups(w) + col_groups(R);  // K-split + argmax
}
size_t lin_amax_entries(const QMat& w, int R) {
  return (size_t)col_groups(R) * tile_groups(w) * 16;
}

int linear_launch(const QMat& w, const __half* x, int R, const LinEpi& epi,
                  const LinScratch& scr, cudaStream_t st) {
  if (R < 1) return fail(SPEC_E_SHAPE, "linear: R must be >= 1");
  if (lin_part_floats(w, R) > scr.part_floats || lin_tickets_needed(w, R) > scr.n_tickets ||
      (epi.kind == EPI_LMHEAD && lin_amax_entries(w, R) > scr.amax_entries))
    return fail(SPEC_E_SHAPE, "linear: scratch too small for this R");
  LinArgs a;
  a.qs = w.qs;
  a.qh = w.qh;
  a.sc = w.sc;
  a.x = x;
  a.N = w.N;
  a.K = w.K;
  a.nch = w.nch;
  a.n_tiles = w.n_tiles;
  a.S = w.S;
  a.R = R;
  a.n_grp = tile_groups(w);
  a.epi = epi;
  a.part = scr.part;
  a.tickets = scr.tickets;
  a.amax_part = scr.amax_part;
  const int ZG = col_groups(R);
  const int nct = col_tiles(R);
  if (w.qtype == 4) {
    if (nct == 1) launch_typed<4, 1>(a, ZG, st);
    else launch_typed<4, 2>(a, ZG, st);
  } else {
    if (nct == 1) launch_typed<6, 1>(a, ZG, st);
    else launch_typed<6, 2>(a, ZG, st);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SPEC_E_CUDA, std::string("linear launch: ") + cudaGetErrorString(e));
  return SPEC_OK;
}

void linear_init_attrs() {
  cudaFuncSetAttribute(linear_q_kernel<4, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, Ring<4>::CTA_BYTES);
  cudaFuncSetAttribute(linear_q_kernel<4, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, Ring<4>::CTA_BYTES);
  cudaFuncSetAttribute(linear_q_kernel<6, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, Ring<6>::CTA_BYTES);
  cudaFuncSetAttribute(linear_q_kernel<6, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, Ring<6>::CTA_BYTES);
}
