// linear.cu -- weights-once multi-row dequant GEMM of the verify pass.
//
// "Speculative Decoding (D5-R) -- Plan", section 1: the batched verify is a
// weights-once round, not a per-row restream; its cost is the weights once
// plus nt times the per-token work.  Here every packed weight byte is read
// from HBM exactly once per call, whatever nt is, and is applied to all
// nt rows in registers:
//
//   * a warp owns a pair of 16-row tiles and a stretch of K; each 64-k chunk
//     of the pair is one contiguous record in HBM, streamed with TMA bulk
//     copies through a per-warp shared-memory ring; the CTA's slice of the
//     activations is staged once in shared memory and shared by its warps;
//   * the 4-bit / 6-bit integers, masked into the mantissa from bit 4 up,
//     are exact fp16 subnormals (16u * 2^-24) and feed
//     mma.sync m16n8k16 (f16 x f16 -> f32) as the A operand; the activations
//     (n8 column tiles of verify rows) are B, and the zero point enters as
//     the C operand (-bias * sum(x), from two MMAs with a constant fragment);
//     the 8-bit integers are centred exactly in fp16 (q * 2^-20, the same
//     unit) and need no zero point;
//   * each 32-block is accumulated in a fresh fp32 fragment and folded into
//     the running sum with one fp32 FMA by its fp16 scale;
//   * K is split into S segments across CTAs and, inside a CTA, into KW
//     slices across warps ((KW, S) fixed per matrix, never per nt); the
//     slices are added in slice order through shared memory, and the last
//     CTA of a tile group to finish (a non-blocking ticket) adds the S
//     partial sums in segment order;
//   * epilogues: store, residual add, SwiGLU, RoPE + KV-cache write, and the
//     LM head's fused per-row argmax.
// Every output element is produced by the same instruction sequence for any
// nt (zero-padded columns never feed real ones), so verify rows are bitwise
// equal across nt ("Speculative Decoding (D5-R) -- Plan", status notes:
// batched verify made bitwise position-invariant).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <string>

#include "common.cuh"

namespace {

constexpr int WARPS = 8;     // warps per CTA
constexpr int TPW = 2;       // tiles (of 16 rows) per warp: one pair
constexpr int NS = 2;        // weight-ring stages per warp
// Chunks per ring stage (consecutive records: one copy, one wait) and the
// CTAs per SM the register budget is set for, by the number of column tiles.
// Two column tiles need ~110 registers (2 CTAs per SM); their shorter stages
// keep the shared memory of a Q6 LM-head CTA low enough for 2 per SM too.
// 8-bit records are twice as long: two chunks a stage at either width.
template <int QT, int NCT>
constexpr int cps() { return (NCT == 1 && QT != 8) ? 3 : 2; }
template <int NCT>
constexpr int min_blocks() { return NCT == 1 ? 3 : 2; }
constexpr int NC_CTA_MAX = 64;  // chunks of one CTA's K range (its staged activation slice)
constexpr int MAX_SPLIT = 64;

// Record of one (pair, 64-k chunk): the integer words of the 2 tiles (nibbles;
// bytes for Q8), their fp16 scales, then (Q6) the high 2-bit fields.
template <int QT>
struct Rec {
  static constexpr int QS_TILE = QT == 8 ? 1024 : 512;  // bytes of one tile's integers
  static constexpr int QS = 0;
  static constexpr int SC = TPW * QS_TILE;              // 2 x 64 B
  static constexpr int QH = SC + TPW * 64;              // 2 x 256 B (Q6)
  static constexpr int BYTES = QH + (QT == 6 ? TPW * 256 : 0);  // 1152 / 1664 / 2176
};
inline int rec_bytes(int qtype) {
  return qtype == 4 ? Rec<4>::BYTES : (qtype == 6 ? Rec<6>::BYTES : Rec<8>::BYTES);
}
inline int stage_chunks(int qtype, int nct) {
  if (qtype == 8) return nct == 1 ? cps<8, 1>() : cps<8, 2>();
  return nct == 1 ? cps<4, 1>() : cps<4, 2>();
}
inline int ring_bytes(int qtype, int nct) {
  return WARPS * NS * stage_chunks(qtype, nct) * rec_bytes(qtype);
}
// Staged activation row: the CTA's K range plus 64 bytes, so that the rows
// g = 0..7 of a fragment load fall in distinct shared-memory banks.
inline int x_stride(int nc) { return nc * 128 + 64; }
inline int smem_bytes(int qtype, int nct, int nc) {
  return ring_bytes(qtype, nct) + 8 * nct * x_stride(nc);
}

// ---------------------------------------------------------------------------
// repack: canonical planes -> streaming records
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

// One thread per (tile T of the padded quads, chunk c, lane).  For lane
// l = 4g + t, the nibble word of k16 step j (block b = j/2, half jj = j%2)
// holds, in nibble slots 0,4,2,6, row g at k = 64c + 32b + 8t + 4jj + 0..3,
// and in slots 1,5,3,7 row g+8 at the same k: exactly the A fragment of
// mma.m16n8k16 after the magic-number extraction, with the k order inside
// each 32-block permuted so that lane t reads 8 consecutive activations.
// Q6 high fields of block b: step 2b at bits 4..11 / 20..27 of one word,
// step 2b+1 where a rotate by 8 brings them to the same places.
__global__ void pack_kernel(int qtype, const uint8_t* __restrict__ qs,
                            const uint8_t* __restrict__ qh,
                            const uint16_t* __restrict__ scales, int N, int K, int nch,
                            int n_groups, PermKind perm, int hd, int rec_bytes,
                            uint8_t* __restrict__ out) {
  const int n_tiles = N / 16;
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t total = (size_t)n_groups * TPW * nch * 32;
  if (idx >= total) return;
  const int lane = (int)(idx % 32);
  const int c = (int)((idx / 32) % nch);
  const int T = (int)(idx / 32 / nch);
  const int Q = T / TPW, i = T % TPW;
  const int g = lane >> 2, t = lane & 3;
  uint8_t* rec = out + ((size_t)Q * nch + c) * rec_bytes;
  const bool real = T < n_tiles;
  const int row_g = real ? perm_row(T * 16 + g, perm, hd, N) : 0;
  const int row_g8 = real ? perm_row(T * 16 + g + 8, perm, hd, N) : 0;
  if (qtype == 8) {
    // Q8: for block b and k pair j, one word holds bytes u = q + 128 of rows
    // g, g, g+8, g+8 at k = 64c + 32b + 8t + 2j, +1 (the same k order as the
    // 4-bit words): a byte permute turns it into two A registers.
    const int nb = K / 32;
    auto u8 = [&](int row, int k) -> uint32_t {
      if (!real || k >= K) return 128u;
      return (uint32_t)((int)(int8_t)qs[((size_t)row * nb + k / 32) * 32 + k % 32] + 128);
    };
    uint32_t w8[8];
    for (int b = 0; b < 2; b++)
      for (int j = 0; j < 4; j++) {
        const int k = 64 * c + 32 * b + 8 * t + 2 * j;
        w8[4 * b + j] = u8(row_g, k) | (u8(row_g, k + 1) << 8) | (u8(row_g8, k) << 16) |
                        (u8(row_g8, k + 1) << 24);
      }
    uint4* dst = reinterpret_cast<uint4*>(rec + Rec<8>::QS + i * Rec<8>::QS_TILE + lane * 32);
    dst[0] = make_uint4(w8[0], w8[1], w8[2], w8[3]);
    dst[1] = make_uint4(w8[4], w8[5], w8[6], w8[7]);
  } else {
    const int slot_row8[8] = {0, 1, 0, 1, 0, 1, 0, 1};
    const int slot_e[8] = {0, 0, 2, 2, 1, 1, 3, 3};
    const int posA[8] = {4, 8, 6, 10, 20, 24, 22, 26};
    uint32_t w[4], hw[2] = {0u, 0u};
    for (int j = 0; j < 4; j++) {
      const int b = j / 2, jj = j % 2;
      uint32_t word = 0;
      for (int s = 0; s < 8; s++) {
        const int k = 64 * c + 32 * b + 8 * t + 4 * jj + slot_e[s];
        const uint32_t u = real ? canon_u(qtype, qs, qh, slot_row8[s] ? row_g8 : row_g, K, k)
                                : (qtype == 4 ? 8u : 32u);
        word |= (u & 0xFu) << (4 * s);
        if (qtype == 6) {
          const int pos = jj == 0 ? posA[s] : (posA[s] + 24) % 32;  // rotl by 8 restores posA
          hw[b] |= ((u >> 4) & 3u) << pos;
        }
      }
      w[j] = word;
    }
    *reinterpret_cast<uint4*>(rec + Rec<4>::QS + i * 512 + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    if (qtype == 6)
      *reinterpret_cast<uint2*>(rec + Rec<6>::QH + i * 256 + lane * 8) = make_uint2(hw[0], hw[1]);
  }
  if (t == 0) {
    const int nb = K / 32;
    auto sc_of = [&](int row, int blk) -> uint32_t {
      return (real && blk < nb) ? (uint32_t)scales[(size_t)row * nb + blk] : 0u;
    };
    const uint32_t s0 = sc_of(row_g, 2 * c) | (sc_of(row_g8, 2 * c) << 16);
    const uint32_t s1 = sc_of(row_g, 2 * c + 1) | (sc_of(row_g8, 2 * c + 1) << 16);
    const int sc_off = qtype == 8 ? Rec<8>::SC : Rec<4>::SC;
    *reinterpret_cast<uint2*>(rec + sc_off + i * 64 + g * 8) = make_uint2(s0, s1);
  }
}

// ---------------------------------------------------------------------------
// the verify GEMM
// ---------------------------------------------------------------------------
struct LinArgs {
  const uint8_t* rec;
  const __half* x;
  int N, K, nch, n_tiles, n_pairs, n_grp, S, R;
  int xstride;        // bytes per staged activation row
  LinEpi epi;
  float* part;        // [S][ZG][n_tiles][NCT][32] float4
  unsigned* tickets;  // [ZG][n_grp] K-split tickets, then [ZG] argmax tickets
  float2* amax_part;  // [ZG][n_grp][16]
  uint32_t* err;      // device error word (ERR_TIMEOUT on a copy that never arrived)
  int first_tries;    // try budget of the first wait (the activation slice)
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// --- mbarrier + bulk-copy (TMA) helpers -----------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// One contiguous global -> shared copy, completion counted on `bar`.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// The same for streamed weights, with an L2 policy of evict first: each
// weight is read once, and the L2 keeps the round's activations and cache
// instead (8-layer decoder round at nt 8: 587 -> 577 us).
__device__ __forceinline__ void bulk_copy_weights(uint32_t dst, const void* src, uint32_t bytes,
                                                  uint32_t bar) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(10000)  // suspend at most ~10 us per try
      : "memory");
  return ok != 0;
}
// Bounded wait for a phase of `bar`: about a second at most, then false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          int tries = LIN_WAIT_TRIES) {
  for (int i = 0; i < tries; i++)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// A fragments of one k16 step from a packed nibble word (+ Q6 high fields),
// as fp16 subnormals: a value u masked into the mantissa is exactly
// u * 2^-24.  Every value is placed from mantissa bit 4 up (16u * 2^-24,
// below 1024 * 2^-24 for 6 bits): the tensor cores accumulate products of
// the very smallest subnormals with less precision, and at this scale the
// sums are as accurate as those of centred fp16 integers.  The zero point is
// subtracted through the MMA's C operand (see compute_chunk) and the 2^-20
// unit is undone once, exactly, in the epilogue.
template <int QT>
__device__ __forceinline__ void dequant_step(uint32_t w, uint32_t hx, uint32_t (&A)[4]) {
  if constexpr (QT == 4) {
    A[0] = (w << 4) & 0x00F000F0u;  // rows g, k 2t..2t+1
    A[1] = w & 0x00F000F0u;         // rows g+8
    A[2] = (w >> 4) & 0x00F000F0u;  // rows g, k 2t+8..2t+9
    A[3] = (w >> 8) & 0x00F000F0u;  // rows g+8
  } else {
    const uint32_t w8 = w >> 8, hx2 = hx >> 2;
    A[0] = ((w & 0x000F000Fu) | (hx & 0x00300030u)) << 4;
    A[1] = (w & 0x00F000F0u) | (hx & 0x03000300u);
    A[2] = ((w8 & 0x000F000Fu) | (hx2 & 0x00300030u)) << 4;
    A[3] = (w8 & 0x00F000F0u) | (hx2 & 0x03000300u);
  }
}

// Two A registers from one Q8 word (bytes u = q + 128 of rows r, r, r', r'
// at k, k+1): the byte permute makes each half 0x64uu, which is 1024 + u
// exactly, and one packed FMA gives (1024 + u) * 2^-20 - 1152 * 2^-20 =
// q * 2^-20.  That value is a multiple of 2^-24 below 2^-12, so it is an
// fp16 number (a subnormal for |q| < 64) and the FMA is exact.  The unit
// 2^-20 is the 4/6-bit fragments' (16u * 2^-24 from mantissa bit 4 up).
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const __half2 unit = __halves2half2(__ushort_as_half(0x0010), __ushort_as_half(0x0010));  // 2^-20
  const __half2 off = __halves2half2(__ushort_as_half(0x9480), __ushort_as_half(0x9480));   // -1152 * 2^-20
  const uint32_t a = __byte_perm(w, 0x64646464u, 0x4140);  // rows r: k, k+1
  const uint32_t b = __byte_perm(w, 0x64646464u, 0x4342);  // rows r': k, k+1
  const __half2 ha = __hfma2(*reinterpret_cast<const __half2*>(&a), unit, off);
  const __half2 hb = __hfma2(*reinterpret_cast<const __half2*>(&b), unit, off);
  lo = *reinterpret_cast<const uint32_t*>(&ha);
  hi = *reinterpret_cast<const uint32_t*>(&hb);
}

// The unit of the dequantised fragments, undone in the epilogue: 2^20.
constexpr float FRAG_UNIT = 1048576.0f;

// The zero-point fragment: -16 * bias * 2^-24 (Q4: bias 8 -> -2^-17; Q6:
// bias 32 -> -2^-15, both exact fp16).  Its product with a block's
// activations is -bias * sum(x) in the fragments' unit.
template <int QT>
__device__ __forceinline__ void zero_point_frag(uint32_t (&A)[4]) {
  const uint32_t z = QT == 4 ? 0x80808080u : 0x82008200u;
  A[0] = z;
  A[1] = z;
  A[2] = z;
  A[3] = z;
}

// One chunk: the pair's 2 tiles x 64 k against the staged activations.
// Per 32-block and column tile, C = -bias * sum(x) (two MMAs with the
// zero-point fragment, shared by both tiles; zero for Q8) starts each
// block's fresh accumulator; the block's two k16 MMAs add sum(u * x); one FMA
// per element (packed in pairs) folds the block scale into the running sum.
template <int QT, int NCT>
__device__ __forceinline__ void compute_chunk(const unsigned char* st, const unsigned char* xs,
                                              int xstride, int j, int lane,
                                              float (&acc)[TPW][NCT][4]) {
  using RC = Rec<QT>;
  const int g = lane >> 2, t = lane & 3;
  uint4 xb[NCT][2];
#pragma unroll
  for (int ct = 0; ct < NCT; ct++) {
    const unsigned char* row = xs + (ct * 8 + g) * xstride + j * 128 + t * 16;
    xb[ct][0] = *reinterpret_cast<const uint4*>(row);
    xb[ct][1] = *reinterpret_cast<const uint4*>(row + 64);
  }
  float zc[NCT][2][4];
  if constexpr (QT != 8) {
    uint32_t Z[4];
    zero_point_frag<QT>(Z);
#pragma unroll
    for (int ct = 0; ct < NCT; ct++)
#pragma unroll
      for (int b = 0; b < 2; b++) {
        mma_16816_zero(zc[ct][b], Z, xb[ct][b].x, xb[ct][b].y);
        mma_16816(zc[ct][b], Z, xb[ct][b].z, xb[ct][b].w);
      }
  }
#pragma unroll
  for (int i = 0; i < TPW; i++) {
    uint4 aw, aw8 = make_uint4(0, 0, 0, 0);
    aw = *reinterpret_cast<const uint4*>(st + RC::QS + i * RC::QS_TILE + lane * (QT == 8 ? 32 : 16));
    if constexpr (QT == 8)
      aw8 = *reinterpret_cast<const uint4*>(st + RC::QS + i * RC::QS_TILE + lane * 32 + 16);
    const uint2 sw = *reinterpret_cast<const uint2*>(st + RC::SC + i * 64 + g * 8);
    uint2 hw = make_uint2(0, 0);
    if constexpr (QT == 6) hw = *reinterpret_cast<const uint2*>(st + RC::QH + i * 256 + lane * 8);
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
      if constexpr (QT == 8) {
        const uint4 q = b == 0 ? aw : aw8;
        dequant8(q.x, A0[0], A0[1]);
        dequant8(q.y, A0[2], A0[3]);
        dequant8(q.z, A1[0], A1[1]);
        dequant8(q.w, A1[2], A1[3]);
      } else {
        dequant_step<QT>(words[2 * b], hA, A0);
        dequant_step<QT>(words[2 * b + 1], hB, A1);
      }
      const float sg = b == 0 ? s0.x : s1.x;   // row g
      const float sg8 = b == 0 ? s0.y : s1.y;  // row g+8
#pragma unroll
      for (int ct = 0; ct < NCT; ct++) {
        float blk[4];
        if constexpr (QT == 8)
          mma_16816_zero(blk, A0, xb[ct][b].x, xb[ct][b].y);
        else
          mma_16816_c(blk, A0, xb[ct][b].x, xb[ct][b].y, zc[ct][b]);
        mma_16816(blk, A1, xb[ct][b].z, xb[ct][b].w);
        // two packed FMAs (each half rounded exactly as fmaf)
        const float2 r01 = __ffma2_rn(make_float2(sg, sg), make_float2(blk[0], blk[1]),
                                      make_float2(acc[i][ct][0], acc[i][ct][1]));
        const float2 r23 = __ffma2_rn(make_float2(sg8, sg8), make_float2(blk[2], blk[3]),
                                      make_float2(acc[i][ct][2], acc[i][ct][3]));
        acc[i][ct][0] = r01.x;
        acc[i][ct][1] = r01.y;
        acc[i][ct][2] = r23.x;
        acc[i][ct][3] = r23.y;
      }
    }
  }
}

__device__ __forceinline__ bool amax_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Global values an epilogue reads, gathered for all of a lane's fragments in
// one batch of loads before any is used (a read-modify-write per element
// would wait a full round trip each).
struct EpiIn {
  float old[4];    // RESID: the rows' current values (rows g, g+8 x 2 columns)
  RowInfo ri[2];   // QKV: the 2 columns' (slot, position)
  float2 cs[2];    // QKV: RoPE (cos, sin) of the tile's pair at each column's position
};

template <int NCT>
__device__ __forceinline__ void epilogue_gather(const LinArgs& a, int T, int ct, int zrow0,
                                                int lane, EpiIn& in) {
  const int g = lane >> 2, t = lane & 3;
  const LinEpi& e = a.epi;
  const int n0 = T * 16 + g, n1 = n0 + 8;
#pragma unroll
  for (int c = 0; c < 2; c++) {
    const int r = zrow0 + ct * 8 + 2 * t + c;
    if (r >= a.R) continue;
    if (e.kind == EPI_RESID) {
      in.old[c] = e.y[(size_t)r * e.ldy + n0];
      in.old[2 + c] = e.y[(size_t)r * e.ldy + n1];
    } else if (e.kind == EPI_QKV) {
      in.ri[c] = e.rows[r];
    }
  }
}

template <int NCT>
__device__ __forceinline__ void epilogue_gather_rope(const LinArgs& a, int T, int lane, EpiIn& in) {
  const LinEpi& e = a.epi;
  const int g = lane >> 2;
  const int per_head = e.hd / 16;
  const int hh = T / per_head, j = T % per_head;
  if (e.rope == nullptr || hh >= e.nq + e.nkv) return;
  const int i0 = 8 * j + g;
#pragma unroll
  for (int c = 0; c < 2; c++) {
    const int rp = in.ri[c].pos < e.max_ctx ? in.ri[c].pos : e.max_ctx - 1;  // invalid rows are flagged
    in.cs[c] = e.rope[(size_t)max(rp, 0) * (e.hd / 2) + i0];
  }
}

// Epilogue for one tile/column-tile fragment of finished sums.
template <int NCT>
__device__ __forceinline__ void epilogue_frag(const LinArgs& a, int T, int ct, int zrow0,
                                              int lane, const float (&v)[4], const EpiIn& in,
                                              float (&bestv)[NCT][2], int (&besti)[NCT][2]) {
  const int g = lane >> 2, t = lane & 3;
  const LinEpi& e = a.epi;
  const int n0 = T * 16 + g, n1 = n0 + 8;
#pragma unroll
  for (int c = 0; c < 2; c++) {
    const int r = zrow0 + ct * 8 + 2 * t + c;
    if (r >= a.R) continue;
    // rows g and g+8, column r; the sums are in the fragments' units of the
    // dequantised values: exact power-of-two scaling
    const float x0 = v[c] * FRAG_UNIT, x1 = v[2 + c] * FRAG_UNIT;
    switch (e.kind) {
      case EPI_STORE:
        e.y[(size_t)r * e.ldy + n0] = x0;
        e.y[(size_t)r * e.ldy + n1] = x1;
        break;
      case EPI_RESID:
        e.y[(size_t)r * e.ldy + n0] = in.old[c] + x0;
        e.y[(size_t)r * e.ldy + n1] = in.old[2 + c] + x1;
        break;
      case EPI_SWIGLU: {
        const float sil = x0 / (1.0f + expf(-x0));
        e.out16[(size_t)r * e.ldo + T * 8 + g] = __float2half_rn(sil * x1);
        break;
      }
      case EPI_QKV: {
        const int per_head = e.hd / 16;
        const int hh = T / per_head, j = T % per_head;
        const int i0 = 8 * j + g, i1 = e.hd / 2 + 8 * j + g;
        const RowInfo ri = in.ri[c];
        float y0 = x0, y1 = x1;
        if (e.rope != nullptr && hh < e.nq + e.nkv) {
          const float2 cs = in.cs[c];
          y0 = fmaf(x0, cs.x, -x1 * cs.y);
          y1 = fmaf(x1, cs.x, x0 * cs.y);
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
        break;
      }
      case EPI_LMHEAD:
        if (e.y != nullptr) {
          e.y[(size_t)r * e.ldy + n0] = x0;
          e.y[(size_t)r * e.ldy + n1] = x1;
        }
        // NaN is an error; for the sampler (row keys requested) so is +-inf
        if (x0 != x0 || x1 != x1 || (e.row_key != nullptr && (isinf(x0) || isinf(x1))))
          atomicOr(e.err, ERR_NONFINITE);
        if (amax_better(x0, n0, bestv[ct][c], besti[ct][c])) {
          bestv[ct][c] = x0;
          besti[ct][c] = n0;
        }
        if (amax_better(x1, n1, bestv[ct][c], besti[ct][c])) {
          bestv[ct][c] = x1;
          besti[ct][c] = n1;
        }
        break;
    }
  }
}

// Register budget: min_blocks<NCT>() CTAs per SM (one column tile: at most
// 80 registers, and the shared memory never holds more than 3 CTAs either).
template <int QT, int NCT, int KW>
__global__ void __launch_bounds__(WARPS * 32, min_blocks<NCT>())
linear_q_kernel(const LinArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  using RC = Rec<QT>;
  constexpr int P = WARPS / KW;  // tile pairs of a CTA; KW warps share each pair's K range
  __shared__ __align__(8) unsigned long long s_bar[WARPS][NS];
  __shared__ __align__(8) unsigned long long s_xbar;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  // column groups are the fastest grid index: the groups that stream the
  // same weights run together and share them through L2
  const int z = blockIdx.x, grp = blockIdx.y, seg = blockIdx.z;
  const int ZG = gridDim.x;
  const int pp = warp % P, ks = warp / P;
  const int pair = grp * P + pp;
  const int tile0 = pair * TPW;
  const int zrow0 = z * 8 * NCT;
  // the CTA's K range (segment seg of S), then this warp's slice ks of KW
  const int c_begin = (int)((long long)seg * a.nch / a.S);
  const int nc = (int)((long long)(seg + 1) * a.nch / a.S) - c_begin;
  const int w_lo = ks * nc / KW;
  const int wn = (ks + 1) * nc / KW - w_lo;
  constexpr int CPS = cps<QT, NCT>();
  constexpr int SB = CPS * RC::BYTES;  // bytes of a full stage
  unsigned char* ring = smem + warp * NS * SB;
  const uint32_t ring_s = smem_addr(ring);
  unsigned char* xs = smem + WARPS * NS * SB;
  const uint32_t bar0 = smem_addr(&s_bar[warp][0]);
  const uint32_t xbar = smem_addr(&s_xbar);

  // ---- the weight ring of this warp: barriers and prologue.  Weights are
  // ---- constant, so this runs before the grid dependency is resolved (with
  // ---- a programmatic launch it overlaps the tail of the previous kernel).
  const bool active = pair < a.n_pairs;
  const uint8_t* src = a.rec + ((size_t)pair * a.nch + c_begin + w_lo) * RC::BYTES;
  if (active && lane == 0) {
    for (int s = 0; s < NS; s++) mbar_init(bar0 + 8 * s, 1);
    mbar_fence_init();
    for (int q = 0; q < NS - 1 && q * CPS < wn; q++) {
      const uint32_t nb = (uint32_t)min(CPS, wn - q * CPS) * RC::BYTES;
      mbar_expect_tx(bar0 + 8 * q, nb);
      bulk_copy_weights(ring_s + q * SB, src + (size_t)q * SB, nb, bar0 + 8 * q);
    }
  }
  // ---- the activation slice (rows zrow0.., chunks c_begin..): zero what no
  // ---- copy writes (rows >= R, a K tail), then one bulk copy per row.
  const int kv = min(nc * 64, a.K - 64 * c_begin);
  const int nrows = max(0, min(8 * NCT, a.R - zrow0));
  for (int rr = warp; rr < 8 * NCT; rr += WARPS) {
    const int from = rr < nrows ? kv * 2 : 0;
    for (int o = from + lane * 16; o < nc * 128; o += 32 * 16)
      *reinterpret_cast<uint4*>(xs + rr * a.xstride + o) = make_uint4(0, 0, 0, 0);
  }
  if (threadIdx.x == 0) {
    mbar_init(xbar, 1);
    mbar_fence_init();
  }
  __syncthreads();  // zero fill of the slice and barrier inits are visible to all
  // The activations, the scratch and the outputs belong to the stream's
  // previous kernels: nothing below may touch global memory other than the
  // weights before they have completed.
  grid_dep_wait();
  if (threadIdx.x == 0) {
    mbar_expect_tx(xbar, (uint32_t)(nrows * kv * 2));
    for (int rr = 0; rr < nrows; rr++)
      bulk_copy(smem_addr(xs + rr * a.xstride), a.x + (size_t)(zrow0 + rr) * a.K + 64 * c_begin,
                (uint32_t)(kv * 2), xbar);
  }
  grid_dep_launch();  // the next kernel may start its own weight prefetch

  float acc[TPW][NCT][4];
#pragma unroll
  for (int i = 0; i < TPW; i++)
#pragma unroll
    for (int ct = 0; ct < NCT; ct++)
#pragma unroll
      for (int e = 0; e < 4; e++) acc[i][ct][e] = 0.0f;

  // every warp waits for the slice (also the idle ones); its budget is the
  // one wait a caller may shorten, to exercise the path below
  bool ok = mbar_wait(xbar, 0, a.first_tries);
  if (active) {
    // stages of CPS consecutive chunks; the loop is unrolled by the ring
    // depth, so stage indices, parities and ring addresses are constants
    const int n_st = (wn + CPS - 1) / CPS;
    int q = 0;
    const uint8_t* nxt = src + (size_t)(NS - 1) * SB;  // next stage to fetch
    for (int q0 = 0; q0 < n_st && ok; q0 += NS) {
      const uint32_t phase = (uint32_t)((q0 / NS) & 1);
#pragma unroll
      for (int u = 0; u < NS; u++) {
        q = q0 + u;
        if (q >= n_st) break;
        ok = mbar_wait(bar0 + 8 * u, phase);
        if (!ok) break;
        if (lane == 0 && q + NS - 1 < n_st) {
          // the stage before this one was consumed in stage q - 1 (every
          // lane passed its closing __syncwarp), so it can be refilled
          const int sn = (u + NS - 1) % NS;
          const uint32_t nb = (uint32_t)min(CPS, wn - (q + NS - 1) * CPS) * RC::BYTES;
          mbar_expect_tx(bar0 + 8 * sn, nb);
          bulk_copy_weights(ring_s + sn * SB, nxt, nb, bar0 + 8 * sn);
        }
        nxt += SB;
#pragma unroll
        for (int h = 0; h < CPS; h++)
          if (q * CPS + h < wn)
            compute_chunk<QT, NCT>(ring + u * SB + h * RC::BYTES, xs, a.xstride,
                                   w_lo + q * CPS + h, lane, acc);
        __syncwarp();
      }
    }
    if (!ok) {
      // a copy never arrived: flag it, then wait (bounded) for this warp's
      // copies still in flight (stages q .. q + NS - 2) before going on
      if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
      for (int qq = q; qq < n_st && qq < q + NS - 1; qq++)
        mbar_wait(bar0 + 8 * (qq % NS), (uint32_t)((qq / NS) & 1));
    }
  } else if (!ok && threadIdx.x == 0) {
    atomicOr(a.err, ERR_TIMEOUT);
  }
  if (!ok && threadIdx.x == 0) mbar_wait(xbar, 0);  // bounded drain of the slice copies

  // ---- the KW slices of a pair: added in slice order through shared
  // ---- memory (the rings are free now); slice 0's warp carries on.
  if constexpr (KW > 1) {
    float4* red = reinterpret_cast<float4*>(smem);
    __syncthreads();
    if (ks > 0 && active) {
#pragma unroll
      for (int i = 0; i < TPW; i++)
#pragma unroll
        for (int ct = 0; ct < NCT; ct++)
          red[((((ks - 1) * P + pp) * TPW + i) * NCT + ct) * 32 + lane] =
              make_float4(acc[i][ct][0], acc[i][ct][1], acc[i][ct][2], acc[i][ct][3]);
    }
    __syncthreads();
    if (ks == 0 && active) {
      for (int k = 1; k < KW; k++) {
#pragma unroll
        for (int i = 0; i < TPW; i++)
#pragma unroll
          for (int ct = 0; ct < NCT; ct++) {
            const float4 v = red[((((k - 1) * P + pp) * TPW + i) * NCT + ct) * 32 + lane];
            acc[i][ct][0] += v.x;
            acc[i][ct][1] += v.y;
            acc[i][ct][2] += v.z;
            acc[i][ct][3] += v.w;
          }
      }
    }
  }
  const bool owner = ks == 0 && active;  // holds the pair's sums from here on

  // ---- K-split: the last CTA of this (column group, tile group) to finish
  // ---- adds the S partial sums in segment order.
  if (a.S > 1) {
    __shared__ int s_last;
    if (owner) {
#pragma unroll
      for (int i = 0; i < TPW; i++) {
        const int T = tile0 + i;
        if (T >= a.n_tiles) continue;
#pragma unroll
        for (int ct = 0; ct < NCT; ct++) {
          const size_t o = ((((size_t)seg * ZG + z) * a.n_tiles + T) * NCT + ct) * 32 + lane;
          reinterpret_cast<float4*>(a.part)[o] =
              make_float4(acc[i][ct][0], acc[i][ct][1], acc[i][ct][2], acc[i][ct][3]);
        }
      }
    }
    // release: the barrier orders every warp's partial stores before thread
    // 0's gpu-scope fence and ticket; acquire: the last CTA's thread 0 fences
    // after its ticket and the barrier passes that on (reads bypass L1)
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const unsigned prev = atomicAdd(&a.tickets[z * a.n_grp + grp], 1u);
      s_last = (prev == (unsigned)(a.S - 1));
      if (s_last) __threadfence();
    }
    __syncthreads();
    if (!s_last) return;
    if (owner) {
      // eight partial loads in flight per lane, over both tiles
      constexpr int SB = 8 / (TPW * NCT);
      const size_t step = (size_t)ZG * a.n_tiles * NCT * 32;  // one segment
      const float4* P0 = reinterpret_cast<const float4*>(a.part) +
                         ((size_t)z * a.n_tiles * NCT) * 32 + lane;
      const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
      float4 sum[TPW][NCT];
#pragma unroll
      for (int i = 0; i < TPW; i++)
#pragma unroll
        for (int ct = 0; ct < NCT; ct++)
          sum[i][ct] = tile0 + i < a.n_tiles ? __ldcg(P0 + ((size_t)(tile0 + i) * NCT + ct) * 32)
                                             : zero4;
      for (int s0 = 1; s0 < a.S; s0 += SB) {
        float4 v[SB][TPW][NCT];
#pragma unroll
        for (int u = 0; u < SB; u++)
#pragma unroll
          for (int i = 0; i < TPW; i++)
#pragma unroll
            for (int ct = 0; ct < NCT; ct++)
              v[u][i][ct] = (s0 + u < a.S && tile0 + i < a.n_tiles)
                                ? __ldcg(P0 + (size_t)(s0 + u) * step +
                                         ((size_t)(tile0 + i) * NCT + ct) * 32)
                                : zero4;
#pragma unroll
        for (int u = 0; u < SB; u++)
          if (s0 + u < a.S) {
#pragma unroll
            for (int i = 0; i < TPW; i++)
#pragma unroll
              for (int ct = 0; ct < NCT; ct++) {
                sum[i][ct].x += v[u][i][ct].x;
                sum[i][ct].y += v[u][i][ct].y;
                sum[i][ct].z += v[u][i][ct].z;
                sum[i][ct].w += v[u][i][ct].w;
              }
          }
      }
#pragma unroll
      for (int i = 0; i < TPW; i++)
#pragma unroll
        for (int ct = 0; ct < NCT; ct++) {
          acc[i][ct][0] = sum[i][ct].x;
          acc[i][ct][1] = sum[i][ct].y;
          acc[i][ct][2] = sum[i][ct].z;
          acc[i][ct][3] = sum[i][ct].w;
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
    for (int c = 0; c < 2; c++) {
      bestv[ct][c] = -INFINITY;
      besti[ct][c] = 0x7fffffff;
    }
  if (owner) {
    EpiIn in[TPW][NCT];
    if (a.epi.kind == EPI_RESID || a.epi.kind == EPI_QKV) {
#pragma unroll
      for (int i = 0; i < TPW; i++)
#pragma unroll
        for (int ct = 0; ct < NCT; ct++)
          if (tile0 + i < a.n_tiles) epilogue_gather<NCT>(a, tile0 + i, ct, zrow0, lane, in[i][ct]);
      if (a.epi.kind == EPI_QKV) {
#pragma unroll
        for (int i = 0; i < TPW; i++)
#pragma unroll
          for (int ct = 0; ct < NCT; ct++)
            if (tile0 + i < a.n_tiles) epilogue_gather_rope<NCT>(a, tile0 + i, lane, in[i][ct]);
      }
    }
#pragma unroll
    for (int i = 0; i < TPW; i++) {
      const int T = tile0 + i;
      if (T >= a.n_tiles) continue;
#pragma unroll
      for (int ct = 0; ct < NCT; ct++)
        epilogue_frag<NCT>(a, T, ct, zrow0, lane, acc[i][ct], in[i][ct], bestv, besti);
    }
  }
  if (a.epi.kind != EPI_LMHEAD) return;

  // ---- fused argmax: warp (over the 8 row lanes g) -> CTA -> grid.
  __shared__ float s_v[WARPS][16];
  __shared__ int s_i[WARPS][16];
  __shared__ int s_last_am;
#pragma unroll
  for (int ct = 0; ct < NCT; ct++)
#pragma unroll
    for (int c = 0; c < 2; c++) {
      float v = bestv[ct][c];
      int id = besti[ct][c];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, off);
        const int oi = __shfl_xor_sync(0xffffffffu, id, off);
        if (amax_better(ov, oi, v, id)) {
          v = ov;
          id = oi;
        }
      }
      if (g == 0) {
        s_v[warp][ct * 8 + 2 * t + c] = v;
        s_i[warp][ct * 8 + 2 * t + c] = id;
      }
    }
  __syncthreads();
  if (threadIdx.x < 8 * NCT) {
    const int col = threadIdx.x;
    float v = s_v[0][col];
    int id = s_i[0][col];
    for (int w = 1; w < WARPS; w++)
      if (amax_better(s_v[w][col], s_i[w][col], v, id)) {
        v = s_v[w][col];
        id = s_i[w][col];
      }
    a.amax_part[((size_t)z * a.n_grp + grp) * 16 + col] = make_float2(v, __int_as_float(id));
  }
  // release / acquire as for the K split: one fence by thread 0 each side
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(&a.tickets[ZG * a.n_grp + z], 1u);
    s_last_am = (prev == (unsigned)(a.n_grp - 1));
    if (s_last_am) __threadfence();
  }
  __syncthreads();
  if (!s_last_am) return;
  // the grid's argmax of each column: one warp per column, eight group
  // partials in flight per lane (the result is the unique (max, lowest
  // index) pair, whatever the order)
  for (int col = warp; col < 8 * NCT; col += WARPS) {
    float v = -INFINITY;
    int id = 0x7fffffff;
    const float2* base = a.amax_part + (size_t)z * a.n_grp * 16 + col;
    for (int g0 = 0; g0 < a.n_grp; g0 += 32 * 8) {
      float2 p[8];
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const int gi = g0 + u * 32 + lane;
        p[u] = gi < a.n_grp ? __ldcg(base + (size_t)gi * 16)
                            : make_float2(-INFINITY, __int_as_float(0x7fffffff));
      }
#pragma unroll
      for (int u = 0; u < 8; u++) {
        const int pi = __float_as_int(p[u].y);
        if (amax_better(p[u].x, pi, v, id)) {
          v = p[u].x;
          id = pi;
        }
      }
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, off);
      const int oi = __shfl_xor_sync(0xffffffffu, id, off);
      if (amax_better(ov, oi, v, id)) {
        v = ov;
        id = oi;
      }
    }
    const int r = zrow0 + col;
    if (lane == 0 && r < a.R && a.epi.argmax != nullptr) a.epi.argmax[r] = id == 0x7fffffff ? 0 : id;
    if (lane == 0 && r < a.R && a.epi.row_key != nullptr) write_row_key(a.epi, r, logit_key(v));
  }
  if (threadIdx.x == 0) a.tickets[ZG * a.n_grp + z] = 0u;
}

using LinKernel = void (*)(LinArgs);
LinKernel kernel_for(int qtype, int nct, int kw) {
#define SPEC_LIN_K(QT_, NCT_, KW_) \
  if (qtype == QT_ && nct == NCT_ && kw == KW_) return linear_q_kernel<QT_, NCT_, KW_>;
  SPEC_LIN_K(4, 1, 1) SPEC_LIN_K(4, 1, 2) SPEC_LIN_K(4, 1, 4) SPEC_LIN_K(4, 1, 8)
  SPEC_LIN_K(4, 2, 1) SPEC_LIN_K(4, 2, 2) SPEC_LIN_K(4, 2, 4) SPEC_LIN_K(4, 2, 8)
  SPEC_LIN_K(6, 1, 1) SPEC_LIN_K(6, 1, 2) SPEC_LIN_K(6, 1, 4) SPEC_LIN_K(6, 1, 8)
  SPEC_LIN_K(6, 2, 1) SPEC_LIN_K(6, 2, 2) SPEC_LIN_K(6, 2, 4) SPEC_LIN_K(6, 2, 8)
  SPEC_LIN_K(8, 1, 1) SPEC_LIN_K(8, 1, 2) SPEC_LIN_K(8, 1, 4) SPEC_LIN_K(8, 1, 8)
  SPEC_LIN_K(8, 2, 1) SPEC_LIN_K(8, 2, 2) SPEC_LIN_K(8, 2, 4) SPEC_LIN_K(8, 2, 8)
#undef SPEC_LIN_K
  return nullptr;
}

struct LinCfg {
  int kw, S;
};

// Latency model of one launch, fitted (least squares over CTA-timeline spans
// of 7 shapes x 5-9 splits each, GB300, rms error ~5-6%) for the nt <= 8
// (one column tile) and nt = 9..16 (two column tiles) kernels: an SM
// retires chunks at min(SM rate, resident warps x warp rate), a launch costs
// a fixed start-up, a K split adds a ticket and the last CTA's partial loads,
// KW > 1 the shared-memory slice sum, and each further wave a start-up.
// The Q8 rates are not fitted: an SM's rate is its share of the copy
// bandwidth in 2176-byte chunks, a warp's that of Q4 (about as many
// instructions per chunk).
struct LinModel {
  double sm_rate[3], warp_rate[3];  // chunks / us (Q4, Q6, Q8)
  double t_start, t_split, t_batch, t_slices, t_wave;  // us
};
constexpr LinModel MODEL_NCT[2] = {
    {{32.4, 26.0, 20.0}, {3.55, 2.82, 3.4}, 2.46, 1.59, 0.70, 0.56, 3.08},
    {{23.9, 20.9, 18.0}, {2.37, 2.10, 2.3}, 4.71, 1.66, 0.66, 0.0, 3.28},
};

double model_time(const LinModel& M, int qtype, int nct, int kw, int S, int n_pairs, int nch,
                  int sms) {
  const int P = WARPS / kw;
  const int n_grp = (n_pairs + P - 1) / P;
  const int nc = (nch + S - 1) / S;
  const int wn = (nc + kw - 1) / kw;  // chunks of the busiest warp
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel_for(qtype, nct, kw), WARPS * 32,
                                                smem_bytes(qtype, nct, nc));
  cudaGetLastError();
  per_sm = std::max(per_sm, 1);
  const int q = qtype == 4 ? 0 : (qtype == 6 ? 1 : 2);
  const double ctas = (double)n_grp * S;
  const double load = std::ceil(ctas / sms);  // CTAs of the busiest SM
  const double resident = std::min((double)per_sm, load);
  const double rate = std::min(M.sm_rate[q], WARPS * resident * M.warp_rate[q]);
  const double waves = std::ceil(ctas / ((double)sms * per_sm));
  double t = load * WARPS * wn / rate + M.t_start + (waves - 1) * M.t_wave;
  if (S > 1) t += M.t_split + M.t_batch * std::ceil((S - 1) / 4.0);
  if (kw > 1) t += M.t_slices;
  return t;
}

// (KW, S) of a matrix: fixed by its shape and the device only (never by nt,
// so rows stay bitwise nt-invariant); the one minimising the modelled
// latency of an nt <= 8 launch plus that of an nt = 9..16 launch.
LinCfg choose_config(int qtype, int n_pairs, int nch, int sms) {
  sms = std::max(sms, 1);
  const int s_min = std::max(1, (nch + NC_CTA_MAX - 1) / NC_CTA_MAX);
  const int s_max = std::max(s_min, std::min(MAX_SPLIT, nch));
  LinCfg best{1, s_min};
  double best_t = 1e30;
  for (int kw : {1, 2, 4, 8})
    for (int S = s_min; S <= s_max; S++) {
      const double t = model_time(MODEL_NCT[0], qtype, 1, kw, S, n_pairs, nch, sms) +
                       model_time(MODEL_NCT[1], qtype, 2, kw, S, n_pairs, nch, sms);
      if (t < best_t - 1e-6) {
        best_t = t;
        best = LinCfg{kw, S};
      }
    }
  return best;
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
int qmat_pack(const spec_qweight* w, PermKind perm, int head_dim, int sms, cudaStream_t st,
              QMat* out) {
  if (w == nullptr || out == nullptr) return fail(SPEC_E_INVALID, "null qweight");
  if (w->qtype != SPEC_Q4 && w->qtype != SPEC_Q6 && w->qtype != SPEC_Q8)
    return fail(SPEC_E_UNSUPPORTED, "qtype must be SPEC_Q4, SPEC_Q6 or SPEC_Q8");
  if (w->N <= 0 || w->K <= 0 || w->N % 16 != 0 || w->K % 32 != 0)
    return fail(SPEC_E_SHAPE, "need N % 16 == 0 and K % 32 == 0");
  if (w->K > 64 * NC_CTA_MAX * MAX_SPLIT) return fail(SPEC_E_SHAPE, "K above 262144 is not supported");
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
  q.n_pairs = (q.n_tiles + TPW - 1) / TPW;
  q.rec_bytes = rec_bytes(q.qtype);
  LinCfg cfg = choose_config(q.qtype, q.n_pairs, q.nch, sms);
  if (const char* e = std::getenv("SPEC_VERIFY_LINEAR_SPLIT")) {
    // Overrides the choice (for tests and tuning): comma-separated entries,
    // "KW:S" for every matrix or "N:K:KW:S" for the N x K ones (the last
    // matching entry wins); invalid entries are ignored.
    std::string list(e);
    size_t at = 0;
    while (at <= list.size()) {
      const size_t end = std::min(list.find(',', at), list.size());
      const std::string item = list.substr(at, end - at);
      at = end + 1;
      int v[4] = {0, 0, 0, 0};
      const int n = std::sscanf(item.c_str(), "%d:%d:%d:%d", &v[0], &v[1], &v[2], &v[3]);
      int kw = 0, S = 0;
      if (n == 2) {
        kw = v[0];
        S = v[1];
      } else if (n == 4 && v[0] == q.N && v[1] == q.K) {
        kw = v[2];
        S = v[3];
      } else {
        continue;
      }
      if ((kw == 1 || kw == 2 || kw == 4 || kw == 8) && S >= 1 &&
          S <= std::min(MAX_SPLIT, q.nch) && (q.nch + S - 1) / S <= NC_CTA_MAX)
        cfg = LinCfg{kw, S};
    }
  }
  q.kw = cfg.kw;
  q.S = cfg.S;
  q.tc_H = tc_choose_halves(q.N, q.nch, sms);
  q.tc_P = tc_choose_ctas(q.N, q.nch, sms, q.tc_H);
  q.n_grp = (q.n_pairs + WARPS / q.kw - 1) / (WARPS / q.kw);
  q.nc_cta = (q.nch + q.S - 1) / q.S;
  const size_t units = (size_t)q.n_pairs * q.nch;
  q.bytes = units * q.rec_bytes;
  if (cudaMalloc(&q.base, q.bytes) != cudaSuccess) {
    cudaGetLastError();
    return fail(SPEC_E_OOM, "cudaMalloc of packed weights failed");
  }
  q.rec = reinterpret_cast<uint8_t*>(q.base);
  const size_t total = units * TPW * 32;
  const int threads = 256;
  pack_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, st>>>(
      q.qtype, (const uint8_t*)w->qs, (const uint8_t*)w->qh, (const uint16_t*)w->scales, q.N,
      q.K, q.nch, q.n_pairs, perm, head_dim, q.rec_bytes, q.rec);
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

size_t lin_part_floats(const QMat& w, int R) {
  return w.S > 1 ? (size_t)w.S * col_groups(R) * w.n_tiles * col_tiles(R) * 32 * 4 : 0;
}
size_t lin_tickets_needed(const QMat& w, int R) {
  return (size_t)col_groups(R) * w.n_grp + col_groups(R);  // K-split + argmax tickets
}
size_t lin_amax_entries(const QMat& w, int R) { return (size_t)col_groups(R) * w.n_grp * 16; }

int linear_launch(const QMat& w, const __half* x, int R, const LinEpi& epi,
                  const LinScratch& scr, cudaStream_t st) {
  if (R < 1) return fail(SPEC_E_SHAPE, "linear: R must be >= 1");
  if (scr.err == nullptr) return fail(SPEC_E_INVALID, "linear: no error word");
  if (lin_part_floats(w, R) > scr.part_floats || lin_tickets_needed(w, R) > scr.n_tickets ||
      (epi.kind == EPI_LMHEAD && lin_amax_entries(w, R) > scr.amax_entries))
    return fail(SPEC_E_SHAPE, "linear: scratch too small for this R");
  LinArgs a;
  a.rec = w.rec;
  a.x = x;
  a.N = w.N;
  a.K = w.K;
  a.nch = w.nch;
  a.n_tiles = w.n_tiles;
  a.n_pairs = w.n_pairs;
  a.n_grp = w.n_grp;
  a.S = w.S;
  a.R = R;
  a.epi = epi;
  a.part = scr.part;
  a.tickets = scr.tickets;
  a.amax_part = scr.amax_part;
  a.err = scr.err;
  a.first_tries = scr.wait_tries;
  a.xstride = x_stride(w.nc_cta);
  const int ZG = col_groups(R);
  const int nct = col_tiles(R);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ZG, w.n_grp, w.S);
  cfg.blockDim = dim3(WARPS * 32);
  cfg.dynamicSmemBytes = smem_bytes(w.qtype, nct, w.nc_cta);
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = programmatic_launch() ? 1 : 0;
  const LinKernel k = kernel_for(w.qtype, nct, w.kw);
  if (k == nullptr) return fail(SPEC_E_INVALID, "linear: no kernel for this configuration");
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k, a);
  if (e != cudaSuccess) return fail(SPEC_E_CUDA, std::string("linear launch: ") + cudaGetErrorString(e));
  return SPEC_OK;
}

void linear_init_attrs() {
  for (int qt : {4, 6, 8})
    for (int nct : {1, 2})
      for (int kw : {1, 2, 4, 8})
        cudaFuncSetAttribute(kernel_for(qt, nct, kw), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes(qt, nct, NC_CTA_MAX));
}
