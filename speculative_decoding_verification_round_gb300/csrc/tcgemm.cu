// tcgemm.cu -- the verify GEMM of multi-sequence rounds on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// "Speculative Decoding (D5-R) -- Plan", section 1: the batched verify is one
// weights-once pass.  With many sequences in a round (the batched workload:
// 12 sequences x 16 rows = 192 rows) the pass is no longer bound by the
// weight stream but by the contraction itself (2 x 192 flops per weight), so
// it runs on tcgen05.mma with the activation rows as the N dimension:
//
//   * a CTA's work is a run of (tile, 64-k chunk) units: a tile is 128 or
//     256 weight rows (4 or 8 pairs of the packed streaming layout) as one
//     or two 128-row halves, each with its own 128 x Npad fp32 accumulator
//     in tensor memory (one TMEM lane per weight row; Npad = the rows
//     rounded up to 16).  The cut is fixed per matrix: one run per tile, a
//     K split (S aligned segments a tile), or one run per SM over all units
//     (a run may end one tile and start the next).  Two halves share each
//     activation tile and chunk handshake (twice the MMAs per chunk);
//   * warp 0 streams the packed weight records into a shared-memory ring with
//     TMA bulk copies (L2 policy evict first: each weight is read once);
//     warp 1 loads the activation tile of each 64-k chunk with a 2-D TMA
//     tensor copy (128-byte swizzle, rows past R read as zero);
//   * warps 3-18 dequantise each chunk into TWO fp16 A tiles per half in the
//     UMMA K-major 128-byte-swizzle layout, hi = fp16(q * scale) and lo =
//     fp16(q * scale - hi): q * scale has at most 11 + 8 significant bits,
//     so lo holds the rest exactly and hi + lo IS the weight -- every
//     product the tensor core forms is exact, as in the oracle;
//   * one thread of warp 2 issues sixteen tcgen05.mma (M 128, N Npad, K 16:
//     hi and lo of each half for each 16-k step) per chunk and commits them
//     to the stages' "empty" barriers;
//   * after the last chunk the same sixteen warps read the accumulators back
//     (tcgen05.ld), add the pieces of a tile cut across CTAs in k order
//     (partials in L2; the CTAs that wait on others are one cooperative
//     launch) and run the fused epilogue (store, residual add, SwiGLU, RoPE
//     + KV write, LM head logits + argmax).
// Each output element is the same sequence of fp32 additions (chunk by chunk
// into an accumulator, then the pieces of its tile in k order) whatever the
// other rows of the batch, so a row's result is the same in every batch
// this kernel runs.
//
// Every wait is bounded (mbarrier try_wait with a suspend hint, about a
// second in all; the pieces' meeting counter, a tenth of a second); one that
// gives up sets ERR_TIMEOUT and the CTA stops issuing work, waits (bounded)
// for what it issued and frees its tensor memory before it returns.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <string>

#include "common.cuh"
#include "tc_ops.cuh"

namespace {

constexpr int TC_DQ_WARPS = 16;     // dequant (then epilogue) warps
constexpr int TC_THREADS = (3 + TC_DQ_WARPS) * 32;  // 19 warps
constexpr int TC_EPI_WARP0 = 3;     // warps 3..18: dequant, then epilogue
constexpr int TC_EPI_THREADS = TC_DQ_WARPS * 32;   // four warps per TMEM lane quadrant
constexpr int EW = 8;               // epilogue columns per TMEM load
constexpr int TC_A_BYTES = TC_M * 128;  // one 64-k chunk of 128 rows, fp16 (one of hi / lo)
constexpr int TC_A_HALF = 2 * TC_A_BYTES;  // hi and lo tiles of one half
constexpr int TC_MAX_A = 3;     // A stages (two with two halves)
constexpr int TC_MAX_ST = 6;    // stages of the activation ring
constexpr int TC_MAX_RAW = 8;
constexpr int TC_MAX_R = 192;   // activation rows of one launch (Npad <= 192)

template <int QT>
struct TcRec {  // the packed record of one (pair, 64-k chunk): see linear.cu
  static constexpr int QS_TILE = QT == 8 ? 1024 : 512;
  static constexpr int SC = 2 * QS_TILE;
  static constexpr int QH = SC + 128;
  static constexpr int BYTES = QH + (QT == 6 ? 512 : 0);
};

struct TcArgs {
  const uint8_t* rec;  // [n_pairs][nch][rec]
  int N, K, nch, n_pairs, n_mt, P, R, Npad, tmem_cols;  // P: CTAs (runs of work)
  int halves;           // 128-row halves (accumulators) of a CTA: 1 or 2
  int acc_stride;       // TMEM columns between the two accumulators
  int a_stages, b_stages, raw_depth;  // ring depths: A tiles, activations, raw records
  LinEpi epi;
  float* part;          // [P][Npad][256] a CTA's partial of a shared tile's piece
  unsigned* tickets;    // [n_mt] K-split arrivals, [n_mt] departures, [1] argmax ticket
  unsigned long long* amax_key;  // [Npad] LM head: packed (value, index) maxima
  uint32_t* err;
  int wait_tries;
};

// The integers of one k16 step's word for rows g and g+8 (4 + 4 values) as
// exact fp16: each u is placed in the low bits of a half, made 1024 + u by
// the fp16 exponent of 1024, then (1024 + u) - (1024 + bias) = q exactly.
// [0]/[1]: k pairs (0,1) and (2,3) of each row.
template <int QT>
__device__ __forceinline__ void dq_word(uint32_t w, uint32_t hx, __half2 (&rg)[2],
                                        __half2 (&rg8)[2]) {
  constexpr uint32_t MAGIC = 0x64006400u;
  const __half2 off = QT == 4 ? __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408))
                              : __halves2half2(__ushort_as_half(0x6420), __ushort_as_half(0x6420));
  uint32_t u[4];
  if constexpr (QT == 4) {
    u[0] = (w & 0x000F000Fu) | MAGIC;          // row g,   k 0,1
    u[1] = ((w >> 8) & 0x000F000Fu) | MAGIC;   // row g,   k 2,3
    u[2] = ((w >> 4) & 0x000F000Fu) | MAGIC;   // row g+8, k 0,1
    u[3] = ((w >> 12) & 0x000F000Fu) | MAGIC;  // row g+8, k 2,3
  } else {
    const uint32_t w8 = w >> 8, hx2 = hx >> 2;
    u[0] = (w & 0x000F000Fu) | (hx & 0x00300030u) | MAGIC;
    u[1] = (w8 & 0x000F000Fu) | (hx2 & 0x00300030u) | MAGIC;
    u[2] = ((w >> 4) & 0x000F000Fu) | ((hx >> 4) & 0x00300030u) | MAGIC;
    u[3] = ((w8 >> 4) & 0x000F000Fu) | ((hx2 >> 4) & 0x00300030u) | MAGIC;
  }
  rg[0] = __hsub2(*reinterpret_cast<const __half2*>(&u[0]), off);
  rg[1] = __hsub2(*reinterpret_cast<const __half2*>(&u[1]), off);
  rg8[0] = __hsub2(*reinterpret_cast<const __half2*>(&u[2]), off);
  rg8[1] = __hsub2(*reinterpret_cast<const __half2*>(&u[3]), off);
}

// Q8: one word holds u = q + 128 of rows r, r, r', r' at k, k+1.
__device__ __forceinline__ void dq_word8(uint32_t w, __half2& rg, __half2& rg8) {
  const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  const uint32_t a = __byte_perm(w, 0x64646464u, 0x4140);
  const uint32_t b = __byte_perm(w, 0x64646464u, 0x4342);
  rg = __hsub2(*reinterpret_cast<const __half2*>(&a), off);
  rg8 = __hsub2(*reinterpret_cast<const __half2*>(&b), off);
}

// w = q * s as an exact pair: hi = fp16(q * s), lo = fp16(q * s - hi).  q is
// an integer of at most 8 bits and s has 11, so q * s has at most 19
// significant bits and a multiple of s's last place; hi takes the leading
// 11 (rounded), and the remainder q * s - hi has at most 8 and is a multiple
// of 2^-24 or coarser: the fused multiply-add rounds nothing.
__device__ __forceinline__ void split2(__half2 q, __half2 s, __half2& hi, __half2& lo) {
  hi = __hmul2(q, s);
  lo = __hfma2(q, s, __hneg2(hi));
}

__device__ __forceinline__ uint4 pack4(__half2 a, __half2 b, __half2 c, __half2 d) {
  return make_uint4(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b),
                    *reinterpret_cast<const uint32_t*>(&c), *reinterpret_cast<const uint32_t*>(&d));
}

// Order-preserving key of a logit (-0 taken as +0, so that the two zeros
// tie and the lower id wins, as in the other argmax paths).
__device__ __forceinline__ uint32_t f32_key(float f) { return logit_key(f); }

// Bounded wait until the counter at p reaches target (acquire).
constexpr int TC_MEET_TRIES = 1 << 20;
__device__ __forceinline__ bool wait_count(const unsigned* p, unsigned target) {
  for (int i = 0; i < TC_MEET_TRIES; i++) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    __nanosleep(64);
  }
  return false;
}
__device__ __forceinline__ void epi_bar() {  // the dequant / epilogue warps
  asm volatile("bar.sync 1, %0;" ::"r"(TC_EPI_THREADS) : "memory");
}

// The dequant of one 64-k chunk of one 16-row tile i of a pair by one lane:
// lane unit (g, t) holds rows g and g+8 of each tile at k = 32b + 8t .. +7.
// The lane -> (g, t) map makes both the record loads and the swizzled
// stores of every 8-lane phase hit 8 distinct bank groups.  Each weight goes
// to the hi tile and its exact remainder to the lo tile.
template <int QT>
__device__ __forceinline__ void dequant_tile(const unsigned char* raw, unsigned char* ahi,
                                             unsigned char* alo, int pair_in_cta, int i, int lane,
                                             int b_lo, int b_hi) {
  using RC = TcRec<QT>;
  const int ph = lane >> 3, j = lane & 7;
  const int p = j & 1, t0 = (j >> 1) & 1, t1 = j >> 2;
  const int g = 4 * (p ^ (ph >> 1)) + 2 * (t0 ^ (ph & 1)) + p, t = 2 * t1 + t0;
  const int l = 4 * g + t;  // the record's lane index of this unit
  {
    const uint2 sw = *reinterpret_cast<const uint2*>(raw + RC::SC + i * 64 + g * 8);
    const __half2 s0 = *reinterpret_cast<const __half2*>(&sw.x);  // (row g, row g+8), block 0
    const __half2 s1 = *reinterpret_cast<const __half2*>(&sw.y);  // block 1
    const int r0 = 32 * pair_in_cta + 16 * i + g;                 // A-tile row of row g
#pragma unroll
    for (int b = 0; b < 2; b++) {
      if (b < b_lo || b >= b_hi) continue;
      const __half2 sg = b == 0 ? __low2half2(s0) : __low2half2(s1);
      const __half2 sg8 = b == 0 ? __high2half2(s0) : __high2half2(s1);
      __half2 qg[4], qg8[4];  // exact integers, k pairs (0,1) .. (6,7)
      if constexpr (QT == 8) {
        const uint4 q = *reinterpret_cast<const uint4*>(raw + i * RC::QS_TILE + l * 32 + b * 16);
        dq_word8(q.x, qg[0], qg8[0]);
        dq_word8(q.y, qg[1], qg8[1]);
        dq_word8(q.z, qg[2], qg8[2]);
        dq_word8(q.w, qg[3], qg8[3]);
      } else {
        const uint4 q = *reinterpret_cast<const uint4*>(raw + i * RC::QS_TILE + l * 16);
        uint32_t hA = 0, hB = 0;
        if constexpr (QT == 6) {
          const uint2 hw = *reinterpret_cast<const uint2*>(raw + RC::QH + i * 256 + l * 8);
          hA = b == 0 ? hw.x : hw.y;
          hB = __funnelshift_l(hA, hA, 8);
        }
        const uint32_t w0 = b == 0 ? q.x : q.z, w1 = b == 0 ? q.y : q.w;
        __half2 a0[2], c0[2], a1[2], c1[2];
        dq_word<QT>(w0, hA, a0, c0);  // k 0..3
        dq_word<QT>(w1, hB, a1, c1);  // k 4..7
        qg[0] = a0[0]; qg[1] = a0[1]; qg[2] = a1[0]; qg[3] = a1[1];
        qg8[0] = c0[0]; qg8[1] = c0[1]; qg8[2] = c1[0]; qg8[3] = c1[1];
      }
      __half2 hg[4], lg[4], hg8[4], lg8[4];
#pragma unroll
      for (int e = 0; e < 4; e++) {
        split2(qg[e], sg, hg[e], lg[e]);
        split2(qg8[e], sg8, hg8[e], lg8[e]);
      }
      const int u = 4 * b + t;
      const uint32_t og = sw128_off(r0, u), og8 = sw128_off(r0 + 8, u);
      *reinterpret_cast<uint4*>(ahi + og) = pack4(hg[0], hg[1], hg[2], hg[3]);
      *reinterpret_cast<uint4*>(ahi + og8) = pack4(hg8[0], hg8[1], hg8[2], hg8[3]);
      *reinterpret_cast<uint4*>(alo + og) = pack4(lg[0], lg[1], lg[2], lg[3]);
      *reinterpret_cast<uint4*>(alo + og8) = pack4(lg8[0], lg8[1], lg8[2], lg8[3]);
    }
  }
}

// Epilogue of EW finished columns (activation rows col0..col0+EW-1) of this
// thread's weight row n: v[c] is the sum for row col0 + c.
__device__ __forceinline__ void tc_epilogue(const TcArgs& a, int n, int col0, const float (&v)[EW],
                                              int lane, uint32_t* s_key, int slot) {
  const LinEpi& e = a.epi;
  const bool real = n < a.N;
  switch (e.kind) {
    case EPI_STORE:
#pragma unroll
      for (int c = 0; c < EW; c++)
        if (real && col0 + c < a.R) e.y[(size_t)(col0 + c) * e.ldy + n] = v[c];
      break;
    case EPI_RESID: {
      // the EW old values in one batch of loads, then the stores
      float old[EW];
#pragma unroll
      for (int c = 0; c < EW; c++)
        old[c] = real && col0 + c < a.R ? e.y[(size_t)(col0 + c) * e.ldy + n] : 0.0f;
#pragma unroll
      for (int c = 0; c < EW; c++)
        if (real && col0 + c < a.R) e.y[(size_t)(col0 + c) * e.ldy + n] = old[c] + v[c];
      break;
    }
    case EPI_SWIGLU: {
      // rows g (gate j) and g+8 (up j) of each 16-row tile are lanes l, l+8
      const int g = n & 15, T = n >> 4;
#pragma unroll
      for (int c = 0; c < EW; c++) {
        const float up = __shfl_xor_sync(0xffffffffu, v[c], 8);
        const int r = col0 + c;
        if (g < 8 && real && r < a.R) {
          const float x0 = v[c];
          const float sil = x0 / (1.0f + expf(-x0));
          e.out16[(size_t)r * e.ldo + T * 8 + g] = __float2half_rn(sil * up);
        }
      }
      break;
    }
    case EPI_QKV: {
      const int g = n & 15, T = n >> 4;
      const int per_head = e.hd / 16;
      const int hh = T / per_head, jj = T % per_head;
      const int i0 = 8 * jj + (g & 7), i1 = e.hd / 2 + 8 * jj + (g & 7);
      const bool rope = e.rope != nullptr && hh < e.nq + e.nkv;
      // the columns' (slot, position) records and RoPE factors in one batch
      // of loads before any is used
      RowInfo ri_c[EW];
      float2 cs_c[EW];
#pragma unroll
      for (int c = 0; c < EW; c++) {
        const int r = min(col0 + c, a.R - 1);
        ri_c[c] = e.rows[r];
      }
#pragma unroll
      for (int c = 0; c < EW; c++) {
        const int rp = ri_c[c].pos < e.max_ctx ? ri_c[c].pos : e.max_ctx - 1;
        cs_c[c] = rope ? e.rope[(size_t)max(rp, 0) * (e.hd / 2) + i0] : make_float2(1.0f, 0.0f);
      }
#pragma unroll
      for (int c = 0; c < EW; c++) {
        const float x1 = __shfl_xor_sync(0xffffffffu, v[c], 8);
        const int r = col0 + c;
        if (g >= 8 || !real || r >= a.R) continue;
        const float x0 = v[c];
        const RowInfo ri = ri_c[c];
        float y0 = x0, y1 = x1;
        if (rope) {
          const float2 cs = cs_c[c];
          y0 = fmaf(x0, cs.x, -x1 * cs.y);
          y1 = fmaf(x1, cs.x, x0 * cs.y);
        }
        __half* dst;
        if (hh < e.nq) {
          dst = e.out16 + ((size_t)r * e.nq + hh) * e.hd;
        } else {
          const bool isk = hh < e.nq + e.nkv;
          const int kvh = isk ? hh - e.nq : hh - e.nq - e.nkv;
          if (ri.pos >= e.max_ctx) continue;  // flagged by the embedding kernel
          dst = (isk ? e.kcache : e.vcache) + (((size_t)ri.slot * e.nkv + kvh) * e.max_ctx + ri.pos) * e.hd;
        }
        dst[i0] = __float2half_rn(y0);
        dst[i1] = __float2half_rn(y1);
      }
      break;
    }
    case EPI_LMHEAD: {
      // the CTA's best (value, lowest id) of each column: a warp reduction
      // of order-preserving keys, then the eight warps through shared memory
      bool bad = false;
#pragma unroll
      for (int c = 0; c < EW; c++) {
        const int r = col0 + c;
        if (r >= a.R) continue;  // uniform across the warp
        if (e.y != nullptr && real) e.y[(size_t)r * e.ldy + n] = v[c];
        // NaN is an error; for the sampler (row keys requested) so is +-inf
        bad |= real && (v[c] != v[c] || (e.row_key != nullptr && isinf(v[c])));
        const uint32_t key = real ? f32_key(v[c]) : 0u;
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
        const uint32_t id = key == kmax && real ? (uint32_t)n : 0xffffffffu;
        const uint32_t imin = __reduce_min_sync(0xffffffffu, id);
        if (lane == 0) {
          s_key[(slot * 2) * TC_MAX_R + r] = kmax;
          s_key[(slot * 2 + 1) * TC_MAX_R + r] = imin;
        }
      }
      if (bad) atomicOr(e.err, ERR_NONFINITE);
      break;
    }
  }
}

// RUNS: the cut may give a CTA two pieces (one run per SM); without it every
// CTA has one piece (one run per tile, or a K split) and the main loops are
// those of a single tile.
template <int QT, bool RUNS>
__global__ void __launch_bounds__(TC_THREADS, 1)
tc_linear_kernel(const __grid_constant__ CUtensorMap tmx, const TcArgs a) {
  using RC = TcRec<QT>;
  extern __shared__ unsigned char smem_dyn[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) unsigned long long s_bar[2 * TC_MAX_A + 2 * TC_MAX_ST + 2 * TC_MAX_RAW + 3];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.halves, STA = a.a_stages, STB = a.b_stages, RAWN = a.raw_depth;
  const int CTA_ROWS = TC_M * H, CTA_PAIRS = 4 * H, A_STAGE = H * TC_A_HALF;
  const int B_BYTES = a.Npad * 128;
  unsigned char* A0 = smem;  // [STA][half][hi, lo] tiles
  unsigned char* B0 = smem + STA * A_STAGE;
  unsigned char* RAW0 = B0 + STB * B_BYTES;
  const int RAW_BYTES = CTA_PAIRS * RC::BYTES;
  // LM head: the best (key, id) of each column from each epilogue warp,
  // [half * 4 + quadrant][key, id][column], in the A ring once every MMA is done
  uint32_t* s_key = reinterpret_cast<uint32_t*>(A0);
  // barriers: a_full[A], a_empty[A], b_full[STB], b_empty[STB], raw_full[RAW],
  // raw_empty[RAW], acc (the last piece's MMAs done), acc0 (the first of two
  // pieces' MMAs done), tfree (the first piece's accumulator read out).  The
  // two rings are freed separately (one commit each), so activation tiles
  // are fetched a full ring ahead of their MMAs.
  const uint32_t bar0 = smem_u32(s_bar);
  auto A_FULL = [&](int s) { return bar0 + 8 * s; };
  auto A_EMPTY = [&](int s) { return bar0 + 8 * (TC_MAX_A + s); };
  auto B_FULL = [&](int s) { return bar0 + 8 * (2 * TC_MAX_A + s); };
  auto B_EMPTY = [&](int s) { return bar0 + 8 * (2 * TC_MAX_A + TC_MAX_ST + s); };
  auto RAW_FULL = [&](int r) { return bar0 + 8 * (2 * TC_MAX_A + 2 * TC_MAX_ST + r); };
  auto RAW_EMPTY = [&](int r) { return bar0 + 8 * (2 * TC_MAX_A + 2 * TC_MAX_ST + TC_MAX_RAW + r); };
  const uint32_t ACC = bar0 + 8 * (2 * TC_MAX_A + 2 * TC_MAX_ST + 2 * TC_MAX_RAW);
  const uint32_t ACC0 = ACC + 8, TFREE = ACC + 16;

  // This CTA's run of work: the (tile, 64-k chunk) units of the matrix in
  // tile-major order are cut into P runs of equal length (+-1), never longer
  // than a tile.  A run is the part of tile tA from chunk kA (lenA chunks)
  // and, when it crosses into the next tile, that tile's first lenB chunks:
  // at most two pieces.  The next tile's head goes first (read out of tensor
  // memory into the run's partial mid-run); tA's part, which ends the tile
  // or lies inside it, stays in tensor memory to the end.  P = n_mt x S cuts
  // every tile into S aligned segments (a plain K split).
  // (32-bit: the host keeps P x n_mt x nch below 2^31)
  int nc, tA, kA, lenA;
  {
    const unsigned T = (unsigned)a.n_mt * (unsigned)a.nch;
    const unsigned U0 = blockIdx.x * T / (unsigned)a.P;
    const unsigned U1 = (blockIdx.x + 1) * T / (unsigned)a.P;
    tA = (int)(U0 / (unsigned)a.nch);
    kA = (int)U0 - tA * a.nch;
    const unsigned E = (unsigned)(tA + 1) * (unsigned)a.nch;  // end of the first tile
    nc = (int)(U1 - U0);
    lenA = RUNS ? (int)((U1 < E ? U1 : E) - U0) : nc;
  }
  const int lenB = nc - lenA;
  const bool two = RUNS && lenB > 0;
  auto pair_of = [&](int c) { return (two && c < lenB ? tA + 1 : tA) * CTA_PAIRS; };
  auto kchunk_of = [&](int c) { return two && c < lenB ? c : kA + c - lenB; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STA; s++) {
      mbar_init(A_FULL(s), TC_EPI_THREADS);
      mbar_init(A_EMPTY(s), 1);
    }
    for (int s = 0; s < STB; s++) {
      mbar_init(B_FULL(s), 1);
      mbar_init(B_EMPTY(s), 1);
    }
    for (int r = 0; r < RAWN; r++) {
      mbar_init(RAW_FULL(r), 1);
      mbar_init(RAW_EMPTY(r), TC_EPI_THREADS);
    }
    mbar_init(ACC, 1);
    mbar_init(ACC0, 1);
    mbar_init(TFREE, TC_EPI_THREADS);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_abort = 0;
  }
  if (warp == 2) {  // tensor memory for the accumulators: whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s_tmem)),
                 "r"(a.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort_flag = &s_abort;
  auto give_up = [&]() {
    atomicOr(a.err, ERR_TIMEOUT);
    *abort_flag = 1;
  };
  // The epilogue warps' TMEM lane quadrant, rows and columns: warp w reads
  // quadrant w % 4 and is the wi-th of the four warps of that quadrant,
  // wi = (w - 3) / 4: with two halves it takes half wi / 2 and every other
  // group of EW columns, with one every fourth group.
  struct EpiMap {
    int quad, wi, cw, col_first, col_step, ncw, m;
    uint32_t trow;
  };
  auto epi_map = [&]() {
    EpiMap e;
    e.quad = warp & 3;
    e.wi = (warp - TC_EPI_WARP0) >> 2;
    const int half = H == 2 ? e.wi >> 1 : 0;
    e.cw = H == 2 ? e.wi & 1 : e.wi;
    e.col_first = e.cw * EW;
    e.col_step = H == 2 ? 2 * EW : 4 * EW;
    e.ncw = H == 2 ? 2 : 4;  // warps sharing a quadrant's columns
    e.m = TC_M * half + 32 * e.quad + lane;  // weight row of the tile
    e.trow = tmem + (uint32_t)(half * a.acc_stride) + ((uint32_t)(32 * e.quad) << 16);
    return e;
  };
  // an epilogue thread's row of the accumulator -> this CTA's partial
  // ([P][Npad][rows] fp32: a warp's 32 rows of a column are 128 bytes)
  auto store_part = [&]() {
    const EpiMap e = epi_map();
    for (int col0 = e.col_first; col0 < a.Npad; col0 += e.col_step) {
      uint32_t v[EW];
      tc_ld(e.trow + col0, v);
      float* dst = a.part + ((size_t)blockIdx.x * a.Npad + col0) * CTA_ROWS + e.m;
#pragma unroll
      for (int c = 0; c < EW; c++) dst[(size_t)c * CTA_ROWS] = __uint_as_float(v[c]);
    }
  };

  int issued = 0;  // copies issued by this thread (producers): drained on abort
  if (warp == 0) {
    // ---- weight records: one bulk copy per pair and chunk (weights are
    // ---- constant: this starts before the grid dependency resolves)
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();
      for (int c = 0; c < nc && !*abort_flag; c++) {
        const int r = c % RAWN, ur = c / RAWN;
        if (ur > 0 && !mbar_wait(RAW_EMPTY(r), (ur - 1) & 1, LIN_WAIT_TRIES, abort_flag)) {
          give_up();
          break;
        }
        const int pair0 = pair_of(c), kc = kchunk_of(c);
        int np = 0;
        for (int p = 0; p < CTA_PAIRS; p++) np += pair0 + p < a.n_pairs;
        issued = c + 1;
        mbar_expect_tx(RAW_FULL(r), (uint32_t)(np * RC::BYTES));
        for (int p = 0; p < np; p++)
          bulk_copy(smem_u32(RAW0 + r * RAW_BYTES + p * RC::BYTES),
                    a.rec + ((size_t)(pair0 + p) * a.nch + kc) * RC::BYTES, RC::BYTES,
                    RAW_FULL(r), pol);
      }
    }
    grid_dep_wait();
  } else if (warp == 1) {
    // ---- activation tiles (written by the previous kernels)
    grid_dep_wait();
    if (lane == 0) {
      for (int c = 0; c < nc && !*abort_flag; c++) {
        const int s = c % STB, us = c / STB;
        if (us > 0 && !mbar_wait(B_EMPTY(s), (us - 1) & 1, LIN_WAIT_TRIES, abort_flag)) {
          give_up();
          break;
        }
        issued = c + 1;
        mbar_expect_tx(B_FULL(s), (uint32_t)B_BYTES);
        tma_load_2d(smem_u32(B0 + s * B_BYTES), &tmx, kchunk_of(c) * 64, 0, B_FULL(s));
      }
    }
  } else if (warp == 2) {
    // ---- MMA issue: one thread
    grid_dep_wait();
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(a.Npad);
      bool announced = false;
      int c = 0;
      for (; c < nc && !*abort_flag; c++) {
        const int sa = c % STA, ua = c / STA, sb = c % STB, ub = c / STB;
        if (!mbar_wait(A_FULL(sa), ua & 1, LIN_WAIT_TRIES, abort_flag) ||
            !mbar_wait(B_FULL(sb), ub & 1, LIN_WAIT_TRIES, abort_flag)) {
          give_up();
          break;
        }
        // a second piece starts in the tensor memory the first one's
        // accumulator held: wait until the epilogue warps have read it out
        if (two && c == lenB) {
          if (!mbar_wait(TFREE, 0, LIN_WAIT_TRIES, abort_flag)) {
            give_up();
            break;
          }
          // the head's partial is written: announce it to its tile's finisher
          __threadfence();
          atomicAdd(&a.tickets[tA + 1], 1u);
          announced = true;
        }
        tc_fence_after();
        const bool fresh = c == 0 || (two && c == lenB);  // a piece's first chunk
        const uint64_t bd = smem_desc_sw128(smem_u32(B0 + sb * B_BYTES));
        // per 16-k step: hi of each half, then lo of each half (each
        // accumulator still adds hi before lo, step by step; the halves'
        // MMAs alternate)
        const unsigned char* at0 = A0 + sa * A_STAGE;
        const uint64_t ah0 = smem_desc_sw128(smem_u32(at0));
        const uint64_t al0 = smem_desc_sw128(smem_u32(at0 + TC_A_BYTES));
        const uint64_t ah1 = smem_desc_sw128(smem_u32(at0 + TC_A_HALF));
        const uint64_t al1 = smem_desc_sw128(smem_u32(at0 + TC_A_HALF + TC_A_BYTES));
        const uint32_t d0 = tmem, d1 = tmem + (uint32_t)a.acc_stride;
#pragma unroll
        for (int kk = 0; kk < 4; kk++) {  // 16 k (32 bytes) per instruction
          const uint32_t acc = (!fresh || kk > 0) ? 1u : 0u;
          tc_mma(d0, ah0 + 2 * kk, bd + 2 * kk, idesc, acc);
          if (H == 2) tc_mma(d1, ah1 + 2 * kk, bd + 2 * kk, idesc, acc);
          tc_mma(d0, al0 + 2 * kk, bd + 2 * kk, idesc, 1u);
          if (H == 2) tc_mma(d1, al1 + 2 * kk, bd + 2 * kk, idesc, 1u);
        }
        tc_commit(A_EMPTY(sa));
        tc_commit(B_EMPTY(sb));
        if (two && c == lenB - 1) tc_commit(ACC0);  // the first piece's MMAs
      }
      if (two && c < lenB) tc_commit(ACC0);  // gave up before it: keep the count
      // a run that gave up still announces its head, so that the counters
      // end the launch at zero (its outputs are void: ERR_TIMEOUT is set)
      if (two && !announced) {
        __threadfence();
        atomicAdd(&a.tickets[tA + 1], 1u);
      }
      tc_commit(ACC);  // completes when every MMA issued above has
    }
  } else {
    // ---- dequant (warps 3..18).  Two halves: warp w' = w - 3 takes 16-row
    // ---- tile w' & 1 of pair (w' & 7) / 2 of half w' / 8, both 32-k blocks.
    // ---- One half: 16-row tile w' / 2 (pair w' / 4, tile (w' / 2) & 1),
    // ---- 32-k block w' & 1.
    const int wq = warp - TC_EPI_WARP0;
    const int dh = H == 2 ? wq >> 3 : 0;
    const int pc = H == 2 ? (wq & 7) >> 1 : wq >> 2, tile = H == 2 ? wq & 1 : (wq >> 1) & 1;
    const int b_lo = H == 2 ? 0 : wq & 1, b_hi = H == 2 ? 2 : b_lo + 1;
    grid_dep_wait();
    for (int c = 0; c < nc && !*abort_flag; c++) {
      const int r = c % RAWN, ur = c / RAWN, s = c % STA, us = c / STA;
      // the first wait's budget is the one a caller may shorten (test hook)
      bool ok = mbar_wait(RAW_FULL(r), ur & 1, c == 0 ? a.wait_tries : LIN_WAIT_TRIES, abort_flag);
      if (ok && us > 0) ok = mbar_wait(A_EMPTY(s), (us - 1) & 1, LIN_WAIT_TRIES, abort_flag);
      if (!ok) {
        give_up();
        break;
      }
      {
        unsigned char* at = A0 + s * A_STAGE + dh * TC_A_HALF;
        const int pp = 4 * dh + pc;  // pair of the CTA
        if (pair_of(c) + pp < a.n_pairs) {
          dequant_tile<QT>(RAW0 + r * RAW_BYTES + pp * RC::BYTES, at, at + TC_A_BYTES, pc, tile,
                           lane, b_lo, b_hi);
        } else {  // rows past the matrix: zeros (the warp's 16-byte units)
          const int nu = 4 * (b_hi - b_lo);
          for (int q = lane; q < 16 * nu; q += 32) {
            const int rr = 32 * pc + 16 * tile + q / nu, u = 4 * b_lo + q % nu;
            *reinterpret_cast<uint4*>(at + sw128_off(rr, u)) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(at + TC_A_BYTES + sw128_off(rr, u)) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      mbar_arrive(RAW_EMPTY(r));
      fence_proxy_async();  // the A tiles, to the tensor core's proxy
      mbar_arrive(A_FULL(s));
      if (two && c == lenB) {
        // the head's accumulator -> this run's partial, once its MMAs are
        // done (tA's first chunk is already staged); the MMA thread then
        // announces it and starts tA's part in the freed tensor memory
        if (!mbar_wait(ACC0, 0, LIN_WAIT_TRIES, abort_flag)) {
          give_up();
          break;
        }
        tc_fence_after();
        store_part();
        tc_fence_before();
        mbar_arrive(TFREE);
      }
    }
  }
  grid_dep_launch();

  // ---- epilogue (warps 3..18): the piece in tensor memory, tile tA's part.
  // ---- A tile that is this CTA's alone is finished from tensor memory.  A
  // ---- tile cut into several pieces is summed in k order: with runs, by
  // ---- the run holding its end (the other pieces' partials, then its own
  // ---- part from tensor memory); with a K split, the tile's CTAs meet and
  // ---- each adds all segments for its own share of the columns (an even
  // ---- share of the reads).  The CTAs that wait on others belong to one
  // ---- cooperative launch: all resident at once.
  if (warp >= TC_EPI_WARP0) {
    const EpiMap em = epi_map();
    const int cw = em.cw, ncw = em.ncw, m = em.m;
    const uint32_t trow = em.trow;
    const int slot = em.wi * 4 + em.quad;
    const int et = threadIdx.x - TC_EPI_WARP0 * 32;  // 0..511
    const int ngrp = a.Npad / EW;
    const unsigned T = (unsigned)a.n_mt * (unsigned)a.nch;
    const bool acc_ok = mbar_wait(ACC, 0, LIN_WAIT_TRIES);
    if (!acc_ok) give_up();
    tc_fence_after();
    bool aborted = *abort_flag != 0;
    // the runs holding the tile's first and last unit: its pieces, in k order
    auto owner = [&](unsigned u) { return (int)(((u + 1) * (unsigned)a.P - 1) / T); };
    const int t = tA;
    const int lo = owner((unsigned)t * (unsigned)a.nch);
    const int hi = owner((unsigned)(t + 1) * (unsigned)a.nch - 1);
    const int nseg = hi - lo + 1;
    const int n = t * CTA_ROWS + m;
    int g0 = 0, g1 = ngrp;  // column groups this CTA finishes
    int nsum = 0;           // partials it adds (runs lo, lo + 1, ...)
    bool from_tmem = true;  // then its own piece
    if (nseg > 1) {
      if (RUNS && (int)blockIdx.x != hi) {  // a piece before the tile's end
        store_part();
        epi_bar();
        if (et == 0) {
          __threadfence();
          atomicAdd(&a.tickets[t], 1u);
        }
        g1 = 0;
      } else if (RUNS) {  // the tile's end: wait for the other pieces
        if (et == 0) {
          if (!wait_count(&a.tickets[t], (unsigned)(nseg - 1))) give_up();
          __threadfence();
          a.tickets[t] = 0u;
        }
        epi_bar();
        aborted = *abort_flag != 0;
        nsum = nseg - 1;
      } else {  // K split
        store_part();
        epi_bar();
        if (et == 0) {
          // arrivals [t], departures [n_mt + t]: the last CTA past the
          // meeting resets both (every CTA of the tile arrives, aborted or not)
          __threadfence();
          atomicAdd(&a.tickets[t], 1u);
          if (!wait_count(&a.tickets[t], (unsigned)nseg)) give_up();
          __threadfence();
          if (atomicAdd(&a.tickets[a.n_mt + t], 1u) == (unsigned)(nseg - 1)) {
            a.tickets[t] = 0u;
            a.tickets[a.n_mt + t] = 0u;
          }
        }
        epi_bar();
        aborted = *abort_flag != 0;
        const int j = (int)blockIdx.x - lo;  // this CTA's segment
        g0 = j * ngrp / nseg;
        g1 = (j + 1) * ngrp / nseg;
        nsum = nseg;
        from_tmem = false;
      }
    }
    const size_t pstride = (size_t)a.Npad * CTA_ROWS;  // floats between partials
    for (int gi = g0 + cw; gi < g1; gi += ncw) {
      const int col0 = gi * EW;
      float v[EW];
      if (nsum > 0) {  // the partials in k order
        const float* src = a.part + (size_t)lo * pstride + (size_t)col0 * CTA_ROWS + m;
#pragma unroll
        for (int c = 0; c < EW; c++) v[c] = __ldcg(src + (size_t)c * CTA_ROWS);
        for (int q = 1; q < nsum; q++) {
          src += pstride;
#pragma unroll
          for (int c = 0; c < EW; c++) v[c] += __ldcg(src + (size_t)c * CTA_ROWS);
        }
      }
      if (from_tmem) {  // then this CTA's own piece
        uint32_t u[EW];
        tc_ld(trow + col0, u);
#pragma unroll
        for (int c = 0; c < EW; c++)
          v[c] = nsum > 0 ? v[c] + __uint_as_float(u[c]) : __uint_as_float(u[c]);
      }
      if (!aborted) tc_epilogue(a, n, col0, v, lane, s_key, slot);
    }
    if (a.epi.kind == EPI_LMHEAD) {
      // (one whole tile per CTA) the CTA's best of each column -> one packed
      // 64-bit maximum per column (value key high, inverted id low: ties go
      // to the lowest id); an aborted CTA still takes its ticket, so the
      // state is reset
      epi_bar();
      for (int r = et; r < a.R && !aborted; r += TC_EPI_THREADS) {
        // the slots that saw column r: the four quadrants of the warps of
        // the column's group (of each half)
        const int cr = H == 2 ? (r / EW) & 1 : (r / EW) & 3;
        const int nsl = 4 * H;
        uint32_t bk = 0u, bi = 0xffffffffu;
        for (int e = 0; e < nsl; e++) {
          const int q = (H == 2 ? (2 * (e >> 2) + cr) : cr) * 4 + (e & 3);
          const uint32_t k2 = s_key[(2 * q) * TC_MAX_R + r], i2 = s_key[(2 * q + 1) * TC_MAX_R + r];
          if (k2 > bk || (k2 == bk && i2 < bi)) {
            bk = k2;
            bi = i2;
          }
        }
        atomicMax(&a.amax_key[r], ((unsigned long long)bk << 32) | (unsigned long long)(~bi));
      }
      epi_bar();
      if (et == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&a.tickets[2 * a.n_mt], 1u);
        s_last = prev == (unsigned)(a.n_mt - 1);
        if (s_last) __threadfence();
      }
      epi_bar();
      if (s_last) {  // every tile's maxima are in: the argmax, and reset
        for (int r = et; r < a.Npad; r += TC_EPI_THREADS) {
          const unsigned long long k = __ldcg(&a.amax_key[r]);
          if (r < a.R && a.epi.argmax != nullptr) a.epi.argmax[r] = (int)(~(uint32_t)k);
          if (r < a.R && a.epi.row_key != nullptr) write_row_key(a.epi, r, (uint32_t)(k >> 32));
          a.amax_key[r] = 0ull;
        }
        if (et == 0) a.tickets[2 * a.n_mt] = 0u;
      }
    }
  }
  // ---- every copy and MMA this CTA issued has landed (the producers' last
  // ---- copies are consumed or drained): free the tensor memory
  if ((warp == 0 || warp == 1) && lane == 0 && *abort_flag) {
    // the last copy issued into each ring slot has landed (bounded): the
    // phase it completes is (uses of the slot - 1)
    const int depth = warp == 0 ? RAWN : STB;
    for (int q = 0; q < depth && q < issued; q++) {
      const int uses = (issued - 1 - q) / depth + 1;
      mbar_wait(warp == 0 ? RAW_FULL(q) : B_FULL(q), (uses - 1) & 1, LIN_WAIT_TRIES);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(a.tmem_cols)
                 : "memory");
  }
}

using TcKernel = void (*)(const CUtensorMap, const TcArgs);
TcKernel tc_kernel_for(int qtype, bool runs) {
  if (qtype == 4) return runs ? tc_linear_kernel<4, true> : tc_linear_kernel<4, false>;
  if (qtype == 6) return runs ? tc_linear_kernel<6, true> : tc_linear_kernel<6, false>;
  if (qtype == 8) return runs ? tc_linear_kernel<8, true> : tc_linear_kernel<8, false>;
  return nullptr;
}

int tc_rec_bytes(int qtype) {
  return qtype == 4 ? TcRec<4>::BYTES : (qtype == 6 ? TcRec<6>::BYTES : TcRec<8>::BYTES);
}

constexpr int TC_SMEM_MAX = 227 * 1024 - 2 * 1024;  // dynamic part (the static part is < 1 KB)

// Ring depths of a launch that fit the shared memory: A stages (two of
// 64 KB with two halves, three of 32 KB with one: the dequant of a chunk
// overlaps the MMAs of the one before), then the raw-record ring (weights
// from DRAM: the longest latency) as deep as two activation stages leave
// room for, up to six, then the activation ring (tiles from L2) as deep as
// the rest allows.
void tc_rings(int qtype, int Npad, int halves, int* sta, int* stb, int* raw) {
  const int raw_bytes = 4 * halves * tc_rec_bytes(qtype), b_bytes = Npad * 128;
  *sta = halves == 2 ? 2 : 3;
  const int fixed = 1024 + *sta * halves * TC_A_HALF;
  auto raw_for = [&](int b) { return std::min(TC_MAX_RAW, (TC_SMEM_MAX - fixed - b * b_bytes) / raw_bytes); };
  const int want = std::min(6, raw_for(2));
  int b = TC_MAX_ST;
  while (b > 2 && raw_for(b) < want) b--;
  *stb = b;
  *raw = std::max(2, raw_for(b));
}
size_t tc_smem_bytes(int qtype, int Npad, int halves, int sta, int stb, int raw) {
  return 1024 + (size_t)sta * halves * TC_A_HALF + (size_t)stb * Npad * 128 +
         (size_t)raw * 4 * halves * tc_rec_bytes(qtype);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    cudaGetLastError();
  });
  return fn;
}

}  // namespace

int tc_npad(int R) { return std::max(16, (R + 15) / 16 * 16); }
int tc_mtiles(const QMat& w) { return (w.N + TC_M * w.tc_H - 1) / (TC_M * w.tc_H); }

// Launch shape of a matrix: CTA height (one or two 128-row halves) and the
// cut of its (tile, chunk) units into runs, from an estimate of the longest
// run in chunk steps of a one-half CTA.  A two-half chunk costs about 1.4
// one-half chunks (the activation tile and the chunk's handshakes serve
// twice the MMAs: measured 1.67 vs 1.2 us inside the 192-row round).  Cuts:
//   * one run per tile, in waves when there are more tiles than SMs;
//   * a K split, S aligned runs per tile (n_mt x S <= SMs): each CTA also
//     writes and meets, a small cost per segment;
//   * one run per SM over all units (a run may end one tile and start the
//     next): the most even, but such a run reads its first piece out of
//     tensor memory before it starts the second (about 2.5 chunks).
// Inside the 192-row round this gives two halves everywhere: QKV 7168x5120
// S = 5, O 5120x5120 S = 7, down 5120x13824 S = 7, gate/up 27648x5120 one
// run per SM (108 tiles: 80 -> 57 chunks for the busiest CTA), the LM head
// one run per tile; one half wins for small N.
// The most pieces any tile has when n_mt x nch units are cut into P runs.
static int tc_max_pieces(int n_mt, int nch, int P) {
  const long long T = (long long)n_mt * nch;
  auto owner = [&](long long u) { return (int)(((u + 1) * P - 1) / T); };
  int most = 1;
  for (int t = 0; t < n_mt; t++)
    most = std::max(most, owner((long long)(t + 1) * nch - 1) - owner((long long)t * nch) + 1);
  return most;
}

static double tc_estimate(int N, int nch, int sms, int halves, int* ctas) {
  const int n_mt = (N + TC_M * halves - 1) / (TC_M * halves);
  const double per_chunk = halves == 2 ? 1.4 : 1.0;
  const long long T = (long long)n_mt * nch;
  int best_p = n_mt;
  double best = std::ceil((double)n_mt / sms) * nch * per_chunk;  // one run per tile
  if (n_mt < sms) {
    for (int S = 2; S <= 8 && S <= nch && n_mt * S <= sms; S++) {
      const double t = std::ceil((double)nch / S) * per_chunk + 0.25 * S;
      if (t < best - 1e-9) {
        best = t;
        best_p = n_mt * S;
      }
    }
    const int P = (int)std::min<long long>(sms, T);
    // runs: a tile's end finishes it from the other pieces' partials, so
    // keep to at most three pieces a tile
    if (P > n_mt && P % n_mt != 0 && tc_max_pieces(n_mt, nch, P) <= 3) {
      const long long run = (T + P - 1) / P;
      const double t = run * per_chunk + 2.5;
      if (t < best - 1e-9) {
        best = t;
        best_p = P;
      }
    }
  }
  if (ctas != nullptr) *ctas = best_p;
  return best;
}

int tc_choose_halves(int N, int nch, int sms) {
  return tc_estimate(N, nch, sms, 2, nullptr) < tc_estimate(N, nch, sms, 1, nullptr) ? 2 : 1;
}

int tc_choose_ctas(int N, int nch, int sms, int halves) {
  int P = 1;
  tc_estimate(N, nch, sms, halves, &P);
  return P;
}

size_t tc_part_floats(const QMat& w, int R) {
  return w.tc_P > tc_mtiles(w) ? (size_t)w.tc_P * tc_npad(std::min(R, TC_MAX_R)) * TC_M * w.tc_H
                    : 0;
}
size_t tc_tickets_needed(const QMat& w) { return 2 * (size_t)tc_mtiles(w) + 1; }

static int tc_launch_block(const QMat& w, const __half* x, int R, const LinEpi& epi,
                           const LinScratch& scr, cudaStream_t st) {
  if (R < 1 || R > TC_MAX_R) return fail(SPEC_E_SHAPE, "tensor-core GEMM: 1 <= rows <= 192 per launch");
  if (scr.err == nullptr) return fail(SPEC_E_INVALID, "tensor-core GEMM: no error word");
  if (tc_part_floats(w, R) > scr.part_floats || tc_tickets_needed(w) > scr.n_tickets ||
      (epi.kind == EPI_LMHEAD && scr.amax_keys == nullptr))
    return fail(SPEC_E_SHAPE, "tensor-core GEMM: scratch too small for this R");
  if ((reinterpret_cast<uintptr_t>(x) & 15u) != 0 || w.K % 8 != 0)
    return fail(SPEC_E_SHAPE, "tensor-core GEMM: x must be 16-byte aligned");
  auto enc = encode_fn();
  if (enc == nullptr) return fail(SPEC_E_CUDA, "cuTensorMapEncodeTiled is not available");
  const int Npad = tc_npad(R);
  // the activations x [R][K] fp16: box of 64 k x Npad rows, 128-byte swizzle;
  // rows past R are out of the tensor and read as zero
  CUtensorMap map;
  const cuuint64_t gdim[2] = {(cuuint64_t)w.K, (cuuint64_t)R};
  const cuuint64_t gstride[1] = {(cuuint64_t)w.K * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)Npad};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult cr = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(x), gdim,
                          gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return fail(SPEC_E_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)cr));
  TcArgs a;
  a.rec = w.rec;
  a.N = w.N;
  a.K = w.K;
  a.nch = w.nch;
  a.n_pairs = w.n_pairs;
  a.n_mt = tc_mtiles(w);
  // the LM head's argmax gathers whole tiles: one run per tile
  a.P = epi.kind == EPI_LMHEAD ? a.n_mt : w.tc_P;
  if ((long long)(a.P + 1) * a.n_mt * a.nch >= (1ll << 31))
    return fail(SPEC_E_SHAPE, "tensor-core GEMM: matrix too large for the 32-bit work cut");
  a.R = R;
  a.Npad = Npad;
  // one accumulator of Npad columns per half, a power of two apart
  a.halves = w.tc_H;
  a.acc_stride = Npad <= 16 ? 16 : (Npad <= 32 ? 32 : (Npad <= 64 ? 64 : (Npad <= 128 ? 128 : 256)));
  a.tmem_cols = std::max(32, a.halves * a.acc_stride);
  tc_rings(w.qtype, Npad, a.halves, &a.a_stages, &a.b_stages, &a.raw_depth);
  a.epi = epi;
  a.part = scr.part;
  a.tickets = scr.tickets;
  a.amax_key = scr.amax_keys;
  a.err = scr.err;
  a.wait_tries = scr.wait_tries > 0 ? LIN_WAIT_TRIES : 0;
  // runs that cross a tile boundary: not every tile cut into aligned segments
  const TcKernel k = tc_kernel_for(w.qtype, a.P > a.n_mt && a.P % a.n_mt != 0);
  if (k == nullptr) return fail(SPEC_E_INVALID, "tensor-core GEMM: no kernel for this format");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.P);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = tc_smem_bytes(w.qtype, Npad, a.halves, a.a_stages, a.b_stages, a.raw_depth);
  if (cfg.dynamicSmemBytes > (size_t)TC_SMEM_MAX)
    return fail(SPEC_E_SHAPE, "tensor-core GEMM: rings do not fit the shared memory");
  cfg.stream = st;
  // the CTAs of a shared tile wait on one another: a cooperative launch,
  // which guarantees they are all resident (such cuts keep to one wave)
  cudaLaunchAttribute at[2];
  int nat = 0;
  if (programmatic_launch()) {
    at[nat].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[nat].val.programmaticStreamSerializationAllowed = 1;
    nat++;
  }
  if (a.P > a.n_mt) {
    at[nat].id = cudaLaunchAttributeCooperative;
    at[nat].val.cooperative = 1;
    nat++;
  }
  cfg.attrs = at;
  cfg.numAttrs = nat;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k, map, a);
  if (e != cudaSuccess) return fail(SPEC_E_CUDA, std::string("tensor-core GEMM launch: ") + cudaGetErrorString(e));
  return SPEC_OK;
}

// Rows in blocks of at most 192 (the accumulators' columns and the rings fit
// the tensor and shared memory); every row is computed by the same
// instructions whichever block it falls in.
int tc_linear_launch(const QMat& w, const __half* x, int R, const LinEpi& epi,
                     const LinScratch& scr, cudaStream_t st) {
  if (R < 1) return fail(SPEC_E_SHAPE, "tensor-core GEMM: R must be >= 1");
  for (int r0 = 0; r0 < R; r0 += TC_MAX_R) {
    LinEpi e = epi;
    const size_t o = (size_t)r0;
    switch (epi.kind) {
      case EPI_STORE:
      case EPI_RESID:
        e.y = epi.y + o * epi.ldy;
        break;
      case EPI_SWIGLU:
        e.out16 = epi.out16 + o * epi.ldo;
        break;
      case EPI_QKV:
        e.out16 = epi.out16 + o * epi.nq * epi.hd;
        e.rows = epi.rows + o;
        break;
      case EPI_LMHEAD:
        if (epi.y != nullptr) e.y = epi.y + o * epi.ldy;
        if (epi.argmax != nullptr) e.argmax = epi.argmax + o;
        e.rk_row0 = epi.rk_row0 + r0;
        break;
    }
    const int rc = tc_launch_block(w, x + o * w.K, std::min(TC_MAX_R, R - r0), e, scr, st);
    if (rc != SPEC_OK) return rc;
  }
  return SPEC_OK;
}

void tc_init_attrs() {
  for (int qt : {4, 6, 8})
    for (bool runs : {false, true})
      cudaFuncSetAttribute(tc_kernel_for(qt, runs), cudaFuncAttributeMaxDynamicSharedMemorySize,
                           TC_SMEM_MAX);
}
