// accept.cu -- acceptance and commit of the verify round.
//
// Greedy ("Speculative Decoding (D5-R) -- Plan", section 3): accept while the
// target's argmax equals the drafted token; always emit one more token, the
// correction at the first mismatch or the bonus after a fully accepted block.
//
// Strict rejection sampling ("DFlash and DSpark Speculative Decoding",
// "Notes": use the strict sampler, which is lossless): accept draft x with
// probability min(1, p_x / q_x), else resample from norm(max(0, p - q)).
// The probabilities are integer weights W_v = floor(exp(z_v - max z) * 2^32)
// with an fp32 exp made of individually rounded operations (Cody-Waite
// reduction with a two-part ln 2, degree-7 Taylor polynomial in Horner form,
// exact power-of-two scaling), so every decision is an exact integer
// comparison and is identical on any IEEE-754 implementation.  Uniforms come
// from Philox4x32-10 (Salmon et al., SC'11) keyed by the seed, with counter
// (emitted-slot index, sequence id, 0): one counter per emitted token, none
// for a rejected suffix ("Model-neutral Speculative Decoding", "The exactness
// transaction").
#include <cooperative_groups.h>
#include <math.h>

#include <algorithm>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace {

typedef unsigned __int128 u128;

// ---------------------------------------------------------------------------
// the sampler's exp and integer weight (fp32, no contraction: __f*_rn)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t int_weight(float x) {
  if (!(x >= -87.0f)) return 0ull;
  const float LOG2E = 0x1.715476p+0f;     // fl32(1 / ln 2)
  const float LN2_HI = 0x1.62e4p-1f;      // ln 2 to 12 significant bits
  const float LN2_LO = 0x1.7f7d1cp-20f;   // fl32(ln 2 - LN2_HI)
  const float C[8] = {0x1p+0f,        0x1p+0f,        0x1p-1f,         0x1.555556p-3f,
                      0x1.555556p-5f, 0x1.111112p-7f, 0x1.6c16c2p-10f, 0x1.a01a02p-13f};
  const float n = rintf(__fmul_rn(x, LOG2E));
  float r = __fsub_rn(x, __fmul_rn(n, LN2_HI));
  r = __fsub_rn(r, __fmul_rn(n, LN2_LO));
  float p = C[7];
#pragma unroll
  for (int k = 6; k >= 0; k--) p = __fadd_rn(__fmul_rn(p, r), C[k]);
  const int e = (int)n + 32;
  if (e < 0) return 0ull;
  const float v = __fmul_rn(p, __int_as_float((e + 127) << 23));
  return (uint64_t)v;  // truncation: exact floor of a non-negative value
}

__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int round = 0; round < 10; round++) {
    if (round > 0) {
      k0 += W0;
      k1 += W1;
    }
    const uint32_t hi0 = __umulhi(M0, c[0]), lo0 = M0 * c[0];
    const uint32_t hi1 = __umulhi(M1, c[2]), lo1 = M1 * c[2];
    const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

__device__ __forceinline__ void uniforms(uint64_t seed, uint64_t slot, uint32_t seq_id,
                                         uint32_t out[4]) {
  out[0] = (uint32_t)slot;
  out[1] = (uint32_t)(slot >> 32);
  out[2] = seq_id;
  out[3] = 0u;  // domain 0: the target sampler
  philox4x32_10(out, (uint32_t)seed, (uint32_t)(seed >> 32));
}

// floor(U * total / 2^32) without overflowing 128 bits
__device__ __forceinline__ u128 scaled_threshold(uint32_t U, u128 total) {
  const u128 hi = total >> 32, lo = total & 0xFFFFFFFFull;
  return (u128)U * hi + (((u128)U * lo) >> 32);
}

// ---------------------------------------------------------------------------
// greedy
// ---------------------------------------------------------------------------
__global__ void accept_greedy_kernel(const int32_t* __restrict__ argmax,
                                     const int32_t* __restrict__ draft, int n_seq, int d,
                                     int32_t* __restrict__ n_acc, int32_t* __restrict__ em) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= n_seq) return;
  const int32_t* am = argmax + (size_t)s * (d + 1);
  const int32_t* dr = draft + (size_t)s * d;
  int32_t* e = em + (size_t)s * (d + 1);
  int a = 0;
  while (a < d && am[a] == dr[a]) {
    e[a] = dr[a];
    a++;
  }
  e[a] = am[a];
  for (int i = a + 1; i <= d; i++) e[i] = -1;
  n_acc[s] = a;
}

// ---------------------------------------------------------------------------
// stochastic, step 1: per-row max z and S = sum W, over every row the accept
// may need (p rows 0..d, then q rows 0..d-1 of every sequence), in two
// streaming passes of many short CTAs, each over a segment of one row:
//   1. the largest logit of the row (z = l / T is monotone in l for T > 0,
//      so max z = fl(max l / T)): one atomicMax of an order-preserving key
//      per CTA, and the non-finite check;
//   2. S = sum of the integer weights: each CTA adds its segment's exact
//      64-bit sum (integer sums do not depend on the order).
// The second pass walks the segments in the reverse order of the first, so
// the rows it starts with are the ones the first pass left in L2.
// ---------------------------------------------------------------------------
constexpr int ST_THREADS = 256;
constexpr int ST_SEG = 4096;  // logits per CTA (about)
constexpr int ST_VEC = 4;     // float4 loads in flight per thread and step

// Order-preserving 32-bit key of a float (-0 taken as +0).  Keys of the
// same row are only compared and turned back into the value.
__device__ __forceinline__ uint32_t max_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// The row's max z from the key of its largest logit.
__device__ __forceinline__ float row_zmax(uint32_t key, float T) {
  const float m = key_value(key);
  return T == 1.0f ? m : __fdiv_rn(m, T);
}
__device__ __forceinline__ float zval(float l, float T) {
  return T == 1.0f ? l : __fdiv_rn(l, T);  // x / 1 is x exactly
}

int st_segments(int V) { return std::max(1, std::min(64, (V + ST_SEG - 1) / ST_SEG)); }

__device__ __forceinline__ const float* stoch_row(const float* p, const float* q, int d, int V,
                                                  int row) {
  const int rows_per_seq = 2 * d + 1;
  const int s = row / rows_per_seq, rr = row % rows_per_seq;
  return rr <= d ? p + ((size_t)s * (d + 1) + rr) * V : q + ((size_t)s * d + (rr - d - 1)) * V;
}

// Calls f(value) for every logit of src[s0, s1): float4 loads over the
// 16-byte-aligned middle, ST_VEC of them issued before any is used, and
// scalar loads at the two ends.
template <class F>
__device__ __forceinline__ void for_segment(const float* src, int s0, int s1, F&& f) {
  const int tid = threadIdx.x;
  int a0 = s0 + (int)((4u - ((uint32_t)(reinterpret_cast<uintptr_t>(src + s0) >> 2) & 3u)) & 3u);
  if (a0 > s1) a0 = s1;
  const int n4 = (s1 - a0) >> 2, a1 = a0 + 4 * n4;
  for (int v = s0 + tid; v < a0; v += ST_THREADS) f(__ldcs(src + v));
  for (int v = a1 + tid; v < s1; v += ST_THREADS) f(__ldcs(src + v));
  const float4* s4 = reinterpret_cast<const float4*>(src + a0);
  for (int i = tid; i < n4; i += ST_THREADS * ST_VEC) {
    float4 t[ST_VEC];
#pragma unroll
    for (int u = 0; u < ST_VEC; u++)
      t[u] = i + u * ST_THREADS < n4 ? __ldcs(s4 + i + u * ST_THREADS)
                                     : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
    for (int u = 0; u < ST_VEC; u++)
      if (i + u * ST_THREADS < n4) {
        f(t[u].x);
        f(t[u].y);
        f(t[u].z);
        f(t[u].w);
      }
  }
}

// q_only: the grid covers the q rows only (the p rows' keys came from the
// LM head); CTA b then takes q row b / nseg of the sequences in order.
__global__ void __launch_bounds__(ST_THREADS)
row_max_kernel(const float* __restrict__ p, const float* __restrict__ q, int d, int V, int nseg,
               int q_only, uint32_t* __restrict__ row_key, uint32_t* __restrict__ err) {
  __shared__ float s_red[ST_THREADS / 32];
  __shared__ int s_bad;
  const int ri = blockIdx.x / nseg, sg = blockIdx.x % nseg;
  const int row = q_only ? (ri / d) * (2 * d + 1) + d + 1 + ri % d : ri;
  const float* src = stoch_row(p, q, d, V, row);
  const int s0 = (int)((long long)sg * V / nseg), s1 = (int)((long long)(sg + 1) * V / nseg);
  if (threadIdx.x == 0) s_bad = 0;
  float mx = -INFINITY;
  bool bad = false;
  for_segment(src, s0, s1, [&](float l) {
    bad |= !isfinite(l);
    mx = fmaxf(mx, l);
  });
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  __syncthreads();
  if (bad) s_bad = 1;
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = s_red[0];
    for (int w = 1; w < ST_THREADS / 32; w++) m = fmaxf(m, s_red[w]);
    atomicMax(&row_key[row], max_key(m));
    if (s_bad) atomicOr(err, ERR_NONFINITE);
  }
}

__global__ void __launch_bounds__(ST_THREADS)
row_sum_kernel(const float* __restrict__ p, const float* __restrict__ q, int d, int V, int nseg,
               float T, const uint32_t* __restrict__ row_key,
               unsigned long long* __restrict__ row_sum) {
  __shared__ unsigned long long s_red[ST_THREADS / 32];
  const int id = (int)gridDim.x - 1 - (int)blockIdx.x;  // reverse of the max pass
  const int row = id / nseg, sg = id % nseg;
  const float* src = stoch_row(p, q, d, V, row);
  const int s0 = (int)((long long)sg * V / nseg), s1 = (int)((long long)(sg + 1) * V / nseg);
  const float zmax = row_zmax(row_key[row], T);
  unsigned long long acc = 0ull;  // integer sums: exact in any order
  for_segment(src, s0, s1, [&](float l) { acc += int_weight(__fsub_rn(zval(l, T), zmax)); });
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t = 0ull;
    for (int w = 0; w < ST_THREADS / 32; w++) t += s_red[w];
    atomicAdd(&row_sum[row], t);
  }
}

// ---------------------------------------------------------------------------
// stochastic, step 2: the accept scan, one warp per sequence.  The scan is
// sequential by definition (stop at the first rejection or invalid draft),
// but its tests are independent: lane i evaluates position base + i (its
// draft, the two weights, its own sampler counter), and the first stopping
// position is one ballot.  Nothing past that position changes the outcome.
// decision[s] = (a, row to sample from, U2, mode: 1 residual / 2 bonus / 0 error)
// ---------------------------------------------------------------------------
constexpr int DC_WARPS = 4;  // sequences per CTA

__global__ void __launch_bounds__(DC_WARPS * 32)
decide_kernel(const float* __restrict__ p, const float* __restrict__ q,
              const int32_t* __restrict__ draft, int n_seq, int d, int V, float T, uint64_t seed,
              const int32_t* __restrict__ seq_ids, const uint64_t* __restrict__ emit_idx,
              int emit_by_slot, int n_slots, const uint32_t* __restrict__ row_key,
              const unsigned long long* __restrict__ row_sum, int4* __restrict__ decision,
              int32_t* __restrict__ n_acc, int32_t* __restrict__ em, uint32_t* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const int s = blockIdx.x * DC_WARPS + (threadIdx.x >> 5);
  if (s >= n_seq) return;  // whole warps
  const int rows_per_seq = 2 * d + 1;
  const uint32_t sid = (uint32_t)seq_ids[s];
  int32_t* e = em + (size_t)s * (d + 1);
  if (emit_by_slot && (int)sid >= n_slots) {  // also catches negative ids
    for (int i = lane; i <= d; i += 32) e[i] = -1;
    if (lane == 0) {
      atomicOr(err, ERR_SEQ);
      decision[s] = make_int4(0, 0, 0, 0);
      n_acc[s] = -1;
    }
    return;
  }
  const uint64_t e0 = emit_idx[emit_by_slot ? (int)sid : s];
  for (int base = 0; base <= d; base += 32) {
    const int a = base + lane;
    // lane a < d: accept test of draft a; lane a == d: the bonus draw
    bool stop = false, invalid = false;
    uint32_t U1 = 0u;
    int x = -1;
    if (a < d) {
      x = draft[(size_t)s * d + a];
      invalid = x < 0 || x >= V;
      if (!invalid) {
        const int rp = s * rows_per_seq + a, rq = s * rows_per_seq + d + 1 + a;
        const float zp = zval(p[((size_t)s * (d + 1) + a) * V + x], T);
        const float zq = zval(q[((size_t)s * d + a) * V + x], T);
        const uint64_t Wx = int_weight(__fsub_rn(zp, row_zmax(row_key[rp], T)));
        const uint64_t Wqx = int_weight(__fsub_rn(zq, row_zmax(row_key[rq], T)));
        const uint64_t S = row_sum[rp], Sq = row_sum[rq];
        uint32_t U[4];
        uniforms(seed, e0 + (uint64_t)a, sid, U);
        bool acc;
        if (Wqx == 0ull) {
          acc = Wx > 0ull;
        } else {
          const u128 lhs = (u128)U[0] * (u128)Wqx * (u128)S;
          const u128 rhs = ((u128)Wx << 32) * (u128)Sq;
          acc = lhs < rhs;
        }
        U1 = U[1];
        stop = !acc;
      } else {
        stop = true;
      }
    } else if (a == d) {
      uint32_t U[4];
      uniforms(seed, e0 + (uint64_t)d, sid, U);
      U1 = U[1];
      stop = true;  // the bonus: every draft accepted
    }
    const unsigned ball = __ballot_sync(0xffffffffu, a <= d && stop);
    if (a <= d) e[a] = -1;
    if (ball == 0u) {  // all 32 positions accepted
      e[a] = x;
      continue;
    }
    const int f = __ffs(ball) - 1;  // first stopping lane
    if (lane < f) e[a] = x;
    if (lane == f) {
      if (invalid) {
        atomicOr(err, ERR_TOKEN);
        decision[s] = make_int4(a, a, 0, 0);
        n_acc[s] = -1;
      } else {
        decision[s] = make_int4(a, a, (int)U1, a == d ? 2 : 1);
        n_acc[s] = a;
      }
    }
    for (int i = base + 32 + lane; i <= d; i += 32) e[i] = -1;
    return;
  }
}

// ---------------------------------------------------------------------------
// stochastic, step 3: resample one row per sequence.  One cluster of RS_CL
// CTAs per sequence cuts the row into RS_CL x RS_WARPS warp ranges; each warp
// sums the exact 128-bit masses of its range (order-free integers); rank 0
// reads every range sum through distributed shared memory, draws the
// threshold and finds the range that holds it; the CTA owning that range
// cuts it into RS_WARPS sub-ranges the same way, and the warp owning the
// right one scans it with a 128-bit warp prefix.
// ---------------------------------------------------------------------------
constexpr int RS_CL = 8;
constexpr int RS_THREADS = 512;
constexpr int RS_WARPS = RS_THREADS / 32;
constexpr int RS_RANGES = RS_CL * RS_WARPS;

__device__ __forceinline__ u128 shfl_u128(u128 v, int src) {
  uint64_t lo = (uint64_t)v, hi = (uint64_t)(v >> 64);
  lo = __shfl_sync(0xffffffffu, lo, src);
  hi = __shfl_sync(0xffffffffu, hi, src);
  return ((u128)hi << 64) | lo;
}
__device__ __forceinline__ u128 shfl_up_u128(u128 v, int delta) {
  uint64_t lo = (uint64_t)v, hi = (uint64_t)(v >> 64);
  lo = __shfl_up_sync(0xffffffffu, lo, delta);
  hi = __shfl_up_sync(0xffffffffu, hi, delta);
  return ((u128)hi << 64) | lo;
}

// The residual (mode 1: max(0, W Sq - Wq S)) or target (mode 2: W) mass of
// one token from its two logits.
__device__ __forceinline__ u128 mass_from(int mode, float lp, float lq, float T, float mp,
                                          float mq, uint64_t S, uint64_t Sq) {
  const uint64_t W = int_weight(__fsub_rn(zval(lp, T), mp));
  if (mode == 2) return (u128)W;
  const uint64_t Wq = int_weight(__fsub_rn(zval(lq, T), mq));
  const u128 a = (u128)W * Sq, b = (u128)Wq * S;
  return a > b ? a - b : (u128)0;
}

constexpr int RS_ILP = 8;  // tokens per lane whose loads are issued before any is used

// The sum of the masses of [v0, v1) over one warp (every lane gets it).
__device__ __forceinline__ u128 warp_mass(int mode, const float* prow, const float* qrow, int v0,
                                          int v1, float T, float mp, float mq, uint64_t S,
                                          uint64_t Sq, int lane) {
  u128 acc = 0;
  for (int vb = v0 + lane; vb < v1; vb += 32 * RS_ILP) {
    float lp[RS_ILP], lq[RS_ILP];
#pragma unroll
    for (int u = 0; u < RS_ILP; u++) {
      const int v = vb + 32 * u;
      lp[u] = v < v1 ? prow[v] : 0.0f;
      lq[u] = v < v1 && mode == 1 ? qrow[v] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < RS_ILP; u++)
      if (vb + 32 * u < v1) acc += mass_from(mode, lp[u], lq[u], T, mp, mq, S, Sq);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += shfl_u128(acc, lane ^ off);
  return acc;
}

__global__ void __launch_bounds__(RS_THREADS)
resample_kernel(const float* __restrict__ p, const float* __restrict__ q, int n_seq, int d,
                int V, float T, const uint32_t* __restrict__ row_key,
                const unsigned long long* __restrict__ row_sum,
                const int4* __restrict__ decision, int32_t* __restrict__ em,
                uint32_t* __restrict__ err) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int s = blockIdx.x / RS_CL;
  const int4 dec = decision[s];
  const int mode = dec.w;
  if (mode == 0) return;  // every CTA of the cluster returns: nothing syncs
  const int a = dec.x, row = dec.y;
  const uint32_t U2 = (uint32_t)dec.z;
  const int rows_per_seq = 2 * d + 1;
  const int rp = s * rows_per_seq + row;
  const int rq = s * rows_per_seq + d + 1 + (row < d ? row : 0);
  const float* prow = p + ((size_t)s * (d + 1) + row) * V;
  const float* qrow = mode == 1 ? q + ((size_t)s * d + row) * V : nullptr;
  const float mp = row_zmax(row_key[rp], T);
  const float mq = mode == 1 ? row_zmax(row_key[rq], T) : 0.0f;
  const uint64_t S = row_sum[rp];
  const uint64_t Sq = mode == 1 ? row_sum[rq] : 0ull;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ u128 s_w[RS_WARPS];
  __shared__ u128 s_rem;
  __shared__ int s_range;
  const int span = (V + RS_RANGES - 1) / RS_RANGES;
  {
    const int wr = rank * RS_WARPS + warp;
    const int v0 = min(V, wr * span), v1 = min(V, v0 + span);
    const u128 m = warp_mass(mode, prow, qrow, v0, v1, T, mp, mq, S, Sq, lane);
    if (lane == 0) s_w[warp] = m;
  }
  cluster.sync();
  if (rank == 0) {
    // every range sum into rank 0's shared memory (one remote load each, in
    // parallel), then the total in range order, the threshold and the range
    // that holds it
    __shared__ u128 s_all[RS_RANGES];
    for (int k = threadIdx.x; k < RS_RANGES; k += RS_THREADS)
      s_all[k] = cluster.map_shared_rank(s_w, k / RS_WARPS)[k % RS_WARPS];
    __syncthreads();
    if (threadIdx.x == 0) {
      u128 total = 0;
      for (int k = 0; k < RS_RANGES; k++) total += s_all[k];
      s_range = -1;
      if (total == 0) {
        atomicOr(err, ERR_NONFINITE);
      } else {
        const u128 t = scaled_threshold(U2, total);
        u128 cum = 0;
        for (int k = 0; k < RS_RANGES; k++) {
          if (cum + s_all[k] > t) {
            s_range = k;
            s_rem = t - cum;
            break;
          }
          cum += s_all[k];
        }
      }
    }
  }
  cluster.sync();
  const int range = *cluster.map_shared_rank(&s_range, 0);
  const u128 rem0 = *cluster.map_shared_rank(&s_rem, 0);
  cluster.sync();  // rank 0's shared memory stays until every CTA has read it
  if (range < 0 || rank != range / RS_WARPS) return;
  // the owning CTA: the range cut into RS_WARPS sub-ranges
  const int u0 = min(V, range * span), u1 = min(V, u0 + span);
  const int sspan = (u1 - u0 + RS_WARPS - 1) / RS_WARPS;
  const int w0 = min(u1, u0 + warp * sspan), w1 = min(u1, w0 + sspan);
  const u128 sub = warp_mass(mode, prow, qrow, w0, w1, T, mp, mq, S, Sq, lane);
  __syncthreads();  // s_w is reused
  if (lane == 0) s_w[warp] = sub;
  __syncthreads();
  __shared__ int s_sub;
  __shared__ u128 s_rem2;
  if (threadIdx.x == 0) {
    u128 cum = 0;
    s_sub = RS_WARPS - 1;
    s_rem2 = 0;
    for (int k = 0; k < RS_WARPS; k++) {
      if (cum + s_w[k] > rem0) {
        s_sub = k;
        s_rem2 = rem0 - cum;
        break;
      }
      cum += s_w[k];
    }
  }
  __syncthreads();
  if (warp != s_sub) return;
  const u128 rem = s_rem2;
  u128 base = 0;
  int found = -1;
  for (int vb = w0; vb < w1 && found < 0; vb += 32) {
    const int v = vb + lane;
    u128 m = v < w1 ? mass_from(mode, prow[v], mode == 1 ? qrow[v] : 0.0f, T, mp, mq, S, Sq)
                    : (u128)0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {  // inclusive warp prefix
      const u128 o = shfl_up_u128(m, off);
      if (lane >= off) m += o;
    }
    const bool hit = v < w1 && base + m > rem;
    const unsigned ball = __ballot_sync(0xffffffffu, hit);
    if (ball) found = vb + __ffs(ball) - 1;
    base += shfl_u128(m, 31);
  }
  if (lane == 0) em[(size_t)s * (d + 1) + a] = found;
}

// Standalone accept: on a device error the outputs read -1 and the sampler
// state is left alone; otherwise emit_idx advances by the emitted count.
__global__ void stoch_finalize_kernel(int n_seq, int d, int32_t* __restrict__ n_acc,
                                      int32_t* __restrict__ em, uint64_t* __restrict__ emit_idx,
                                      const uint32_t* __restrict__ err) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= n_seq) return;
  const int a = n_acc[s];
  int32_t* e = em + (size_t)s * (d + 1);
  if (*err != 0u || a < 0 || a > d || e[a] < 0) {
    n_acc[s] = -1;
    for (int i = 0; i <= d; i++) e[i] = -1;
    return;
  }
  emit_idx[s] += (uint64_t)(a + 1);
}

// Commit ("Model-neutral Speculative Decoding", "The exactness transaction",
// steps 5-6): advance the position and the sampler slot by the emitted count
// and make the last emitted token the next anchor; on a device error nothing
// is committed and the round's outputs read -1.
__global__ void commit_kernel(const int32_t* __restrict__ seq_ids, int n_seq, int d, int n_slots,
                              const int32_t* __restrict__ n_acc_in,
                              int32_t* __restrict__ n_acc, int32_t* __restrict__ em,
                              int32_t* __restrict__ n_past, uint64_t* __restrict__ emit_idx,
                              int32_t* __restrict__ anchor, const uint32_t* __restrict__ err) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= n_seq) return;
  const int a = n_acc_in[s];
  int32_t* e = em + (size_t)s * (d + 1);
  const int slot = seq_ids[s];
  const bool bad = *err != 0u || a < 0 || a > d || slot < 0 || slot >= n_slots || e[a] < 0;
  if (bad) {
    n_acc[s] = -1;
    for (int i = 0; i <= d; i++) e[i] = -1;
    return;
  }
  n_acc[s] = a;
  n_past[slot] += a + 1;
  emit_idx[slot] += (uint64_t)(a + 1);
  anchor[slot] = e[a];
}

// Greedy accept and commit in one pass, for the verify round: one warp per
// sequence, lane i holding row i's argmax and draft i (d + 1 <= 32), so the
// first mismatch is one ballot and nothing waits on a chain of loads.  A
// programmatic dependent of the LM head: the drafts and the slot, which the
// round's target pass does not write, are read before the grid dependency
// resolves; the argmax, the error word and the state after.
static_assert(SPEC_MAX_NT <= 32, "one warp holds a sequence's d + 1 rows");
__global__ void accept_commit_greedy_kernel(const GreedyRoundArgs a) {
  const int lane = threadIdx.x & 31;
  const int s = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int d = a.d;
  const bool live = s < a.n_seq;
  int slot = 0, dtok = -1;
  if (live) {
    slot = a.seq_ids[s];
    if (lane < d) dtok = a.draft[(size_t)s * d + lane];
  }
  grid_dep_wait();
  if (!live) return;  // whole warps
  const int am = lane <= d ? a.argmax[(size_t)s * (d + 1) + lane] : -1;
  const unsigned match = __ballot_sync(0xffffffffu, lane < d && am == dtok);
  const int n = __ffs(~match) - 1;  // the first row whose argmax is not its draft, or d
  const int last = __shfl_sync(0xffffffffu, am, n);
  const bool bad = *a.err != 0u || slot < 0 || slot >= a.n_slots || last < 0;
  if (lane <= d) {
    int v = -1;
    if (!bad) v = lane < n ? dtok : (lane == n ? last : -1);
    a.emitted[(size_t)s * (d + 1) + lane] = v;
  }
  if (lane == 0) {
    if (bad) {
      a.n_acc[s] = -1;
    } else {
      a.n_acc[s] = n;
      a.n_past[slot] += n + 1;
      a.emit_idx[slot] += (uint64_t)(n + 1);
      a.anchor[slot] = last;
    }
  }
}

}  // namespace

size_t stoch_rows_needed(int n_seq, int d) { return (size_t)n_seq * (2 * (size_t)d + 1); }

void launch_accept_greedy(const int32_t* argmax, const int32_t* draft, int n_seq, int d,
                          int32_t* n_acc, int32_t* emitted, cudaStream_t st) {
  accept_greedy_kernel<<<(n_seq + 127) / 128, 128, 0, st>>>(argmax, draft, n_seq, d, n_acc,
                                                            emitted);
}

int launch_accept_stochastic(const float* p, const float* q, const int32_t* draft, int n_seq,
                             int d, int V, float T, uint64_t seed, const int32_t* seq_ids,
                             uint64_t* emit_idx, int emit_by_slot, int n_slots, int32_t* n_acc,
                             int32_t* emitted, const StochScratch& scr, uint32_t* err,
                             cudaStream_t st, bool p_keys_ready) {
  const size_t nrows = stoch_rows_needed(n_seq, d);
  const int nseg = st_segments(V);
  if (nrows * (size_t)nseg > (size_t)INT32_MAX || (size_t)n_seq * RS_CL > (size_t)INT32_MAX)
    return fail(SPEC_E_SHAPE, "stochastic accept: n_seq * (2d + 1) too large");
  if (nrows > scr.rows_cap || (size_t)n_seq > scr.seq_cap)
    return fail(SPEC_E_SHAPE, "stochastic accept: scratch too small");
  // the per-row maxima (keys) and sums are accumulated by atomics from zero
  // (the round's LM head has written the p rows' keys and zeroed the q rows')
  if (!p_keys_ready) CUDA_TRY(cudaMemsetAsync(scr.row_key, 0, nrows * sizeof(uint32_t), st));
  CUDA_TRY(cudaMemsetAsync(scr.row_sum, 0, nrows * sizeof(unsigned long long), st));
  const unsigned grid = (unsigned)(nrows * (size_t)nseg);
  const size_t qrows = (size_t)n_seq * d;
  if (!p_keys_ready)
    row_max_kernel<<<grid, ST_THREADS, 0, st>>>(p, q, d, V, nseg, 0, scr.row_key, err);
  else if (qrows > 0)
    row_max_kernel<<<(unsigned)(qrows * nseg), ST_THREADS, 0, st>>>(p, q, d, V, nseg, 1, scr.row_key,
                                                                     err);
  row_sum_kernel<<<grid, ST_THREADS, 0, st>>>(p, q, d, V, nseg, T, scr.row_key, scr.row_sum);
  decide_kernel<<<(n_seq + DC_WARPS - 1) / DC_WARPS, DC_WARPS * 32, 0, st>>>(
      p, q, draft, n_seq, d, V, T, seed, seq_ids, emit_idx, emit_by_slot, n_slots, scr.row_key,
      scr.row_sum, scr.decision, n_acc, emitted, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SPEC_E_CUDA, std::string("stochastic accept: ") + cudaGetErrorString(e));
  cudaLaunchConfig_t cfg = {};
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)(n_seq * RS_CL));
  cfg.blockDim = dim3(RS_THREADS);
  cfg.dynamicSmemBytes = 0;
  attr[0].val.clusterDim.x = RS_CL;
  e = cudaLaunchKernelEx(&cfg, resample_kernel, p, q, n_seq, d, V, T, (const uint32_t*)scr.row_key,
                         (const unsigned long long*)scr.row_sum, (const int4*)scr.decision, emitted,
                         err);
  if (e != cudaSuccess) return fail(SPEC_E_CUDA, std::string("stochastic accept: ") + cudaGetErrorString(e));
  return SPEC_OK;
}

void launch_commit(const int32_t* seq_ids, int n_seq, int d, int n_slots, const int32_t* n_acc_in,
                   int32_t* n_acc, int32_t* emitted, int32_t* n_past, uint64_t* emit_idx,
                   int32_t* anchor, const uint32_t* err, cudaStream_t st) {
  commit_kernel<<<(n_seq + 127) / 128, 128, 0, st>>>(seq_ids, n_seq, d, n_slots, n_acc_in, n_acc,
                                                     emitted, n_past, emit_idx, anchor, err);
}

void launch_accept_commit_greedy(const GreedyRoundArgs& a, cudaStream_t st) {
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = programmatic_launch() ? 1 : 0;
  cfg.gridDim = dim3((a.n_seq + 3) / 4);  // 4 sequences (warps) per CTA
  cfg.blockDim = dim3(128);
  cudaLaunchKernelEx(&cfg, accept_commit_greedy_kernel, a);
}

cudaError_t accept_commit_node_retarget(cudaGraphExec_t ex, cudaGraphNode_t node,
                                        const int32_t* draft, const int32_t* seq_ids,
                                        int32_t* n_acc, int32_t* emitted) {
  cudaKernelNodeParams p;
  cudaError_t e = cudaGraphKernelNodeGetParams(node, &p);
  if (e != cudaSuccess) return e;
  if (p.func != reinterpret_cast<void*>(accept_commit_greedy_kernel) || p.kernelParams == nullptr)
    return cudaErrorInvalidValue;
  GreedyRoundArgs a = *static_cast<const GreedyRoundArgs*>(p.kernelParams[0]);
  a.draft = draft;
  a.seq_ids = seq_ids;
  a.n_acc = n_acc;
  a.emitted = emitted;
  void* args[] = {&a};
  p.kernelParams = args;
  p.extra = nullptr;
  return cudaGraphExecKernelNodeSetParams(ex, node, &p);
}

void stoch_finalize(int n_seq, int d, int32_t* n_acc, int32_t* emitted, uint64_t* emit_idx,
                    const uint32_t* err, cudaStream_t st) {
  stoch_finalize_kernel<<<(n_seq + 127) / 128, 128, 0, st>>>(n_seq, d, n_acc, emitted, emit_idx,
                                                             err);
}

void accept_init_attrs() {}

// ---------------------------------------------------------------------------
// Allocation-free variant of the standalone stochastic accept.
//
// Its scratch (per-row max and integer-weight sums, per-sequence decisions,
// and an error word) lives in one fixed-size array in the module's global
// memory instead of memory from cudaMalloc.  Every GPU that loads this
// library keeps the array (about 64 KB) until the process exits.  Host code
// may not use the array's name as a device address; its address is looked up
// once per device with cudaGetSymbolAddress, on the first call made while
// that device is current.
// ---------------------------------------------------------------------------
constexpr int NOALLOC_MAX_ROWS = 4096;  // n_seq * (2d + 1)
constexpr int NOALLOC_MAX_SEQS = 1024;

struct NoAllocScratch {
  uint32_t row_key[NOALLOC_MAX_ROWS];
  unsigned long long row_sum[NOALLOC_MAX_ROWS];
  int4 decision[NOALLOC_MAX_SEQS];
  uint32_t err;
};

static __device__ __align__(256) NoAllocScratch g_noalloc_scratch;

static std::mutex g_noalloc_mu;
static std::vector<std::pair<int, NoAllocScratch*>> g_noalloc_ptrs;

// Device address of this device's copy of the array (set-up on first use).
static int noalloc_scratch(NoAllocScratch** out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  for (auto& e : g_noalloc_ptrs)
    if (e.first == dev) {
      *out = e.second;
      return SPEC_OK;
    }
  NoAllocScratch* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr)
    return fail(SPEC_E_CUDA, std::string("cudaGetSymbolAddress of the fixed scratch: ") +
                                 cudaGetErrorString(e));
  accept_init_attrs();  // the row-statistics kernel's shared-memory limit, once per device
  g_noalloc_ptrs.emplace_back(dev, p);
  *out = p;
  return SPEC_OK;
}

extern "C" int spec_accept_stochastic_noalloc(const float* p_logits, const float* q_logits,
                                              const int32_t* draft, int n_seq, int d, int V,
                                              float temperature, uint64_t seed,
                                              const int32_t* seq_ids, uint64_t* emit_idx,
                                              int32_t* n_acc, int32_t* emitted, void* stream) {
  if (p_logits == nullptr || seq_ids == nullptr || emit_idx == nullptr || n_acc == nullptr ||
      emitted == nullptr || (d > 0 && (draft == nullptr || q_logits == nullptr)))
    return fail(SPEC_E_INVALID, "null argument");
  if (n_seq < 1 || d < 0 || V < 1) return fail(SPEC_E_SHAPE, "n_seq >= 1, d >= 0, V >= 1 required");
  if (!(temperature > 0.0f) || !isfinite(temperature))
    return fail(SPEC_E_INVALID, "temperature must be finite and > 0");
  if (n_seq > NOALLOC_MAX_SEQS || (long long)n_seq * (2LL * d + 1) > NOALLOC_MAX_ROWS)
    return fail(SPEC_E_SHAPE,
                "spec_accept_stochastic_noalloc: n_seq * (2d + 1) must be <= 4096 and n_seq <= "
                "1024 (fixed scratch); use spec_accept_stochastic for larger batches");
  NoAllocScratch* sp = nullptr;
  int rc = noalloc_scratch(&sp);
  if (rc != SPEC_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: the error word must start at zero
  CUDA_TRY(cudaMemsetAsync(&sp->err, 0, sizeof(uint32_t), st));
  StochScratch scr;
  scr.row_key = sp->row_key;
  scr.row_sum = sp->row_sum;
  scr.decision = sp->decision;
  scr.rows_cap = NOALLOC_MAX_ROWS;
  scr.seq_cap = NOALLOC_MAX_SEQS;
  rc = launch_accept_stochastic(p_logits, q_logits, draft, n_seq, d, V, temperature, seed, seq_ids,
                                emit_idx, 0, 0, n_acc, emitted, scr, &sp->err, st);
  if (rc != SPEC_OK) return rc;
  stoch_finalize(n_seq, d, n_acc, emitted, emit_idx, &sp->err, st);
  CUDA_TRY(cudaGetLastError());
  return SPEC_OK;
}
