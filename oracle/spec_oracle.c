/*
 * spec_oracle.c -- plain, slow CPU oracle for the speculative-decoding
 * target-verification round.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code with the CUDA path.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fopenmp -shared -fPIC.
 * -ffp-contract=off matters: the sampler functions below are defined as a
 * sequence of individually rounded fp32 operations, and must not be fused.
 *
 * What each function follows (page title, section):
 *  - Model math (dequant, linear, RMSNorm, RoPE, attention, SwiGLU, LM head)
 *    is the plain definition of one target pass over nt = d+1 rows
 *    ("Speculative Decoding (D5-R) -- Plan", section 3 "Mechanism -- one
 *    round": one nt=d+1 forward whose rows are the next token plus the d
 *    drafted candidates at contiguous positions).  Accumulation in fp64.
 *  - Greedy accept ("Speculative Decoding (D5-R) -- Plan", section 3, "accept
 *    while equal to the drafted token; always emit >= 1 token"; and
 *    "Model-neutral Speculative Decoding", "The exactness transaction",
 *    steps 4-6).
 *  - Strict rejection sampling ("DFlash and DSpark Speculative Decoding",
 *    "How DSpark Works" and "Notes": lossless under the strict rejection
 *    sampler), with the sampler-advance rule of "Model-neutral Speculative
 *    Decoding", "The exactness transaction" (the target sampler advances once
 *    per emitted sample, never for a rejected suffix).  The target and draft
 *    probabilities are defined as integer weights (see int_weight below) so
 *    that every accept/resample decision is an exact integer comparison.
 *  - Philox4x32-10 from Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers:
 *    As Easy as 1, 2, 3" (SC'11).  Pinned against cuRAND's host-side
 *    PHILOX4_32_10 generator (a library routine run on the CPU), which
 *    exercises the key schedule and counter words 0-2; counter word 3 is
 *    pinned only at the value 0, which is the only value the target sampler
 *    uses.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef unsigned __int128 u128;

/* ------------------------------------------------------------------------ */
/* fp16 <-> wider, by the compiler's IEEE binary16 type (round to nearest    */
/* even, one rounding from double).                                          */
/* ------------------------------------------------------------------------ */
static double h2d(uint16_t h) {
  _Float16 f;
  memcpy(&f, &h, 2);
  return (double)f;
}
static uint16_t d2h(double x) {
  _Float16 f = (_Float16)x;
  uint16_t h;
  memcpy(&h, &f, 2);
  return h;
}

void oracle_f64_to_f16(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = d2h(x[i]);
}
void oracle_f16_to_f64(const uint16_t* h, int64_t n, double* out) {
  for (int64_t i = 0; i < n; i++) out[i] = h2d(h[i]);
}

/* ------------------------------------------------------------------------ */
/* Block-quantised weights, canonical planes.                                */
/*   Q4: qs[n][b][16] bytes; byte j holds element j (low nibble) and element */
/*       j+16 (high nibble) of block b, stored as u = q + 8, q in [-8, 7].   */
/*   Q6: low 4 bits of u = q + 32 in qs (same nibble order as Q4); high 2    */
/*       bits in qh[n][b][8]: element j at bits 2*(j%4) of byte j/4.         */
/*   Q8: qs[n][b][32] bytes; byte j is element j of block b as a two's-     */
/*       complement int8, q in [-128, 127] (the q8_0 element order).        */
/*   scales[n][b] fp16.  w[n][k] = float(scale) * float(q), exact in fp32.   */
/* ------------------------------------------------------------------------ */
static int q_elem(int qtype, const uint8_t* qs, const uint8_t* qh, int64_t n,
                  int64_t nb, int64_t k) {
  int64_t b = k / 32;
  int j = (int)(k % 32);
  if (qtype == 8) {
    int v = qs[(n * nb + b) * 32 + j];
    return v >= 128 ? v - 256 : v;
  }
  uint8_t byte = qs[(n * nb + b) * 16 + (j % 16)];
  int lo = (j < 16) ? (byte & 0xF) : (byte >> 4);
  if (qtype == 4) return lo - 8;
  uint8_t hb = qh[(n * nb + b) * 8 + j / 4];
  int hi = (hb >> (2 * (j % 4))) & 3;
  return (lo | (hi << 4)) - 32;
}

/* Dequantise rows [n0, n0+rows) to fp32 (exact). */
void oracle_dequant(int qtype, const uint8_t* qs, const uint8_t* qh,
                    const uint16_t* scales, int64_t N, int64_t K, int64_t n0,
                    int64_t rows, float* w) {
  int64_t nb = K / 32;
  for (int64_t i = 0; i < rows; i++) {
    int64_t n = n0 + i;
    for (int64_t k = 0; k < K; k++) {
      float s = (float)h2d(scales[n * nb + k / 32]);
      w[i * K + k] = s * (float)q_elem(qtype, qs, qh, n, nb, k);
    }
  }
  (void)N;
}

/* y[r][n] = (float) sum_k (double)w[n][k] * (double)x[r][k], sequential k.   */
void oracle_linear(int qtype, const uint8_t* qs, const uint8_t* qh,
                   const uint16_t* scales, int64_t N, int64_t K,
                   const uint16_t* x, int64_t R, float* y) {
  int64_t nb = K / 32;
  double* xd = (double*)malloc(sizeof(double) * R * K);
  for (int64_t i = 0; i < R * K; i++) xd[i] = h2d(x[i]);
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * K);
#pragma omp for schedule(static)
    for (int64_t n = 0; n < N; n++) {
      for (int64_t k = 0; k < K; k++) {
        float s = (float)h2d(scales[n * nb + k / 32]);
        w[k] = (double)(s * (float)q_elem(qtype, qs, qh, n, nb, k));
      }
      for (int64_t r = 0; r < R; r++) {
        double acc = 0.0;
        const double* xr = xd + r * K;
        for (int64_t k = 0; k < K; k++) acc += w[k] * xr[k];
        y[r * N + n] = (float)acc;
      }
    }
    free(w);
  }
  free(xd);
}

/* ------------------------------------------------------------------------ */
/* RMSNorm: out = fp16( h * gamma / sqrt(mean(h^2) + eps) ), fp64 inside.    */
/* ------------------------------------------------------------------------ */
void oracle_rmsnorm(const float* h, const float* gamma, int64_t R, int64_t H,
                    double eps, uint16_t* out) {
  for (int64_t r = 0; r < R; r++) {
    double ss = 0.0;
    for (int64_t i = 0; i < H; i++) ss += (double)h[r * H + i] * (double)h[r * H + i];
    double inv = 1.0 / sqrt(ss / (double)H + eps);
    for (int64_t i = 0; i < H; i++)
      out[r * H + i] = d2h((double)h[r * H + i] * inv * (double)gamma[i]);
  }
}

/* ------------------------------------------------------------------------ */
/* Rotate-half rotary embedding of one head vector at absolute position pos:*/
/* pairs (i, i + hd/2) rotated by pos * theta^(-2i/hd).  fp64.               */
/* ------------------------------------------------------------------------ */
static void rope_head(const double* x, double* y, int hd, int64_t pos, double theta) {
  int half = hd / 2;
  for (int i = 0; i < half; i++) {
    double f = pow(theta, -2.0 * (double)i / (double)hd);
    double a = (double)pos * f;
    double c = cos(a), s = sin(a);
    y[i] = x[i] * c - x[i + half] * s;
    y[i + half] = x[i + half] * c + x[i] * s;
  }
}

void oracle_rope(const float* x, int64_t rows, int hd, const int64_t* pos,
                 double theta, uint16_t* out) {
  double* xi = (double*)malloc(sizeof(double) * hd);
  double* yo = (double*)malloc(sizeof(double) * hd);
  for (int64_t r = 0; r < rows; r++) {
    for (int i = 0; i < hd; i++) xi[i] = (double)x[r * hd + i];
    rope_head(xi, yo, hd, pos[r], theta);
    for (int i = 0; i < hd; i++) out[r * hd + i] = d2h(yo[i]);
  }
  free(xi);
  free(yo);
}

/* ------------------------------------------------------------------------ */
/* Causal GQA attention for one query head vector q[hd] (fp16) at absolute  */
/* position P against a cache k/v[pos][hd] (fp16): positions 0..P.  fp64.   */
/* ------------------------------------------------------------------------ */
static void attend_one(const uint16_t* q, const uint16_t* kc, const uint16_t* vc,
                       int hd, int64_t P, double* sc, double* o) {
  double scale = 1.0 / sqrt((double)hd);
  double m = -INFINITY;
  for (int64_t j = 0; j <= P; j++) {
    double s = 0.0;
    for (int d = 0; d < hd; d++) s += h2d(q[d]) * h2d(kc[j * hd + d]);
    sc[j] = s * scale;
    if (sc[j] > m) m = sc[j];
  }
  double l = 0.0;
  for (int d = 0; d < hd; d++) o[d] = 0.0;
  for (int64_t j = 0; j <= P; j++) {
    double p = exp(sc[j] - m);
    l += p;
    for (int d = 0; d < hd; d++) o[d] += p * h2d(vc[j * hd + d]);
  }
  for (int d = 0; d < hd; d++) o[d] /= l;
}

/* q: [rows][nq][hd]; kcache/vcache: [nkv][max_ctx][hd] of ONE sequence;     */
/* pos[rows] absolute positions; out: [rows][nq][hd] fp16.                   */
void oracle_attention(const uint16_t* q, int64_t rows, int nq, int nkv, int hd,
                      const uint16_t* kcache, const uint16_t* vcache,
                      int64_t max_ctx, const int64_t* pos, uint16_t* out) {
  int group = nq / nkv;
#pragma omp parallel
  {
    double* sc = (double*)malloc(sizeof(double) * max_ctx);
    double* o = (double*)malloc(sizeof(double) * hd);
#pragma omp for schedule(static) collapse(2)
    for (int64_t r = 0; r < rows; r++) {
      for (int h = 0; h < nq; h++) {
        int kvh = h / group;
        attend_one(q + (r * nq + h) * hd, kcache + (int64_t)kvh * max_ctx * hd,
                   vcache + (int64_t)kvh * max_ctx * hd, hd, pos[r], sc, o);
        for (int d = 0; d < hd; d++) out[(r * nq + h) * hd + d] = d2h(o[d]);
      }
    }
    free(sc);
    free(o);
  }
}

/* SwiGLU: out = fp16( silu(g) * u ), silu(g) = g / (1 + exp(-g)).  fp64.    */
void oracle_swiglu(const float* g, const float* u, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; i++) {
    double gv = (double)g[i];
    out[i] = d2h(gv / (1.0 + exp(-gv)) * (double)u[i]);
  }
}

/* ------------------------------------------------------------------------ */
/* One target pass over the verify rows of n_seq sequences.                  */
/*   tokens[s][nt]: row 0 is the anchor, rows 1..d the drafted tokens.       */
/*   Row i of sequence s sits at absolute position n_past[s] + i.            */
/*   kcache/vcache: [L][n_seq][nkv][max_ctx][hd] fp16 (in/out: the pass      */
/*   writes the new k/v rows, "positions are data").                         */
/*   Weights: per-layer canonical planes; wqkv rows are [q heads | k heads | */
/*   v heads], wgu rows are [gate ; up].                                     */
/*   logits: [n_seq*nt][V] fp32.                                             */
/* ------------------------------------------------------------------------ */
typedef struct {
  int qtype;
  const uint8_t* qs;
  const uint8_t* qh;
  const uint16_t* scales;
  int64_t N, K;
} oracle_qw;

typedef struct {
  int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  int64_t max_ctx;
  double rms_eps, rope_theta;
  int use_rope;
} oracle_desc;

static void lin(const oracle_qw* w, const uint16_t* x, int64_t R, float* y) {
  oracle_linear(w->qtype, w->qs, w->qh, w->scales, w->N, w->K, x, R, y);
}

void oracle_forward(const oracle_desc* D, const uint16_t* embed,
                    const float* norm_w, const oracle_qw* wqkv,
                    const oracle_qw* wo, const oracle_qw* wgu,
                    const oracle_qw* wd, const oracle_qw* lm, int n_seq, int nt,
                    const int32_t* tokens, const int64_t* n_past,
                    uint16_t* kcache, uint16_t* vcache, float* logits) {
  const int64_t H = D->hidden, hd = D->head_dim, nq = D->n_q_heads,
                nkv = D->n_kv_heads, F = D->ffn;
  const int64_t R = (int64_t)n_seq * nt;
  const int64_t nqkv = (nq + 2 * nkv) * hd;
  const int64_t seq_stride = nkv * D->max_ctx * hd;
  float* h = (float*)malloc(sizeof(float) * R * H);
  uint16_t* x = (uint16_t*)malloc(sizeof(uint16_t) * R * (F > H ? F : H) +
                                  sizeof(uint16_t) * R * nq * hd);
  float* big = (float*)malloc(sizeof(float) * R * (2 * F > nqkv ? 2 * F : nqkv));
  uint16_t* qh16 = (uint16_t*)malloc(sizeof(uint16_t) * R * nq * hd);
  uint16_t* ao = (uint16_t*)malloc(sizeof(uint16_t) * R * nq * hd);
  float* o = (float*)malloc(sizeof(float) * R * H);
  int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * R);
  float* g = (float*)malloc(sizeof(float) * R * F);
  float* u = (float*)malloc(sizeof(float) * R * F);
  double* tmp_in = (double*)malloc(sizeof(double) * hd);
  double* tmp_out = (double*)malloc(sizeof(double) * hd);

  for (int s = 0; s < n_seq; s++)
    for (int i = 0; i < nt; i++) pos[(int64_t)s * nt + i] = n_past[s] + i;
  /* embedding gather (exact fp16 -> fp32) */
  for (int64_t r = 0; r < R; r++)
    for (int64_t i = 0; i < H; i++)
      h[r * H + i] = (float)h2d(embed[(int64_t)tokens[r] * H + i]);

  for (int l = 0; l < D->n_layers; l++) {
    uint16_t* kl = kcache + (int64_t)l * n_seq * seq_stride;
    uint16_t* vl = vcache + (int64_t)l * n_seq * seq_stride;
    /* attention block */
    oracle_rmsnorm(h, norm_w + (int64_t)(2 * l) * H, R, H, D->rms_eps, x);
    lin(&wqkv[l], x, R, big);
    for (int64_t r = 0; r < R; r++) {
      int s = (int)(r / nt);
      const float* row = big + r * nqkv;
      for (int64_t hh = 0; hh < nq + 2 * nkv; hh++) {
        const float* src = row + hh * hd;
        for (int d = 0; d < hd; d++) tmp_in[d] = (double)src[d];
        if (D->use_rope && hh < nq + nkv)
          rope_head(tmp_in, tmp_out, (int)hd, pos[r], D->rope_theta);
        else
          memcpy(tmp_out, tmp_in, sizeof(double) * hd);
        if (hh < nq) {
          for (int d = 0; d < hd; d++) qh16[(r * nq + hh) * hd + d] = d2h(tmp_out[d]);
        } else {
          int64_t kvh = (hh < nq + nkv) ? hh - nq : hh - nq - nkv;
          uint16_t* dst = ((hh < nq + nkv) ? kl : vl) + s * seq_stride +
                          (kvh * D->max_ctx + pos[r]) * hd;
          for (int d = 0; d < hd; d++) dst[d] = d2h(tmp_out[d]);
        }
      }
    }
    for (int s = 0; s < n_seq; s++)
      oracle_attention(qh16 + (int64_t)s * nt * nq * hd, nt, (int)nq, (int)nkv,
                       (int)hd, kl + s * seq_stride, vl + s * seq_stride,
                       D->max_ctx, pos + (int64_t)s * nt,
                       ao + (int64_t)s * nt * nq * hd);
    lin(&wo[l], ao, R, o);
    for (int64_t i = 0; i < R * H; i++) h[i] = (float)((double)h[i] + (double)o[i]);
    /* feed-forward block */
    oracle_rmsnorm(h, norm_w + (int64_t)(2 * l + 1) * H, R, H, D->rms_eps, x);
    lin(&wgu[l], x, R, big);
    for (int64_t r = 0; r < R; r++) {
      memcpy(g + r * F, big + r * 2 * F, sizeof(float) * F);
      memcpy(u + r * F, big + r * 2 * F + F, sizeof(float) * F);
    }
    oracle_swiglu(g, u, R * F, x);
    lin(&wd[l], x, R, o);
    for (int64_t i = 0; i < R * H; i++) h[i] = (float)((double)h[i] + (double)o[i]);
  }
  oracle_rmsnorm(h, norm_w + (int64_t)(2 * D->n_layers) * H, R, H, D->rms_eps, x);
  lin(lm, x, R, logits);

  free(h); free(x); free(big); free(qh16); free(ao); free(o); free(pos);
  free(g); free(u); free(tmp_in); free(tmp_out);
}

/* ------------------------------------------------------------------------ */
/* Greedy accept.                                                            */
/* argmax: lowest index among the maximal values; NaN -> returns -1.         */
/* ------------------------------------------------------------------------ */
int64_t oracle_argmax(const float* row, int64_t V) {
  int64_t best = 0;
  for (int64_t v = 0; v < V; v++) {
    if (isnan(row[v])) return -1;
    if (row[v] > row[best]) best = v;
  }
  return best;
}

/* argmax[s][d+1], draft[s][d] -> n_acc[s], emitted[s][d+1] (unused slots = -1).
 * a = number of leading i < d with argmax[i] == draft[i]; emitted is
 * draft[0..a-1] followed by argmax[a] (the correction, or the bonus when a == d).
 * Returns 0, or -1 if any argmax is negative (NaN row). */
int oracle_accept_greedy(const int32_t* argmax, const int32_t* draft, int n_seq,
                         int d, int32_t* n_acc, int32_t* emitted) {
  for (int s = 0; s < n_seq; s++) {
    const int32_t* am = argmax + (int64_t)s * (d + 1);
    const int32_t* dr = draft + (int64_t)s * d;
    int32_t* em = emitted + (int64_t)s * (d + 1);
    for (int i = 0; i <= d; i++) em[i] = -1;
    for (int i = 0; i <= d; i++)
      if (am[i] < 0) return -1;
    int a = 0;
    while (a < d && am[a] == dr[a]) {
      em[a] = dr[a];
      a++;
    }
    em[a] = am[a];
    n_acc[s] = a;
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Strict rejection sampling with integer weights.                           */
/* ------------------------------------------------------------------------ */

/* exp_own(x), x <= 0, fp32.  Cody-Waite range reduction with a two-part    */
/* ln 2, then a degree-7 Taylor polynomial (coefficients 1/k! rounded to     */
/* fp32) in Horner form.  Every operation is one rounded fp32 multiply or    */
/* add (no fused multiply-add), so the function is reproducible exactly by   */
/* any IEEE-754 binary32 implementation doing the same operations.           */
/* Returns the mantissa part p and the exponent n with exp(x) ~= p * 2^n.    */
static const float EXP_LOG2E = 0x1.715476p+0f;  /* fl32(1 / ln 2) */
static const float EXP_LN2_HI = 0x1.62e4p-1f;   /* ln 2 to 12 bits: n * LN2_HI exact */
static const float EXP_LN2_LO = 0x1.7f7d1cp-20f; /* fl32(ln 2 - LN2_HI) */
static const float EXP_C[8] = {                  /* fl32(1 / k!) */
    0x1p+0f,        0x1p+0f,         0x1p-1f,         0x1.555556p-3f,
    0x1.555556p-5f, 0x1.111112p-7f,  0x1.6c16c2p-10f, 0x1.a01a02p-13f};

static float f32_from_bits(uint32_t b) {
  float f;
  memcpy(&f, &b, 4);
  return f;
}

static void exp_parts(float x, float* p_out, int* n_out) {
  volatile float t = x * EXP_LOG2E;
  float n = rintf(t);
  volatile float a = n * EXP_LN2_HI;
  volatile float r = x - a;
  volatile float b = n * EXP_LN2_LO;
  r = r - b;
  float p = EXP_C[7];
  for (int k = 6; k >= 0; k--) {
    volatile float m = p * r;
    p = m + EXP_C[k];
  }
  *p_out = p;
  *n_out = (int)n;
}

/* exp_own as a float (for the pins); x < -87 returns 0. */
float oracle_exp_own(float x) {
  if (!(x >= -87.0f)) return 0.0f;
  float p;
  int n;
  exp_parts(x, &p, &n);
  /* scale by 2^n through exponent bits; n in [-126, 0] here */
  return p * f32_from_bits((uint32_t)(n + 127) << 23);
}

/* Integer weight W = floor(exp_own(x) * 2^32) for x = z - max(z) <= 0.
 * The product p * 2^(n+32) is exact in fp32 (power-of-two scale, no
 * overflow), so W is the exact floor.  W of the row maximum is 2^32. */
uint64_t oracle_int_weight(float x) {
  if (!(x >= -87.0f)) return 0;
  float p;
  int n;
  exp_parts(x, &p, &n);
  if (n + 32 < 0) return 0;
  float v = p * f32_from_bits((uint32_t)(n + 32 + 127) << 23);
  return (uint64_t)v; /* truncation == floor for v >= 0 */
}

/* Row statistics on temperature-scaled logits: z = l / T (one rounded fp32
 * division), m = max z, W_v = int_weight(z_v - m), S = sum W_v.
 * Returns -1 if a logit is not finite. */
int oracle_row_weights(const float* logits, int64_t V, float T, uint64_t* W,
                       uint64_t* S_out) {
  float m = -INFINITY;
  for (int64_t v = 0; v < V; v++) {
    if (!isfinite(logits[v])) return -1;
    volatile float z = logits[v] / T;
    if (z > m) m = z;
  }
  uint64_t S = 0;
  for (int64_t v = 0; v < V; v++) {
    volatile float z = logits[v] / T;
    volatile float x = z - m;
    W[v] = oracle_int_weight(x);
    S += W[v];
  }
  *S_out = S;
  return 0;
}

/* Philox4x32-10 (Salmon et al., SC'11): 10 rounds of
 *   (c0,c1,c2,c3) -> (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0))
 * with the key bumped by the Weyl constants between rounds. */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                          uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; round++) {
    if (round > 0) {
      k0 += W0;
      k1 += W1;
    }
    uint64_t p0 = (uint64_t)M0 * c0, p1 = (uint64_t)M1 * c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The sampler's uniform draw for emitted slot j of sequence seq_id:
 * key = (seed lo, seed hi), counter = (j lo, j hi, seq_id, domain).
 * Domain 0 = target sampler, 1 = a harness's draft sampler. */
void oracle_uniforms(uint64_t seed, uint64_t slot, uint32_t seq_id,
                     uint32_t domain, uint32_t out[4]) {
  uint32_t ctr[4] = {(uint32_t)slot, (uint32_t)(slot >> 32), seq_id, domain};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  oracle_philox4x32_10(ctr, key, out);
}

/* Accept test for draft x:  u < p_x / q_x  with u = U1 / 2^32, i.e.
 *   U1 * Wq_x * S  <  2^32 * W_x * Sq   (exact, 128-bit).
 * If Wq_x == 0: accept iff W_x > 0. */
int oracle_accept_decide(uint64_t Wx, uint64_t S, uint64_t Wqx, uint64_t Sq,
                         uint32_t U1) {
  if (Wqx == 0) return Wx > 0;
  u128 lhs = (u128)U1 * (u128)Wqx * (u128)S;
  u128 rhs = ((u128)Wx << 32) * (u128)Sq;
  return lhs < rhs;
}

/* Pick from cumulative integer masses: the smallest v with
 * sum_{u<=v} mass_u > t, where t = floor(U2 * total / 2^32). */
static u128 scaled_threshold(uint32_t U2, u128 total) {
  u128 hi = total >> 32, lo = total & 0xFFFFFFFFu;
  return (u128)U2 * hi + (((u128)U2 * lo) >> 32);
}

/* Resample after a rejection from norm(max(0, p - q)):
 * R_v = max(0, W_v*Sq - Wq_v*S), 128-bit. */
int64_t oracle_residual_pick(const uint64_t* W, uint64_t S, const uint64_t* Wq,
                             uint64_t Sq, int64_t V, uint32_t U2) {
  u128 total = 0;
  for (int64_t v = 0; v < V; v++) {
    u128 a = (u128)W[v] * Sq, b = (u128)Wq[v] * S;
    if (a > b) total += a - b;
  }
  if (total == 0) return -1;
  u128 t = scaled_threshold(U2, total);
  u128 cum = 0;
  for (int64_t v = 0; v < V; v++) {
    u128 a = (u128)W[v] * Sq, b = (u128)Wq[v] * S;
    if (a > b) cum += a - b;
    if (cum > t) return v;
  }
  return -1;
}

/* Sample from p itself (bonus token after a fully accepted block, or the
 * plain autoregressive sampler). */
int64_t oracle_weight_pick(const uint64_t* W, uint64_t S, int64_t V, uint32_t U2) {
  u128 t = scaled_threshold(U2, (u128)S);
  u128 cum = 0;
  for (int64_t v = 0; v < V; v++) {
    cum += W[v];
    if (cum > t) return v;
  }
  return -1;
}

/* Full stochastic accept for n_seq sequences, sequentially.
 * p_logits[s][d+1][V], q_logits[s][d][V] (draft distribution that produced
 * draft[s][i] for slot i), temperature T applied to both.
 * emit_idx[s] (in/out): index of the next emitted token of sequence s; slot
 * emit_idx+i uses Philox counter (emit_idx+i, seq_ids[s], 0).  Rows after
 * the first rejection are never read.  Returns 0, or -1 on a non-finite
 * logit or an out-of-range draft id (then nothing is updated for that
 * sequence and later ones). */
int oracle_accept_stochastic(const float* p_logits, const float* q_logits,
                             const int32_t* draft, int n_seq, int d, int64_t V,
                             float T, uint64_t seed, const int32_t* seq_ids,
                             uint64_t* emit_idx, int32_t* n_acc,
                             int32_t* emitted) {
  uint64_t* W = (uint64_t*)malloc(sizeof(uint64_t) * V);
  uint64_t* Wq = (uint64_t*)malloc(sizeof(uint64_t) * V);
  int rc = 0;
  for (int s = 0; s < n_seq && rc == 0; s++) {
    const float* P = p_logits + (int64_t)s * (d + 1) * V;
    const float* Q = q_logits + (int64_t)s * d * V;
    int32_t* em = emitted + (int64_t)s * (d + 1);
    for (int i = 0; i <= d; i++) em[i] = -1;
    int a = 0;
    int done = 0;
    for (int i = 0; i < d; i++) {
      int32_t x = draft[(int64_t)s * d + i];
      uint64_t S, Sq;
      uint32_t U[4];
      if (x < 0 || x >= V) { rc = -1; break; }
      if (oracle_row_weights(P + (int64_t)i * V, V, T, W, &S) ||
          oracle_row_weights(Q + (int64_t)i * V, V, T, Wq, &Sq)) { rc = -1; break; }
      oracle_uniforms(seed, emit_idx[s] + (uint64_t)i, (uint32_t)seq_ids[s], 0, U);
      if (oracle_accept_decide(W[x], S, Wq[x], Sq, U[0])) {
        em[i] = x;
        a = i + 1;
        continue;
      }
      int64_t v = oracle_residual_pick(W, S, Wq, Sq, V, U[1]);
      if (v < 0) { rc = -1; break; }
      em[i] = (int32_t)v;
      a = i;
      done = 1;
      break;
    }
    if (rc) break;
    if (!done) {
      uint64_t S;
      uint32_t U[4];
      if (oracle_row_weights(P + (int64_t)d * V, V, T, W, &S)) { rc = -1; break; }
      oracle_uniforms(seed, emit_idx[s] + (uint64_t)d, (uint32_t)seq_ids[s], 0, U);
      em[d] = (int32_t)oracle_weight_pick(W, S, V, U[1]);
      a = d;
    }
    n_acc[s] = a;
    emit_idx[s] += (uint64_t)(a + 1);
  }
  free(W);
  free(Wq);
  return rc;
}
