// depth.cu -- the adaptive draft-depth controller: host code only, no GPU
// work.  Source: "Speculative Decoding (D5-R) -- Plan", status notes, which
// name only the ingredients of the page's controller (smoothed acceptance
// estimates, a short window of measured round costs, hysteresis, trying
// depths that have no measurement yet, an upper cap on d).  The concrete
// rules below are this library's reading of those ingredients.
//
// Rules (the header states them for callers):
//  * position i = 1..d_max holds decayed Beta counts (a_i, b_i); a round at
//    depth d where a sequence accepted n drafts adds a_i += 1 for i <= n and,
//    if n < d, b_{n+1} += 1; every count is first multiplied by `decay`;
//  * p_i = (a_i + prior_accept) / (a_i + b_i + prior_accept + prior_reject);
//  * E(d) = sum_{k=0..d} prod_{i<=k} p_i; c(d) = min of the depth's last
//    `cost_window` round times; r(d) = E(d) / c(d);
//  * while a depth in [d_min, d_max] has no round time, the deepest such
//    depth is next; otherwise the smallest depth of maximal r replaces the
//    current one if its r exceeds the current r by the factor 1 + hysteresis.
// This file is compiled without floating-point contraction, so every
// expression is rounded operation by operation (the same doubles as any
// other IEEE implementation of these rules).
#include <cmath>
#include <new>
#include <string>
#include <vector>

#include "common.cuh"

struct spec_depth_ctl {
  spec_depth_params prm;
  std::vector<double> acc, rej;                // [d_max + 1], index 0 unused
  std::vector<std::vector<double>> costs;      // per depth, newest last
  int32_t d_cur;
};

namespace {

double p_of(const spec_depth_ctl* c, int i) {
  const double a = c->acc[i], b = c->rej[i];
  return (a + c->prm.prior_accept) / (a + b + c->prm.prior_accept + c->prm.prior_reject);
}

double expected_tokens(const spec_depth_ctl* c, int d) {
  double e = 1.0, prod = 1.0;
  for (int i = 1; i <= d; i++) {
    prod = prod * p_of(c, i);
    e = e + prod;
  }
  return e;
}

bool seen(const spec_depth_ctl* c, int d) { return !c->costs[d].empty(); }

double rate(const spec_depth_ctl* c, int d) {
  if (!seen(c, d)) return INFINITY;
  double m = c->costs[d][0];
  for (double v : c->costs[d]) m = v < m ? v : m;
  return expected_tokens(c, d) / m;
}

int32_t choose(const spec_depth_ctl* c) {
  const int lo = c->prm.d_min, hi = c->prm.d_max;
  for (int d = hi; d >= lo; d--)
    if (!seen(c, d)) return d;
  int best = lo;
  double best_r = rate(c, lo);
  for (int d = lo + 1; d <= hi; d++) {
    const double r = rate(c, d);
    if (r > best_r) {
      best = d;
      best_r = r;
    }
  }
  if (best != c->d_cur && best_r > (1.0 + c->prm.hysteresis) * rate(c, c->d_cur)) return best;
  return c->d_cur;
}

bool params_ok(const spec_depth_params& p) {
  return p.d_min >= 0 && p.d_min <= p.d_max && p.d_max <= SPEC_MAX_NT - 1 &&
         p.prior_accept >= 0.0 && p.prior_reject >= 0.0 &&
         p.prior_accept + p.prior_reject > 0.0 && std::isfinite(p.prior_accept) &&
         std::isfinite(p.prior_reject) && p.decay > 0.0 && p.decay <= 1.0 &&
         p.hysteresis >= 0.0 && std::isfinite(p.hysteresis) && p.cost_window >= 1 &&
         p.cost_window <= 64;
}

}  // namespace

extern "C" void spec_depth_params_default(spec_depth_params* p) {
  if (p == nullptr) return;
  p->d_min = 1;
  p->d_max = 7;
  p->prior_accept = 1.0;
  p->prior_reject = 0.0;
  p->decay = 0.95;
  p->hysteresis = 0.10;
  p->cost_window = 4;
}

extern "C" int spec_depth_ctl_create(const spec_depth_params* params, spec_depth_ctl** out) {
  if (out == nullptr) return fail(SPEC_E_INVALID, "null argument");
  *out = nullptr;
  spec_depth_params p;
  if (params != nullptr) {
    p = *params;
  } else {
    spec_depth_params_default(&p);
  }
  if (!params_ok(p)) return fail(SPEC_E_INVALID, "depth controller: parameters out of range");
  spec_depth_ctl* c = new (std::nothrow) spec_depth_ctl;
  if (c == nullptr) return fail(SPEC_E_OOM, "depth controller");
  c->prm = p;
  c->acc.assign(p.d_max + 1, 0.0);
  c->rej.assign(p.d_max + 1, 0.0);
  c->costs.assign(p.d_max + 1, std::vector<double>());
  c->d_cur = p.d_max;
  *out = c;
  return SPEC_OK;
}

extern "C" int spec_depth_ctl_destroy(spec_depth_ctl* c) {
  delete c;
  return SPEC_OK;
}

extern "C" int spec_depth_ctl_next(const spec_depth_ctl* c, int32_t* d) {
  if (c == nullptr || d == nullptr) return fail(SPEC_E_INVALID, "null argument");
  *d = c->d_cur;
  return SPEC_OK;
}

extern "C" int spec_depth_ctl_observe(spec_depth_ctl* c, int32_t d, int32_t n_seq,
                                      const int32_t* n_acc, double round_seconds,
                                      int32_t* next_d) {
  if (c == nullptr || (n_seq > 0 && n_acc == nullptr))
    return fail(SPEC_E_INVALID, "null argument");
  if (d < c->prm.d_min || d > c->prm.d_max || n_seq < 0)
    return fail(SPEC_E_SHAPE, "depth controller: d outside [d_min, d_max] or n_seq < 0");
  if (!(round_seconds > 0.0) || !std::isfinite(round_seconds))
    return fail(SPEC_E_INVALID, "depth controller: round time must be finite and > 0");
  for (int i = 1; i <= c->prm.d_max; i++) {
    c->acc[i] = c->acc[i] * c->prm.decay;
    c->rej[i] = c->rej[i] * c->prm.decay;
  }
  for (int s = 0; s < n_seq; s++) {
    const int n = n_acc[s];
    if (n < 0) continue;  // a failed sequence observes nothing
    const int m = n < d ? n : d;
    for (int i = 1; i <= m; i++) c->acc[i] = c->acc[i] + 1.0;
    if (n < d) c->rej[n + 1] = c->rej[n + 1] + 1.0;
  }
  std::vector<double>& w = c->costs[d];
  w.push_back(round_seconds);
  if ((int)w.size() > c->prm.cost_window) w.erase(w.begin());
  c->d_cur = choose(c);
  if (next_d != nullptr) *next_d = c->d_cur;
  return SPEC_OK;
}

extern "C" int spec_depth_ctl_estimates(const spec_depth_ctl* c, double* p, double* r) {
  if (c == nullptr) return fail(SPEC_E_INVALID, "null argument");
  const int hi = c->prm.d_max;
  if (p != nullptr) {
    p[0] = 1.0;
    for (int i = 1; i <= hi; i++) p[i] = p_of(c, i);
  }
  if (r != nullptr)
    for (int d = 0; d <= hi; d++) r[d] = d < c->prm.d_min ? 0.0 : rate(c, d);
  return SPEC_OK;
}
