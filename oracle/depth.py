"""Oracle of the adaptive draft-depth controller (test infrastructure: only
tests, __graft_entry__.smoke() and bench.py's cpu_baseline leg use oracle/).

"Speculative Decoding (D5-R) -- Plan", status notes (adaptive draft depth):
the depth of each round is chosen from beta-smoothed per-depth acceptance
estimates and min-of-4 round-cost windows, with a 10% switch hysteresis and
optimism for depths not yet seen, capped at d = 7 by the identity boundary.
The page gives the ingredients only; the plainest reading, written out step
by step (every float is an IEEE double, every expression evaluated left to
right with one rounding per operation):

* Acceptance.  Position i (1..d_max) holds decayed Beta counts (a_i, b_i).
  A round at depth d in which a sequence accepted n drafts observes
  positions 1..min(n+1, d): positions 1..n accepted (a_i += 1), position
  n+1 rejected (b_{n+1} += 1) when n < d.  Before a round's observations
  are added, every count is multiplied by the decay factor.  The estimate
  is p_i = (a_i + prior_accept) / (a_i + b_i + prior_accept + prior_reject);
  with prior_reject = 0 a position never observed has p_i = 1 (optimism).
* Expected emitted tokens at depth d: E(d) = sum_{k=0..d} prod_{i<=k} p_i
  (the accepted prefix plus the one correction/bonus token).
* Cost.  Each depth keeps its last `cost_window` round times; c(d) is their
  minimum.  A depth with no round time yet is unseen.
* Choice.  If an unseen depth exists in [d_min, d_max], the deepest unseen
  depth is chosen (its rate is taken as +infinity: optimism).  Otherwise
  r(d) = E(d) / c(d) and d* = the smallest depth of maximal r; the
  controller moves from its current depth d_cur to d* only if
  r(d*) > (1 + hysteresis) * r(d_cur).
* The first round runs at d_max.
"""
from __future__ import annotations

import math

DEFAULTS = dict(d_min=1, d_max=7, prior_accept=1.0, prior_reject=0.0, decay=0.95,
                hysteresis=0.10, cost_window=4)


class DepthController:
    def __init__(self, d_min=1, d_max=7, prior_accept=1.0, prior_reject=0.0, decay=0.95,
                 hysteresis=0.10, cost_window=4):
        self.d_min, self.d_max = int(d_min), int(d_max)
        self.pa, self.pr = float(prior_accept), float(prior_reject)
        self.decay, self.hyst = float(decay), float(hysteresis)
        self.window = int(cost_window)
        self.acc = [0.0] * (self.d_max + 1)   # index 1..d_max
        self.rej = [0.0] * (self.d_max + 1)
        self.costs = [[] for _ in range(self.d_max + 1)]  # newest last
        self.d_cur = self.d_max

    def p(self, i: int) -> float:
        a, b = self.acc[i], self.rej[i]
        return (a + self.pa) / (a + b + self.pa + self.pr)

    def expected_tokens(self, d: int) -> float:
        e, prod = 1.0, 1.0
        for i in range(1, d + 1):
            prod = prod * self.p(i)
            e = e + prod
        return e

    def cost(self, d: int) -> float | None:
        return min(self.costs[d]) if self.costs[d] else None

    def rate(self, d: int) -> float:
        c = self.cost(d)
        return math.inf if c is None else self.expected_tokens(d) / c

    def next_depth(self) -> int:
        return self.d_cur

    def observe(self, d: int, n_acc, round_seconds: float) -> int:
        """One finished round at depth d: the sequences' accepted counts (a
        negative count, a failed sequence, is skipped) and its time.
        Returns the depth of the next round."""
        for i in range(1, self.d_max + 1):
            self.acc[i] = self.acc[i] * self.decay
            self.rej[i] = self.rej[i] * self.decay
        for n in n_acc:
            n = int(n)
            if n < 0:
                continue
            for i in range(1, min(n, d) + 1):
                self.acc[i] = self.acc[i] + 1.0
            if n < d:
                self.rej[n + 1] = self.rej[n + 1] + 1.0
        w = self.costs[d]
        w.append(float(round_seconds))
        if len(w) > self.window:
            del w[0]
        self.d_cur = self._choose()
        return self.d_cur

    def _choose(self) -> int:
        for d in range(self.d_max, self.d_min - 1, -1):
            if not self.costs[d]:
                return d
        best, best_r = self.d_min, self.rate(self.d_min)
        for d in range(self.d_min + 1, self.d_max + 1):
            r = self.rate(d)
            if r > best_r:
                best, best_r = d, r
        if best != self.d_cur and best_r > (1.0 + self.hyst) * self.rate(self.d_cur):
            return best
        return self.d_cur
