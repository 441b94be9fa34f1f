"""Exact-rational check of the strict rejection sampler at a small vocabulary.

TEST INFRASTRUCTURE (oracle side).  Losslessness under strict rejection
sampling ("DFlash and DSpark Speculative Decoding", "How DSpark Works": both
methods are lossless under rejection sampling; use the strict sampler) means:
whatever the draft distribution q, each emitted token, given the tokens
emitted before it, is distributed as the target's own p at that position.

For a toy target/draft pair over V tokens whose next-token distributions
depend on the whole prefix, this module enumerates every draft block and
every accept/resample outcome, and returns for each (slot j, emitted prefix)
the exact conditional distribution of the token emitted at slot j:

  * ``ideal``:  accept with min(1, p_x/q_x), resample from norm(max(0, p-q)),
    bonus from p, all as exact fractions of the integer weights.  The
    lossless theorem says the conditionals equal p exactly.
  * ``implementation``: the oracle's integer decision rules, counted over all
    2^32 values of the uniform word (accept counts and resample intervals are
    computed in closed form and checked at their boundaries against the
    oracle's own decision functions).  Each conditional is within a few
    2^-32 of p.
"""
from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np

from . import accept_decide, residual_pick, row_weights, weight_pick

TWO32 = 1 << 32


def _ceil_div(a: int, b: int) -> int:
    return -((-a) // b)


class ToyPair:
    """Target and draft next-token logits as deterministic functions of the
    prefix: p-logits N(0, p_std^2), q-logits = p-logits + N(0, q_noise^2),
    drawn per prefix from a seeded generator; both turned into integer
    weights by the oracle's sampler definition at temperature T."""

    def __init__(self, V=16, seed=0, p_std=2.0, q_noise=0.5, T=1.0):
        self.V, self.seed, self.p_std, self.q_noise, self.T = V, seed, p_std, q_noise, T
        self._cache = {}

    def weights(self, prefix: tuple):
        if prefix not in self._cache:
            key = [self.seed, len(prefix), *prefix]
            g = np.random.default_rng(key)
            p = (g.standard_normal(self.V) * self.p_std).astype(np.float32)
            q = (p + g.standard_normal(self.V) * self.q_noise).astype(np.float32)
            W, S = row_weights(p, self.T)
            Wq, Sq = row_weights(q, self.T)
            self._cache[prefix] = ([int(v) for v in W], S, [int(v) for v in Wq], Sq)
        return self._cache[prefix]


# -------------------------------------------------------------------------
# decision probabilities
# -------------------------------------------------------------------------
def accept_prob_ideal(Wx, S, Wqx, Sq) -> Fraction:
    if Wqx == 0:
        return Fraction(1 if Wx > 0 else 0)
    return min(Fraction(1), Fraction(Wx * Sq, Wqx * S))


def accept_count_impl(Wx, S, Wqx, Sq, check=True) -> int:
    """#U1 in [0, 2^32) with U1*Wq_x*S < 2^32*W_x*Sq (all if Wq_x == 0 and
    W_x > 0).  Checked at the boundary against the oracle's decision."""
    if Wqx == 0:
        c = TWO32 if Wx > 0 else 0
    else:
        c = min(TWO32, _ceil_div(TWO32 * Wx * Sq, Wqx * S))
    if check:
        if c > 0:
            assert accept_decide(Wx, S, Wqx, Sq, c - 1)
        if c < TWO32:
            assert not accept_decide(Wx, S, Wqx, Sq, c)
    return c


def residual_ideal(W, S, Wq, Sq):
    R = [max(0, w * Sq - wq * S) for w, wq in zip(W, Wq)]
    T = sum(R)
    return [Fraction(r, T) for r in R]


def _interval_counts(masses, check_fn):
    """Counts of U2 in [0, 2^32) picking each index, for
    t = floor(U2 * total / 2^32), pick = smallest v with cum_v > t."""
    total = sum(masses)
    N = lambda c: min(TWO32, _ceil_div(c * TWO32, total))
    counts, cum = [], 0
    for v, m in enumerate(masses):
        lo = N(cum)
        cum += m
        hi = N(cum)
        counts.append(hi - lo)
        if check_fn is not None and hi > lo:
            assert check_fn(lo) == v, (v, lo)
            assert check_fn(hi - 1) == v, (v, hi - 1)
    assert sum(counts) == TWO32
    return counts


def residual_counts_impl(W, S, Wq, Sq, check=True):
    R = [max(0, w * Sq - wq * S) for w, wq in zip(W, Wq)]
    fn = (lambda u: residual_pick(np.array(W, np.uint64), S,
                                  np.array(Wq, np.uint64), Sq, u)) if check else None
    return _interval_counts(R, fn)


def bonus_counts_impl(W, S, check=True):
    fn = (lambda u: weight_pick(np.array(W, np.uint64), S, u)) if check else None
    return _interval_counts(W, fn)


# -------------------------------------------------------------------------
# enumeration
# -------------------------------------------------------------------------
def emitted_conditionals(pair: ToyPair, d: int, mode: str = "ideal", check=True):
    """Returns dict[(j, prefix)] -> list of V Fractions: the distribution of
    the token emitted at slot j given the emitted prefix (and that the round
    reached slot j).  mode is 'ideal' or 'implementation'."""
    V = pair.V
    mass = {}  # (j, prefix) -> [Fraction]*V, unnormalised

    def add(j, prefix, v, m):
        row = mass.setdefault((j, prefix), [Fraction(0)] * V)
        row[v] += m

    frontier = {(): Fraction(1)}
    for j in range(d + 1):
        nxt = {}
        for prefix, m in frontier.items():
            W, S, Wq, Sq = pair.weights(prefix)
            if j == d:
                if mode == "ideal":
                    probs = [Fraction(w, S) for w in W]
                else:
                    probs = [Fraction(c, TWO32) for c in bonus_counts_impl(W, S, check)]
                for v in range(V):
                    add(j, prefix, v, m * probs[v])
                continue
            if mode == "ideal":
                res = residual_ideal(W, S, Wq, Sq)
            else:
                res = [Fraction(c, TWO32) for c in residual_counts_impl(W, S, Wq, Sq, check)]
            for x in range(V):
                qx = Fraction(Wq[x], Sq)
                if qx == 0:
                    continue
                if mode == "ideal":
                    a = accept_prob_ideal(W[x], S, Wq[x], Sq)
                else:
                    a = Fraction(accept_count_impl(W[x], S, Wq[x], Sq, check), TWO32)
                if a > 0:
                    add(j, prefix, x, m * qx * a)
                    nxt[prefix + (x,)] = nxt.get(prefix + (x,), Fraction(0)) + m * qx * a
                if a < 1:
                    rej = m * qx * (1 - a)
                    for v in range(V):
                        if res[v]:
                            add(j, prefix, v, rej * res[v])
        frontier = nxt
    out = {}
    for key, row in mass.items():
        tot = sum(row)
        out[key] = [r / tot for r in row]
    return out


def target_conditional(pair: ToyPair, prefix: tuple):
    W, S, _, _ = pair.weights(prefix)
    return [Fraction(w, S) for w in W]


def max_deviation(pair: ToyPair, d: int, mode: str, check=True) -> Fraction:
    cond = emitted_conditionals(pair, d, mode, check)
    worst = Fraction(0)
    for (j, prefix), row in cond.items():
        tgt = target_conditional(pair, prefix)
        worst = max(worst, max(abs(a - b) for a, b in zip(row, tgt)))
    return worst


def all_prefixes(V, n):
    return itertools.product(range(V), repeat=n)
