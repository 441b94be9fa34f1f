"""Adaptive draft depth ("Speculative Decoding (D5-R) -- Plan", status notes:
beta-smoothed per-depth acceptance, min-of-4 cost windows, 10% hysteresis,
optimism for unseen depths, d <= 7).  The oracle (oracle/depth.py) is pinned
to closed forms and hand-worked rounds; the library's controller must make
the same decisions with the same doubles.  CPU only: the controller does no
GPU work."""
import math

import numpy as np
import pytest

from oracle.depth import DepthController as Oracle


def test_expected_tokens_is_the_geometric_sum():
    """Constant acceptance p at every position (a prior of mean p, no
    observations): E(d) = (1 - p^(d+1)) / (1 - p)."""
    for p, m in [(0.75, 4.0), (0.5, 2.0), (0.875, 8.0)]:
        c = Oracle(prior_accept=p * m, prior_reject=(1 - p) * m)
        for d in range(0, 8):
            assert c.expected_tokens(d) == pytest.approx((1 - p ** (d + 1)) / (1 - p), rel=1e-15)


def test_a_round_observes_the_accepted_prefix_and_the_first_rejection():
    c = Oracle(decay=0.5)
    c.observe(7, [3, 7, 0, -1], 1e-3)   # -1: a failed sequence observes nothing
    assert c.acc[1:] == [2.0, 2.0, 2.0, 1.0, 1.0, 1.0, 1.0]
    assert c.rej[1:] == [1.0, 0.0, 0.0, 1.0, 0.0, 0.0, 0.0]
    c.observe(2, [2], 1e-3)              # all of a depth-2 block accepted: no rejection
    assert c.acc[1:3] == [2.0, 2.0] and c.rej[1:3] == [0.5, 0.0]
    assert c.acc[3:] == [1.0, 0.5, 0.5, 0.5, 0.5]
    # with prior (1, 0): p_1 = (2 + 1) / (2 + 0.5 + 1)
    assert c.p(1) == 3.0 / 3.5


def test_unseen_depths_are_explored_deepest_first():
    c = Oracle(d_min=1, d_max=7)
    assert c.next_depth() == 7
    order = []
    for _ in range(7):
        d = c.next_depth()
        order.append(d)
        c.observe(d, [d], 1e-3)          # everything accepted, equal cost
    assert order == [7, 6, 5, 4, 3, 2, 1]
    # all seen, all accepted, equal costs: the deepest depth has the most tokens
    assert c.next_depth() == 7


def test_hysteresis_keeps_a_depth_within_ten_percent():
    """Acceptance fixed by the prior (p = 1/2, no observations used); the
    round times make depth 2 better than depth 1 by 5% (kept) or by 15%
    (switched)."""
    for gain, expect in [(1.05, 1), (1.15, 2)]:
        c = Oracle(d_min=1, d_max=2, prior_accept=1e9, prior_reject=1e9, decay=1.0)
        c.observe(2, [], 1.0)
        c.observe(1, [], 1.0)
        assert c.next_depth() == 1 or c.next_depth() == 2
        c.d_cur = 1
        e1, e2 = c.expected_tokens(1), c.expected_tokens(2)
        # depth 2's time so that r(2) = gain * r(1)
        c.costs[2] = []
        nxt = c.observe(2, [], e2 / (gain * e1))
        assert nxt == expect, (gain, nxt)


def rates_true(p, alpha, beta, d_max):
    return [((1 - p ** (d + 1)) / (1 - p)) / (alpha + beta * d) for d in range(d_max + 1)]


@pytest.mark.parametrize("p,alpha,beta", [(0.9, 1.0, 0.1), (0.5, 1.0, 0.3), (0.3, 1.0, 0.5)])
def test_converges_near_the_optimal_depth(p, alpha, beta):
    """Bernoulli drafts (each position accepted with probability p, 16
    sequences a round) and round time alpha + beta * d: after 300 rounds the
    chosen depth's true rate is within the hysteresis (and estimation noise)
    of the best depth's."""
    g = np.random.default_rng(3)
    c = Oracle(d_min=1, d_max=7)
    d = c.next_depth()
    for _ in range(300):
        draws = g.random((16, d)) < p
        n = [int(np.argmin(row)) if not row.all() else d for row in draws]
        d = c.observe(d, n, alpha + beta * d)
    r = rates_true(p, alpha, beta, 7)
    assert r[d] >= max(r[1:]) / 1.15, (d, r)


def test_library_controller_matches_the_oracle_bit_for_bit():
    """Seeded streams of rounds (depths as the controller picks them, random
    accept counts, including failed sequences, and random round times): the
    library returns the same depths, and the same p_i and r(d) doubles."""
    import speculative_decoding_verification_round_gb300 as sv
    for seed, kw in [(1, {}), (2, dict(d_min=0, d_max=15, decay=0.9, hysteresis=0.05,
                                       cost_window=3, prior_accept=2.0, prior_reject=1.0))]:
        g = np.random.default_rng(seed)
        o = Oracle(**kw)
        c = sv.DepthController(**kw)
        try:
            assert c.next_depth() == o.next_depth()
            for _ in range(400):
                d = o.next_depth()
                n = g.integers(-1, d + 1, size=int(g.integers(0, 9))).tolist()
                t = float(g.uniform(0.5e-3, 1.5e-3))
                assert c.observe(d, n, t) == o.observe(d, n, t)
                p, r = c.estimates()
                assert p[1:] == [o.p(i) for i in range(1, o.d_max + 1)]
                for dd in range(o.d_max + 1):
                    ro = 0.0 if dd < o.d_min else o.rate(dd)
                    assert r[dd] == ro or (math.isinf(r[dd]) and math.isinf(ro))
        finally:
            c.close()


def test_library_controller_rejects_bad_input():
    import speculative_decoding_verification_round_gb300 as sv
    with pytest.raises(sv.SpecError):
        sv.DepthController(d_min=3, d_max=2)
    with pytest.raises(sv.SpecError):
        sv.DepthController(d_max=sv.SPEC_MAX_NT)
    with pytest.raises(sv.SpecError):
        sv.DepthController(decay=0.0)
    c = sv.DepthController()
    try:
        with pytest.raises(sv.SpecError):
            c.observe(0, [0], 1e-3)          # below d_min
        with pytest.raises(sv.SpecError):
            c.observe(7, [1], float("nan"))
        assert c.next_depth() == 7           # unchanged by the refused rounds
    finally:
        c.close()
