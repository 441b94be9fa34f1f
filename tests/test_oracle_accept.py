"""Pins of the oracle's accept step: greedy patterns written out by hand,
the sampler's exp and integer weights against fp64 math, Philox against
cuRAND's host generator, and exact-rational losslessness at V=16.  CPU only."""
import ctypes
import math
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import softmax

from speculative_decoding_verification_round_gb300 import synth

TWO32 = 1 << 32


# --------------------------------------------------------------------------
# greedy
# --------------------------------------------------------------------------
def test_greedy_accept_hand_built_patterns(orc):
    d = 4
    draft = np.array([[10, 11, 12, 13]] * 6, np.int32)
    am = np.array([
        [99, 11, 12, 13, 14],   # mismatch at 0 -> emit [99]
        [10, 98, 12, 13, 14],   # mismatch at 1 -> emit [10, 98]
        [10, 11, 97, 13, 14],   # -> [10, 11, 97]
        [10, 11, 12, 96, 14],   # -> [10, 11, 12, 96]
        [10, 11, 12, 13, 95],   # all accepted -> bonus 95
        [10, 7, 12, 13, 14],    # later rows match but are never used
    ], np.int32)
    n_acc, em = orc.accept_greedy(am, draft)
    assert n_acc.tolist() == [0, 1, 2, 3, 4, 1]
    assert em[0].tolist() == [99, -1, -1, -1, -1]
    assert em[1].tolist() == [10, 98, -1, -1, -1]
    assert em[2].tolist() == [10, 11, 97, -1, -1]
    assert em[3].tolist() == [10, 11, 12, 96, -1]
    assert em[4].tolist() == [10, 11, 12, 13, 95]
    assert em[5].tolist() == [10, 7, -1, -1, -1]
    _ = d


def test_greedy_d0_is_plain_decode(orc):
    n_acc, em = orc.accept_greedy(np.array([[5], [0]], np.int32), np.zeros((2, 0), np.int32))
    assert n_acc.tolist() == [0, 0] and em[:, 0].tolist() == [5, 0]


def test_argmax_ties_lowest_index_and_nan(orc):
    assert orc.argmax(np.array([1, 3, 3, 2], np.float32)) == 1
    assert orc.argmax(np.array([-np.inf, -np.inf], np.float32)) == 0
    assert orc.argmax(np.array([1, np.nan, 3], np.float32)) == -1


# --------------------------------------------------------------------------
# exp and integer weights
# --------------------------------------------------------------------------
def test_exp_own_within_4ulp_of_fp64_exp(orc):
    g = np.random.default_rng(20)
    xs = np.concatenate([-g.random(20000) * 87.0, -g.random(5000) * 1e-3,
                         np.array([0.0, -1e-30, -0.5, -0.34657359, -0.3465736,
                                   -10.0, -86.99])]).astype(np.float32)
    for x in xs:
        e = orc.exp_own(float(x))
        ref = math.exp(float(x))
        assert abs(e - ref) <= 4 * 2 ** -24 * ref, (x, e, ref)
    assert orc.exp_own(0.0) == 1.0
    assert orc.exp_own(-88.0) == 0.0 and orc.exp_own(float("-inf")) == 0.0


def test_int_weight_is_floor_of_scaled_exp(orc):
    assert orc.int_weight(0.0) == TWO32
    assert orc.int_weight(-30.0) == 0       # e^-30 * 2^32 < 1
    g = np.random.default_rng(21)
    for x in (-g.random(3000) * 23.0).astype(np.float32):
        W = orc.int_weight(float(x))
        exact = math.exp(float(x)) * TWO32
        assert abs(W - exact) <= exact * 2 ** -21 + 1, (x, W, exact)


def test_row_weights_approximate_softmax(orc):
    g = np.random.default_rng(22)
    V = 5000
    for T in (1.0, 0.7):
        lg = (g.standard_normal(V) * 2).astype(np.float32)
        W, S = orc.row_weights(lg, T)
        assert int(W.max()) == TWO32 and S == int(W.sum())
        ref = softmax(lg.astype(np.float64) / T)
        dev = np.abs(W.astype(np.float64) / S - ref)
        assert dev.max() < 1e-6 and dev.sum() < 1e-5


# --------------------------------------------------------------------------
# Philox4x32-10 against cuRAND's host-side generator (a library routine)
# --------------------------------------------------------------------------
def _curand():
    for p in ("/usr/local/cuda/lib64/libcurand.so", "libcurand.so",
              "libcurand.so.10"):
        try:
            return ctypes.CDLL(p)
        except OSError:
            continue
    return None


def _curand_block(L, seed, block):
    """cuRAND host PHILOX4_32_10 output block `block` (4 words).  Its host
    generator runs 65536 subsequences: block b is counter
    (b // 65536 as 64 bits, b % 65536, 0) under key = seed."""
    gen = ctypes.c_void_p()
    assert L.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0
    assert L.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
    assert L.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(4 * block)) == 0
    out = np.zeros(4, np.uint32)
    assert L.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(4)) == 0
    L.curandDestroyGenerator(gen)
    return out


def test_philox_matches_curand_host_generator(orc):
    L = _curand()
    if L is None:
        pytest.skip("libcurand not loadable")
    g = np.random.default_rng(23)
    for _ in range(40):
        seed = int(g.integers(0, 2 ** 63)) * 2 + int(g.integers(0, 2))
        it = int(g.integers(0, 2 ** 40))
        sub = int(g.integers(0, 65536))
        ref = _curand_block(L, seed, it * 65536 + sub)
        ours = orc.philox4x32_10([it & 0xFFFFFFFF, it >> 32, sub, 0],
                                 [seed & 0xFFFFFFFF, seed >> 32])
        assert np.array_equal(ours, ref)
    # the sampler's mapping: counter = (slot lo, slot hi, seq id, domain 0)
    ref = _curand_block(L, 12345, (7 << 16) + 3)
    assert np.array_equal(orc.uniforms(12345, 7, 3, 0), ref)


def test_philox_uniform_and_counter_sensitive(orc):
    words = np.array([orc.uniforms(99, slot, 5, 0) for slot in range(4000)])
    top = (words >> 28).ravel()                       # 16 bins
    counts = np.bincount(top, minlength=16)
    exp = top.size / 16
    chi2 = ((counts - exp) ** 2 / exp).sum()
    assert chi2 < 50                                  # df=15, p ~ 1e-5
    base = orc.uniforms(99, 1000, 5, 0)
    for other in (orc.uniforms(99, 1001, 5, 0), orc.uniforms(99, 1000, 6, 0),
                  orc.uniforms(99, 1000, 5, 1), orc.uniforms(100, 1000, 5, 0)):
        flips = sum(bin(int(a) ^ int(b)).count("1") for a, b in zip(base, other))
        assert 40 < flips < 88                         # ~64 of 128 bits


# --------------------------------------------------------------------------
# accept / resample decisions
# --------------------------------------------------------------------------
def test_accept_decide_is_exact_u_less_than_ratio(orc):
    g = np.random.default_rng(24)
    for _ in range(3000):
        S = int(g.integers(TWO32, 2 ** 50))
        Sq = int(g.integers(TWO32, 2 ** 50))
        Wx = int(g.integers(0, TWO32 + 1))
        Wqx = int(g.integers(1, TWO32 + 1))
        U1 = int(g.integers(0, TWO32))
        ideal = Fraction(U1, TWO32) < Fraction(Wx * Sq, Wqx * S)
        assert orc.accept_decide(Wx, S, Wqx, Sq, U1) == ideal
    assert orc.accept_decide(5, TWO32, 0, TWO32, TWO32 - 1)
    assert not orc.accept_decide(0, TWO32, 0, TWO32, 0)


def test_picks_match_brute_force(orc):
    g = np.random.default_rng(25)
    for _ in range(300):
        V = int(g.integers(2, 12))
        W = g.integers(0, TWO32 + 1, V).astype(np.uint64)
        W[g.integers(0, V)] = TWO32
        Wq = g.integers(0, TWO32 + 1, V).astype(np.uint64)
        Wq[g.integers(0, V)] = TWO32
        S, Sq = int(W.sum()), int(Wq.sum())
        U2 = int(g.integers(0, TWO32))
        t = (U2 * S) >> 32
        cum = np.cumsum([int(w) for w in W])
        assert orc.weight_pick(W, S, U2) == int(np.argmax(np.array(cum, dtype=object) > t))
        R = [max(0, int(w) * Sq - int(q) * S) for w, q in zip(W, Wq)]
        if sum(R) == 0:
            continue
        t = (U2 * sum(R)) >> 32
        c, pick = 0, None
        for v, r in enumerate(R):
            c += r
            if c > t:
                pick = v
                break
        assert orc.residual_pick(W, S, Wq, Sq, U2) == pick


@pytest.mark.parametrize("d,seed", [(1, 1), (2, 2), (1, 3)])
def test_lossless_exact_v16(orc, d, seed):
    from oracle import exact_v16 as ev
    pair = ev.ToyPair(V=16, seed=seed)
    assert ev.max_deviation(pair, d, "ideal") == 0          # the lossless theorem, exactly
    dev = ev.max_deviation(pair, d, "implementation")        # the integer rules
    assert dev < Fraction(1, 10 ** 7)


@pytest.mark.slow
def test_lossless_exact_v16_d3(orc):
    from oracle import exact_v16 as ev
    pair = ev.ToyPair(V=16, seed=4, T=0.7)
    assert ev.max_deviation(pair, 3, "ideal") == 0
    assert ev.max_deviation(pair, 3, "implementation", check=False) < Fraction(1, 10 ** 7)


def test_lossless_detects_a_planted_mistake(orc):
    """The exact check is sharp: resampling from p instead of norm(max(0,p-q))
    (a plausible mistake) breaks it."""
    from oracle import exact_v16 as ev
    pair = ev.ToyPair(V=16, seed=5)
    orig = ev.residual_ideal
    try:
        ev.residual_ideal = lambda W, S, Wq, Sq: [Fraction(w, S) for w in W]
        assert ev.max_deviation(pair, 1, "ideal") > Fraction(1, 1000)
    finally:
        ev.residual_ideal = orig


# --------------------------------------------------------------------------
# the sequential stochastic accept
# --------------------------------------------------------------------------
def _small_case(seed=26, n_seq=3, d=5, V=300):
    g = np.random.default_rng(seed)
    p, q = synth.stochastic_logits(g, n_seq, d, V)
    draft = g.integers(0, V, (n_seq, d)).astype(np.int32)
    return p, q, draft


def test_stochastic_identical_p_q_accepts_everything(orc):
    p, q, _ = _small_case()
    n_seq, d1, V = p.shape
    d = d1 - 1
    draft = np.array([[int(np.argmax(p[s, i])) for i in range(d)] for s in range(n_seq)], np.int32)
    n_acc, em, ei = orc.accept_stochastic(p, p[:, :d], draft, 1.0, 7, [0, 1, 2], [0, 10, 20])
    assert n_acc.tolist() == [d] * n_seq
    assert np.array_equal(em[:, :d], draft)
    assert ei.tolist() == [d + 1, 10 + d + 1, 20 + d + 1]


def test_stochastic_suffix_after_rejection_is_never_read(orc):
    p, q, draft = _small_case(seed=27, n_seq=6, d=6)
    T, seed, sid, ei0 = 1.0, 11, np.arange(6), np.arange(6) * 100
    n_acc, em, ei = orc.accept_stochastic(p, q, draft, T, seed, sid, ei0)
    assert np.array_equal(ei, ei0 + n_acc + 1)              # one counter per emitted token
    assert all(((em[s] >= 0).sum() == n_acc[s] + 1) for s in range(6))
    g = np.random.default_rng(28)
    p2, q2, dr2 = p.copy(), q.copy(), draft.copy()
    for s in range(6):
        a = n_acc[s]
        p2[s, a + 1:] = g.standard_normal(p2[s, a + 1:].shape)
        if a + 1 < q2.shape[1]:
            q2[s, a + 1:] = g.standard_normal(q2[s, a + 1:].shape)
            dr2[s, a + 1:] = g.integers(0, p.shape[2], dr2[s, a + 1:].shape)
    n2, em2, ei2 = orc.accept_stochastic(p2, q2, dr2, T, seed, sid, ei0)
    assert np.array_equal(n2, n_acc) and np.array_equal(em2, em) and np.array_equal(ei2, ei)


def test_stochastic_d0_samples_from_p_at_the_slot_counter(orc):
    g = np.random.default_rng(29)
    p = (g.standard_normal((2, 1, 64)) * 2).astype(np.float32)
    n_acc, em, ei = orc.accept_stochastic(p, np.zeros((2, 0, 64), np.float32),
                                          np.zeros((2, 0), np.int32), 0.7, 3, [4, 9], [5, 6])
    for s, (sid, slot) in enumerate([(4, 5), (9, 6)]):
        W, S = orc.row_weights(p[s, 0], 0.7)
        assert em[s, 0] == orc.weight_pick(W, S, int(orc.uniforms(3, slot, sid, 0)[1]))
    assert n_acc.tolist() == [0, 0] and ei.tolist() == [6, 7]
