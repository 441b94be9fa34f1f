"""LM head + greedy accept (the H=1024, V=32000, nt=3 LM-head workload) and
strict rejection sampling (12 sequences, d=7, V=248320; plus a V=16
distribution check) on the GPU against the oracle."""
import numpy as np
import pytest

from speculative_decoding_verification_round_gb300 import synth

from util import LOGIT_RTOL, MARGIN, dev_weight, oracle_qweight, rel_err, top2_margin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


def lm_only_model(sv, dev, w, H, V, max_rows):
    import torch
    W = dict(lm_head=dev_weight(w, dev),
             norm_w=torch.ones((1, H), dtype=torch.float32, device=dev))
    nt = min(max_rows, 16)
    return sv.Model(dict(n_layers=0, hidden=H, vocab=V, max_nt=nt,
                         max_seqs=(max_rows + nt - 1) // nt), W)


@pytest.mark.parametrize("H,V,R,qtype", [(1024, 32000, 3, 4), (256, 2048, 16, 6), (128, 160, 1, 4),
                                         (512, 4096, 40, 4)])
def test_lm_head_logits_argmax_greedy(orc, dev, H, V, R, qtype):
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    wl = synth.WL_LMHEAD_GREEDY
    g = np.random.default_rng(wl["seed"] + H + V)
    w = synth.q_weight(g, qtype, V, H)
    x = synth.f16_normal(g, (R, H))
    m = lm_only_model(sv, dev, w, H, V, R)
    xd = torch.from_numpy(x.view(np.int16)).to(dev)
    logits = torch.empty((R, V), dtype=torch.float32, device=dev)
    am = torch.empty(R, dtype=torch.int32, device=dev)
    sv.spec_lm_head(m, xd, R, logits, am)
    assert sv.spec_error_check(m) == 0
    ref = orc.linear(oracle_qweight(orc, w), x)
    assert rel_err(logits.cpu().numpy(), ref) <= LOGIT_RTOL
    got_am = am.cpu().numpy()
    lg = logits.cpu().numpy()
    for r in range(R):
        # the GPU argmax is exactly the argmax of the GPU's own logits
        assert got_am[r] == orc.argmax(lg[r])
        if top2_margin(ref[r]) > MARGIN:
            assert got_am[r] == orc.argmax(ref[r])
    # argmax without logits gives the same ids
    am2 = torch.empty(R, dtype=torch.int32, device=dev)
    sv.spec_lm_head(m, xd, R, None, am2)
    assert np.array_equal(am2.cpu().numpy(), got_am)
    # greedy accept on drafts that agree with the target w.p. 0.74
    if R >= 2:
        d = R - 1
        ref_am = np.array([orc.argmax(ref[r]) for r in range(R)], np.int32)
        draft = synth.greedy_drafts(g, ref_am[:d], V, wl["p_agree"])[None, :]
        n_acc = torch.empty(1, dtype=torch.int32, device=dev)
        em = torch.empty((1, d + 1), dtype=torch.int32, device=dev)
        sv.spec_accept_greedy(am.view(1, R), torch.from_numpy(draft).to(dev), 1, d, n_acc, em)
        n_ref, em_ref = orc.accept_greedy(got_am[None, :], draft)
        assert int(n_acc.item()) == int(n_ref[0])
        assert np.array_equal(em.cpu().numpy(), em_ref)


def test_greedy_accept_patterns_every_mismatch_position(orc, dev):
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    d = 7
    g = np.random.default_rng(3)
    draft = g.integers(0, 1000, (d + 2, d)).astype(np.int32)
    am = np.zeros((d + 2, d + 1), np.int32)
    for s in range(d + 2):
        am[s, :d] = draft[s]
        am[s, d] = 5000 + s
        if s <= d - 1:
            am[s, s] = 9999            # mismatch at position s
    n_acc = torch.empty(d + 2, dtype=torch.int32, device=dev)
    em = torch.empty((d + 2, d + 1), dtype=torch.int32, device=dev)
    sv.spec_accept_greedy(torch.from_numpy(am).to(dev), torch.from_numpy(draft).to(dev), d + 2, d,
                          n_acc, em)
    n_ref, em_ref = orc.accept_greedy(am, draft)
    assert np.array_equal(n_acc.cpu().numpy(), n_ref)
    assert np.array_equal(em.cpu().numpy(), em_ref)
    assert n_ref.tolist()[:d] == list(range(d)) and n_ref[d] == d


def sample_drafts_oracle(orc, q, T, seed, seq_ids, emit_idx):
    """Drafts sampled from q by the harness's own sampler (Philox domain 1)."""
    n_seq, d, V = q.shape
    out = np.zeros((n_seq, d), np.int32)
    for s in range(n_seq):
        for i in range(d):
            W, S = orc.row_weights(q[s, i], T)
            U = orc.uniforms(seed, int(emit_idx[s]) + i, int(seq_ids[s]), 1)
            out[s, i] = orc.weight_pick(W, S, int(U[0]))
    return out


def run_stochastic(sv, dev, p, q, draft, T, seed, seq_ids, emit_idx):
    import torch
    n_seq, d1, V = p.shape
    d = d1 - 1
    pd = torch.from_numpy(p).to(dev)
    qd = torch.from_numpy(q).to(dev) if d > 0 else None
    ei = torch.from_numpy(np.asarray(emit_idx, np.int64)).to(dev)
    n_acc = torch.empty(n_seq, dtype=torch.int32, device=dev)
    em = torch.empty((n_seq, d1), dtype=torch.int32, device=dev)
    sv.spec_accept_stochastic(pd, qd, torch.from_numpy(draft).to(dev) if d > 0 else None, n_seq, d,
                              V, T, seed, torch.from_numpy(np.asarray(seq_ids, np.int32)).to(dev),
                              ei, n_acc, em)
    bits = sv.spec_error_check(None)
    return n_acc.cpu().numpy(), em.cpu().numpy(), ei.cpu().numpy().astype(np.uint64), bits


def test_stochastic_accept_full_size_bit_exact(orc, dev):
    import speculative_decoding_verification_round_gb300 as sv
    wl = synth.WL_ACCEPT_STOCH
    g = np.random.default_rng(wl["seed"])
    n_seq, d, V, T = wl["n_seq"], wl["d"], wl["vocab"], wl["temperature"]
    p, q = synth.stochastic_logits(g, n_seq, d, V, wl["p_std"], wl["q_noise"])
    seq_ids = np.arange(n_seq) * 3 + 1
    emit_idx = g.integers(0, 10 ** 6, n_seq).astype(np.uint64)
    seed = 0x5EED
    draft = sample_drafts_oracle(orc, q, T, seed, seq_ids, emit_idx)
    n_g, em_g, ei_g, bits = run_stochastic(sv, dev, p, q, draft, T, seed, seq_ids, emit_idx)
    assert bits == 0
    n_r, em_r, ei_r = orc.accept_stochastic(p, q, draft, T, seed, seq_ids, emit_idx)
    assert np.array_equal(n_g, n_r) and np.array_equal(em_g, em_r) and np.array_equal(ei_g, ei_r)
    assert np.array_equal(ei_g, emit_idx + n_r.astype(np.uint64) + 1)
    # realistic acceptance with q close to p
    assert n_r.mean() > 2.0


@pytest.mark.parametrize("n_seq,d,V,T", [(5, 0, 1000, 1.0), (3, 15, 777, 0.7), (20, 3, 64, 1.3)])
def test_stochastic_accept_shapes_bit_exact(orc, dev, n_seq, d, V, T):
    import speculative_decoding_verification_round_gb300 as sv
    g = np.random.default_rng(n_seq * 100 + d)
    p, q = synth.stochastic_logits(g, n_seq, d, V)
    seq_ids = g.permutation(1000)[:n_seq]
    emit_idx = g.integers(0, 2 ** 40, n_seq).astype(np.uint64)
    draft = sample_drafts_oracle(orc, q, T, 9, seq_ids, emit_idx) if d else np.zeros((n_seq, 0), np.int32)
    n_g, em_g, ei_g, bits = run_stochastic(sv, dev, p, q, draft, T, 9, seq_ids, emit_idx)
    assert bits == 0
    n_r, em_r, ei_r = orc.accept_stochastic(p, q, draft, T, 9, seq_ids, emit_idx)
    assert np.array_equal(n_g, n_r) and np.array_equal(em_g, em_r) and np.array_equal(ei_g, ei_r)


def test_stochastic_rejected_suffix_never_read(orc, dev):
    import speculative_decoding_verification_round_gb300 as sv
    g = np.random.default_rng(11)
    n_seq, d, V, T = 8, 6, 3000, 1.0
    p, q = synth.stochastic_logits(g, n_seq, d, V)
    q = q + g.standard_normal(q.shape).astype(np.float32) * 2.0   # more rejections
    seq_ids, ei0 = np.arange(n_seq), np.zeros(n_seq, np.uint64)
    draft = sample_drafts_oracle(orc, q, T, 4, seq_ids, ei0)
    n_g, em_g, ei_g, _ = run_stochastic(sv, dev, p, q, draft, T, 4, seq_ids, ei0)
    p2, q2, d2 = p.copy(), q.copy(), draft.copy()
    for s in range(n_seq):
        a = n_g[s]
        p2[s, a + 1:] = 50.0 * g.standard_normal(p2[s, a + 1:].shape)
        q2[s, a + 1:] = 50.0 * g.standard_normal(q2[s, a + 1:].shape)
        d2[s, a + 1:] = g.integers(0, V, d2[s, a + 1:].shape)
    n2, em2, ei2, _ = run_stochastic(sv, dev, p2, q2, d2, T, 4, seq_ids, ei0)
    assert np.array_equal(n2, n_g) and np.array_equal(em2, em_g) and np.array_equal(ei2, ei_g)


def test_stochastic_nonfinite_logit_fails_closed(dev):
    import speculative_decoding_verification_round_gb300 as sv
    g = np.random.default_rng(12)
    p, q = synth.stochastic_logits(g, 2, 2, 100)
    p[1, 0, 7] = np.nan
    draft = np.zeros((2, 2), np.int32)
    n_g, em_g, ei_g, bits = run_stochastic(sv, dev, p, q, draft, 1.0, 1, [0, 1], [5, 6])
    assert bits != 0
    assert (n_g == -1).all() and (em_g == -1).all() and ei_g.tolist() == [5, 6]


def test_stochastic_v16_distribution_chi2(orc, dev):
    """GPU Monte Carlo of 10^7 rounds (d = 1, V = 16) against the exact
    distribution of the first emitted token that the exact-rational
    enumeration gives for the integer decision rules.  Drafts are drawn from
    the draft's integer weights (exactly Wq/Sq, by a host generator); the
    target row after the draft depends on it; every round has its own
    sampler counter (emitted slot, sequence id)."""
    from scipy.stats import chi2
    import speculative_decoding_verification_round_gb300 as sv
    from oracle import exact_v16 as ev
    V, n_seq, batches, T = 16, 1 << 16, 153, 1.0   # 10,027,008 rounds
    pair = ev.ToyPair(V=V, seed=21, T=T)
    exp0 = np.array([float(x) for x in
                     ev.emitted_conditionals(pair, 1, "implementation", check=False)[(0, ())]])
    # the same logits the toy pair draws (prefix () and prefix (x,))
    g = np.random.default_rng([21, 0])
    lp0 = (g.standard_normal(V) * 2.0).astype(np.float32)
    lq0 = (lp0 + g.standard_normal(V) * 0.5).astype(np.float32)
    lp1 = np.stack([(np.random.default_rng([21, 1, x]).standard_normal(V) * 2.0).astype(np.float32)
                    for x in range(V)])
    Wq, Sq = orc.row_weights(lq0, T)
    cum = np.cumsum(np.asarray(Wq, np.uint64).astype(np.int64))
    assert int(cum[-1]) == int(Sq)
    q = np.broadcast_to(lq0, (n_seq, 1, V)).copy()
    seq_ids = np.arange(n_seq)
    hr = np.random.default_rng(2024)
    counts = np.zeros(V)
    for b in range(batches):
        u = hr.integers(0, int(Sq), n_seq)
        draft = np.searchsorted(cum, u, side="right").astype(np.int32)[:, None]
        p = np.empty((n_seq, 2, V), np.float32)
        p[:, 0] = lp0
        p[:, 1] = lp1[draft[:, 0]]
        emit = np.full(n_seq, 2 * b, np.uint64)  # slots 2b, 2b+1: distinct per batch
        n_g, em_g, _, bits = run_stochastic(sv, dev, p, q, draft, T, 31337, seq_ids, emit)
        assert bits == 0
        counts += np.bincount(em_g[:, 0], minlength=V)
    n = counts.sum()
    assert n == n_seq * batches >= 10 ** 7
    mask = exp0 * n > 5
    stat = (((counts - exp0 * n) ** 2) / (exp0 * n))[mask].sum()
    assert stat < chi2.ppf(1 - 1e-3, mask.sum() - 1), (stat, counts, exp0 * n)


def test_stochastic_accept_first_call_in_fresh_process():
    """The standalone accept works as the first call a process makes (no
    model or matrix created before it sets the kernels' attributes)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (
        "import numpy as np, torch\n"
        "import speculative_decoding_verification_round_gb300 as sv\n"
        "dev = torch.device('cuda:0')\n"
        "g = np.random.default_rng(5)\n"
        "n, d, V = 3, 4, 50000\n"
        "p = torch.from_numpy(g.standard_normal((n, d + 1, V), dtype=np.float32)).to(dev)\n"
        "q = torch.from_numpy(g.standard_normal((n, d, V), dtype=np.float32)).to(dev)\n"
        "dr = torch.zeros((n, d), dtype=torch.int32, device=dev)\n"
        "sid = torch.arange(n, dtype=torch.int32, device=dev)\n"
        "ei = torch.zeros(n, dtype=torch.int64, device=dev)\n"
        "na = torch.empty(n, dtype=torch.int32, device=dev)\n"
        "em = torch.empty((n, d + 1), dtype=torch.int32, device=dev)\n"
        "sv.spec_accept_stochastic(p, q, dr, n, d, V, 1.0, 7, sid, ei, na, em)\n"
        "torch.cuda.synchronize()\n"
        "assert sv.spec_error_check(None) == 0\n"
        "print('ok', na.cpu().tolist())\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr
