"""spec_accept_stochastic_noalloc: the allocation-free entry point (for
callers that cannot call cudaMalloc, e.g. while capturing a CUDA graph or
under a custom device allocator) must give exactly the results of
spec_accept_stochastic, call after call, through the C ABI.

This file is named to be collected last, and it builds all of its inputs
itself, so it passes both alone in a fresh process and after the rest of the
suite."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _inputs(seed, n_seq, d, V):
    g = np.random.default_rng(seed)
    p = (g.standard_normal((n_seq, d + 1, V)) * 2.0).astype(np.float32)
    q = (p[:, :d] + g.standard_normal((n_seq, d, V)) * 0.5).astype(np.float32)
    # drafts: mostly the target's own top token (long accepted runs), some random
    top = np.argmax(q, axis=2).astype(np.int32)
    rnd = g.integers(0, V, (n_seq, d)).astype(np.int32)
    draft = np.where(g.random((n_seq, d)) < 0.8, top, rnd).astype(np.int32)
    seq_ids = g.permutation(5000)[:n_seq].astype(np.int32)
    emit_idx = g.integers(0, 2 ** 40, n_seq).astype(np.int64)
    return p, q, draft, seq_ids, emit_idx


def _run(fn, dev, p, q, draft, seq_ids, emit_idx, T, seed):
    import torch
    n_seq, d1, V = p.shape
    d = d1 - 1
    ei = torch.from_numpy(emit_idx.copy()).to(dev)
    n_acc = torch.full((n_seq,), -7, dtype=torch.int32, device=dev)
    em = torch.full((n_seq, d1), -7, dtype=torch.int32, device=dev)
    fn(torch.from_numpy(p).to(dev), torch.from_numpy(q).to(dev) if d else None,
       torch.from_numpy(draft).to(dev) if d else None, n_seq, d, V, T, seed,
       torch.from_numpy(seq_ids).to(dev), ei, n_acc, em)
    torch.cuda.synchronize()
    return n_acc.cpu().numpy(), em.cpu().numpy(), ei.cpu().numpy()


def test_noalloc_matches_allocating_entry_point_twice_in_a_row():
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    assert torch.cuda.is_available()
    dev = torch.device("cuda:0")
    T, seed = 0.8, 2024
    # call 1: 12 sequences, d=7, a large vocabulary
    p, q, draft, sid, ei = _inputs(1, 12, 7, 50000)
    ref = _run(sv.spec_accept_stochastic, dev, p, q, draft, sid, ei, T, seed)
    got = _run(sv.spec_accept_stochastic_noalloc, dev, p, q, draft, sid, ei, T, seed)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)
    assert (got[0] >= 0).all() and (got[2] == ei + got[0] + 1).all()
    # call 2, right after, on the same fixed scratch: the next round of the
    # same sequences (advanced sampler slots) with new logits and drafts
    p2, q2, draft2, _, _ = _inputs(2, 12, 7, 50000)
    ref2 = _run(sv.spec_accept_stochastic, dev, p2, q2, draft2, sid, ref[2], T, seed)
    got2 = _run(sv.spec_accept_stochastic_noalloc, dev, p2, q2, draft2, sid, got[2], T, seed)
    for a, b in zip(got2, ref2):
        assert np.array_equal(a, b)


def test_noalloc_error_and_size_limits():
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    dev = torch.device("cuda:0")
    # a NaN logit: outputs -1, sampler state untouched; the next call is clean
    p, q, draft, sid, ei = _inputs(3, 3, 2, 300)
    p[1, 0, 5] = np.nan
    got = _run(sv.spec_accept_stochastic_noalloc, dev, p, q, draft, sid, ei, 1.0, 5)
    assert (got[0] == -1).all() and (got[1] == -1).all() and (got[2] == ei).all()
    p[1, 0, 5] = 0.0
    ref = _run(sv.spec_accept_stochastic, dev, p, q, draft, sid, ei, 1.0, 5)
    got = _run(sv.spec_accept_stochastic_noalloc, dev, p, q, draft, sid, ei, 1.0, 5)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)
    # more rows than the fixed scratch holds: a clear error, nothing launched
    n_seq, d, V = 300, 7, 16       # 300 * 15 = 4500 > 4096 rows
    big = torch.zeros((n_seq, d + 1, V), dtype=torch.float32, device=dev)
    qb = torch.zeros((n_seq, d, V), dtype=torch.float32, device=dev)
    dr = torch.zeros((n_seq, d), dtype=torch.int32, device=dev)
    ids = torch.arange(n_seq, dtype=torch.int32, device=dev)
    e = torch.zeros(n_seq, dtype=torch.int64, device=dev)
    na = torch.zeros(n_seq, dtype=torch.int32, device=dev)
    em = torch.zeros((n_seq, d + 1), dtype=torch.int32, device=dev)
    with pytest.raises(sv.SpecError, match="fixed scratch"):
        sv.spec_accept_stochastic_noalloc(big, qb, dr, n_seq, d, V, 1.0, 1, ids, e, na, em)
