"""spec_linear_q on the GPU against the oracle, and bitwise row invariance
across nt (the weights-once verify GEMM)."""
import numpy as np
import pytest

from speculative_decoding_verification_round_gb300 import synth

from util import dev_weight, host_weight, oracle_qweight, rel_err

pytestmark = pytest.mark.gpu

NTS = [1, 2, 3, 4, 8, 9, 16]


@pytest.fixture(scope="module")
def dev():
    import torch
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


def run_linear(sv, qm, x_dev, nt):
    import torch
    y = torch.empty((nt, qm.N), dtype=torch.float32, device=x_dev.device)
    sv.spec_linear_q(qm, x_dev[:nt].contiguous(), nt, y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("qtype,N,K", [(4, 48, 96), (6, 64, 160), (4, 16, 32), (6, 272, 544),
                                       (4, 512, 1024), (8, 48, 96), (8, 272, 544), (8, 16, 32)])
def test_linear_small_matches_oracle(orc, dev, qtype, N, K):
    """Several tiles and K chunks, ragged K tail (K % 64 == 32), ragged
    tile groups; every nt of the sweep."""
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    g = np.random.default_rng(100 + N + K)
    w = synth.q_weight(g, qtype, N, K)
    x = synth.f16_normal(g, (16, K))
    qm = sv.QMat(dev_weight(w, dev), max_rows=16)
    xd = torch.from_numpy(x.view(np.int16)).to(dev)
    ref = orc.linear(oracle_qweight(orc, w), x)
    y16 = run_linear(sv, qm, xd, 16)
    assert rel_err(y16, ref) < 1e-5
    for nt in NTS:
        y = run_linear(sv, qm, xd, nt)
        assert np.array_equal(y, y16[:nt]), f"row invariance broken at nt={nt}"


@pytest.mark.parametrize("qtype,N,K", [(4, 5120, 13824), (6, 13824, 5120), (8, 5120, 13824)])
def test_linear_full_size_sweep(orc, dev, qtype, N, K):
    """The linear sweep at full size: every nt, all outputs against the
    oracle (nt=16), and bitwise invariance of every row across nt."""
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    gen = synth.torch_gen(7 + qtype, dev)
    wd = synth.q_weight_torch(gen, qtype, N, K, dev)
    x = synth.f16_normal_torch(gen, (16, K), dev)
    qm = sv.QMat(wd, max_rows=16)
    ref = orc.linear(oracle_qweight(orc, host_weight(wd)), x.cpu().view(torch.int16).numpy().view(np.uint16))
    y16 = run_linear(sv, qm, x.view(torch.int16), 16)
    assert rel_err(y16, ref) < 1e-5
    for nt in NTS:
        y = run_linear(sv, qm, x.view(torch.int16), nt)
        assert np.array_equal(y, y16[:nt]), f"row invariance broken at nt={nt}"


@pytest.mark.parametrize("split", ["1:1", "1:5", "2:3", "4:1", "4:17", "8:2", "8:6"])
@pytest.mark.parametrize("qtype,N,K", [(4, 272, 1056), (6, 144, 2080), (8, 208, 1568)])
def test_linear_every_split_matches_oracle(orc, dev, monkeypatch, qtype, N, K, split):
    """Every in-CTA K slicing (KW warps per tile pair) and several K segment
    counts S, forced through SPEC_VERIFY_LINEAR_SPLIT: an odd number of tiles
    (a padding tile), a ragged K tail, S up to one chunk per segment, slices
    with no chunk at all.  All outputs against the oracle, rows bitwise equal
    across nt, and the LM-head-free store path for R > 16."""
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    monkeypatch.setenv("SPEC_VERIFY_LINEAR_SPLIT", split)
    g = np.random.default_rng(hash((qtype, N, K)) % 1000)
    w = synth.q_weight(g, qtype, N, K)
    x = synth.f16_normal(g, (40, K))
    qm = sv.QMat(dev_weight(w, dev), max_rows=40)
    xd = torch.from_numpy(x.view(np.int16)).to(dev)
    ref = orc.linear(oracle_qweight(orc, w), x)
    y40 = run_linear(sv, qm, xd, 40)
    assert rel_err(y40, ref) < 1e-5
    y16 = run_linear(sv, qm, xd, 16)
    assert np.array_equal(y16, y40[:16])
    for nt in (1, 7, 8, 9):
        assert np.array_equal(run_linear(sv, qm, xd, nt), y16[:nt]), f"nt={nt}"
    assert sv.spec_error_check(None) == 0


def test_linear_many_rows_column_groups(orc, dev):
    """R > 16 (several column groups in one launch, as the batched 12-sequence
    round uses): rows equal the nt <= 16 results bitwise."""
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    g = np.random.default_rng(5)
    N, K, R = 256, 512, 45
    w = synth.q_weight(g, 4, N, K)
    x = synth.f16_normal(g, (R, K))
    qm = sv.QMat(dev_weight(w, dev), max_rows=64)
    xd = torch.from_numpy(x.view(np.int16)).to(dev)
    yR = run_linear(sv, qm, xd, R)
    assert rel_err(yR, orc.linear(oracle_qweight(orc, w), x)) < 1e-5
    for r0 in (0, 16, 32, 40):
        nt = min(5, R - r0)
        y = torch.empty((nt, N), dtype=torch.float32, device=dev)
        sv.spec_linear_q(qm, xd[r0:r0 + nt].contiguous(), nt, y)
        assert np.array_equal(y.cpu().numpy(), yR[r0:r0 + nt])


def test_linear_rejects_bad_shapes(dev):
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    g = np.random.default_rng(6)
    w = synth.q_weight(g, 4, 32, 64)
    qm = sv.QMat(dev_weight(w, dev), max_rows=4)
    x = torch.zeros((8, 64), dtype=torch.int16, device=dev)
    y = torch.zeros((8, 32), dtype=torch.float32, device=dev)
    with pytest.raises(sv.SpecError):
        sv.spec_linear_q(qm, x, 5, y)        # above max_rows
    with pytest.raises(sv.SpecError):
        sv.spec_linear_q(qm, x, 0, y)
    bad = dict(dev_weight(w, dev), N=24)      # N % 16 != 0
    with pytest.raises(sv.SpecError):
        sv.QMat(bad)
