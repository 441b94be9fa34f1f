"""The tensor-core (tcgen05) verify GEMM of multi-sequence rounds
(spec_linear_q_tc) on the GPU.

Each weight reaches the tensor core as an exact pair of fp16 numbers, hi =
fp16(q * scale) and lo = q * scale - hi, so every product the MMA forms is
exact and the only difference from the oracle's fp64 sum is the tensor
core's fp32 accumulation: one chain of K / 8 accumulator updates per K
segment (a hi and a lo MMA per 16-k step).  The recursive-summation bound
for such a chain is (updates) * u * sum_k |w_k x_k| with u = 2^-23 (one unit
in the last place of an fp32 partial sum, whether the adder rounds or
truncates); the check below uses it.  The sharp check is against the error
one fp16 rounding of each weight would leave (sigma = 2^-11 / sqrt(3) *
sqrt(sum_k (w_k x_k)^2)): the error stays well below half of it, which
shows the split is exact.  Rows must not depend on the batch: every row
equals the same row computed in a batch of another size, bit for bit."""
import numpy as np
import pytest

from speculative_decoding_verification_round_gb300 import synth

from util import dev_weight, host_weight, oracle_qweight

pytestmark = pytest.mark.gpu


def acc_bound(K, s1):
    """Recursive summation of K / 8 updates in fp32 (products exact)."""
    return (K / 8.0) * 2.0 ** -23 * s1


@pytest.fixture(scope="module")
def dev():
    import torch
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


def run_tc(sv, qm, xd, R):
    import torch
    y = torch.empty((R, qm.N), dtype=torch.float32, device=xd.device)
    sv.spec_linear_q_tc(qm, xd[:R].contiguous(), R, y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def references(orc, w_host, x_bits):
    """(exact-weight product in fp64, sum_k |w_k x_k|, sum_k (w_k x_k)^2)."""
    W = orc.dequant(oracle_qweight(orc, w_host)).astype(np.float64)       # exact
    X = x_bits.view(np.float16).astype(np.float64)
    return X @ W.T, np.abs(X) @ np.abs(W).T, (X * X) @ (W * W).T


def check(y, refs, K):
    ref, s1, s2 = refs
    err = np.abs(y - ref)
    bound = acc_bound(K, s1)
    sigma = 2.0 ** -11 / np.sqrt(3.0) * np.sqrt(s2)   # what fp16-rounded weights would leave
    frac = float(np.max(err / np.maximum(sigma, 1e-30)))
    rel = err / (1.0 + np.abs(ref))
    print(f"  K {K}: max |y-ref|/(1+|ref|) = {rel.max():.2e}; max |y-ref| / summation bound = "
          f"{float(np.max(err / bound)):.3f}; max |y-ref| / rounding sigma = {frac:.3f}")
    assert (err <= bound).all(), float(np.max(err / bound))
    assert frac <= 0.5, frac


@pytest.mark.parametrize("qtype,N,K", [(4, 48, 96), (6, 272, 544), (8, 208, 1568), (4, 16, 32),
                                       (6, 144, 2080), (4, 400, 1056)])
def test_tc_small_matches_oracle(orc, dev, qtype, N, K):
    """Partial CTA tiles (N below 128, pairs past N), a ragged K tail, every
    format, several K segments; R below, at and above one 16-row step."""
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    g = np.random.default_rng(300 + N + K)
    w = synth.q_weight(g, qtype, N, K)
    x = synth.f16_normal(g, (40, K))
    qm = sv.QMat(dev_weight(w, dev), max_rows=40)
    xd = torch.from_numpy(x.view(np.int16)).to(dev)
    refs = references(orc, w, x)
    y40 = run_tc(sv, qm, xd, 40)
    check(y40, refs, K)
    for R in (1, 3, 16, 17, 33):
        assert np.array_equal(run_tc(sv, qm, xd, R), y40[:R]), f"row independence broken at R={R}"
    assert sv.spec_error_check(None) == 0


@pytest.mark.parametrize("qtype,N,K", [(4, 5120, 13824), (6, 13824, 5120), (8, 5120, 13824),
                                       (4, 27648, 5120), (4, 13920, 5120), (8, 10016, 5120),
                                       (4, 4096, 14336), (6, 28672, 4096), (8, 25616, 5120)])
def test_tc_full_size_matches_oracle(orc, dev, qtype, N, K):
    """The linear sweep's matrices, the batched workload's gate/up and the
    8-layer decoder's down and gate/up at the batched round's 192 rows (one
    full launch); rows at other batch sizes bitwise equal.  Cuts: K splits
    (5120x13824, 13824x5120, 4096x14336, ...) and one run per SM, whose runs
    end one tile and start the next (27648x5120, 28672x4096, 25616x5120);
    13920, 10016 and 25616 rows leave the last 256-row tile ragged (96, 32
    and 16 real rows)."""
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    gen = synth.torch_gen(40 + qtype, dev)
    wd = synth.q_weight_torch(gen, qtype, N, K, dev)
    x = synth.f16_normal_torch(gen, (300, K), dev)
    qm = sv.QMat(wd, max_rows=300)
    xb = x.view(torch.int16)
    y192 = run_tc(sv, qm, xb, 192)
    wh = host_weight(wd)
    xh = x.cpu().view(torch.int16).numpy().view(np.uint16)
    rows = np.r_[0:8, 100:108, 184:192]  # a sample of rows (the fp64 products are large)
    check(y192[rows], references(orc, wh, xh[rows]), K)
    y300 = run_tc(sv, qm, xb, 300)      # two launches: 192 + 108 rows
    assert np.array_equal(y300[:192], y192)
    for R in (1, 16, 100, 256):
        assert np.array_equal(run_tc(sv, qm, xb, R), y300[:R]), f"R={R}"
    check(y300[290:300], references(orc, wh, xh[290:300]), K)
    assert sv.spec_error_check(None) == 0
