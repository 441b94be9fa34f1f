"""spec_verify_attn on the GPU: against the oracle's fp64 causal GQA
attention, and row i of an nt-row batch bitwise equal to the nt = 1 call at
the same absolute position."""
import numpy as np
import pytest

from speculative_decoding_verification_round_gb300 import synth

from util import dev_weight

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    assert torch.cuda.is_available()
    return torch.device("cuda:0")


def attn_model(sv, dev, g, nq, nkv, hd, max_ctx, max_nt, max_seqs):
    """A one-layer model: only its KV cache and shapes matter here."""
    import torch
    H, F, V = 64, 32, 32
    mk = lambda qt, N, K: dev_weight(synth.q_weight(g, qt, N, K), dev)
    W = dict(wqkv=[mk(4, (nq + 2 * nkv) * hd, H)], wo=[mk(4, H, nq * hd)], wgu=[mk(4, 2 * F, H)],
             wd=[mk(4, H, F)], lm_head=mk(4, V, H),
             embed=torch.zeros((V, H), dtype=torch.int16, device=dev),
             norm_w=torch.ones((3, H), dtype=torch.float32, device=dev))
    return sv.Model(dict(n_layers=1, hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=hd, ffn=F,
                         vocab=V, max_ctx=max_ctx, max_nt=max_nt, max_seqs=max_seqs), W)


@pytest.mark.parametrize("nq,nkv,hd,n_seq,nt,n_past,max_ctx", [
    (32, 8, 128, 1, 8, 300, 400),      # GQA 4, three chunks with a ragged tail
    (40, 8, 128, 3, 16, 512, 600),     # GQA 5, 80 query rows per kv head
    (4, 4, 64, 2, 1, 0, 64),           # first position, no context
    (8, 2, 128, 1, 5, 123, 130),       # ends 2 positions before max_ctx
    (14, 2, 64, 1, 1, 4000, 4100),     # GQA 7 (the 0.5B-class draft), one decode row
    (14, 2, 64, 2, 3, 257, 300),       # GQA 7, two m tiles per kv head
])
def test_attention_matches_oracle_and_is_position_invariant(orc, dev, nq, nkv, hd, n_seq, nt,
                                                            n_past, max_ctx):
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    g = np.random.default_rng(nq * 7 + nt)
    m = attn_model(sv, dev, g, nq, nkv, hd, max_ctx, nt, n_seq)
    slots = list(range(n_seq))
    kc = synth.f16_normal(g, (n_seq, nkv, max_ctx, hd))
    vc = synth.f16_normal(g, (n_seq, nkv, max_ctx, hd))
    for s in slots:
        sv.spec_kv_fill(m, 0, s, 0, max_ctx, torch.from_numpy(kc[s].view(np.int16)).to(dev),
                        torch.from_numpy(vc[s].view(np.int16)).to(dev))
    pasts = [n_past + 3 * s for s in slots]
    pasts = [min(p, max_ctx - nt) for p in pasts]
    sv.spec_state_set(m, slots, n_past=pasts)
    R = n_seq * nt
    q = synth.f16_normal(g, (R, nq, hd))
    kn = synth.f16_normal(g, (R, nkv, hd))
    vn = synth.f16_normal(g, (R, nkv, hd))
    T = lambda a: torch.from_numpy(a.view(np.int16)).to(dev)
    sid = torch.tensor(slots, dtype=torch.int32, device=dev)
    out = torch.empty((R, nq * hd), dtype=torch.int16, device=dev)
    sv.spec_verify_attn(m, 0, n_seq, sid, nt, T(q), T(kn), T(vn), out)
    assert sv.spec_error_check(m) == 0
    got = out.cpu().numpy().view(np.float16).astype(np.float64).reshape(R, nq, hd)
    for s in slots:
        kcs, vcs = kc[s].copy(), vc[s].copy()
        for i in range(nt):
            kcs[:, pasts[s] + i] = kn[s * nt + i]
            vcs[:, pasts[s] + i] = vn[s * nt + i]
        ref = orc.attention(q[s * nt:(s + 1) * nt], kcs, vcs, np.arange(pasts[s], pasts[s] + nt))
        ref = ref.view(np.float16).astype(np.float64)
        # at most one fp16 rounding step apart: |d| <= 2^-10 |ref|
        err = np.max(np.abs(got[s * nt:(s + 1) * nt] - ref) / (1.0 + np.abs(ref)))
        assert err <= 2.0 ** -10, err
    # nt = 1 at each position reproduces each row bit for bit
    one = torch.empty((1, nq * hd), dtype=torch.int16, device=dev)
    for s in slots:
        for i in range(nt):
            r = s * nt + i
            sv.spec_state_set(m, [s], n_past=[pasts[s] + i])
            sv.spec_verify_attn(m, 0, 1, sid[s:s + 1], 1, T(q[r:r + 1]), T(kn[r:r + 1]),
                                T(vn[r:r + 1]), one)
            assert torch.equal(one[0], out[r]), (s, i)


def test_attention_rows_do_not_depend_on_the_batch(dev):
    """A sequence's rows are bitwise the same alone and in a batch of twelve
    (the batched workload's shape: GQA 5, 16 rows, m tiles in groups of two):
    the batch's chunk columns fill the SMs and take the build held to three
    CTAs an SM, the lone sequence's the two-CTA build."""
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    nq, nkv, hd, nt, max_ctx, n_seq = 40, 8, 128, 16, 600, 12
    g = np.random.default_rng(77)
    m = attn_model(sv, dev, g, nq, nkv, hd, max_ctx, nt, n_seq)
    kc = synth.f16_normal(g, (n_seq, nkv, max_ctx, hd))
    vc = synth.f16_normal(g, (n_seq, nkv, max_ctx, hd))
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)
    for s in range(n_seq):
        sv.spec_kv_fill(m, 0, s, 0, max_ctx, T(kc[s]), T(vc[s]))
    pasts = [500 + 7 * s for s in range(n_seq)]
    sv.spec_state_set(m, list(range(n_seq)), n_past=pasts)
    R = n_seq * nt
    q = synth.f16_normal(g, (R, nq, hd))
    kn = synth.f16_normal(g, (R, nkv, hd))
    vn = synth.f16_normal(g, (R, nkv, hd))
    sid = torch.arange(n_seq, dtype=torch.int32, device=dev)
    out = torch.empty((R, nq * hd), dtype=torch.int16, device=dev)
    sv.spec_verify_attn(m, 0, n_seq, sid, nt, T(q), T(kn), T(vn), out)
    alone = torch.empty((nt, nq * hd), dtype=torch.int16, device=dev)
    sv.spec_verify_attn(m, 0, 1, sid[:1], nt, T(q[:nt]), T(kn[:nt]), T(vn[:nt]), alone)
    assert sv.spec_error_check(m) == 0
    assert torch.equal(alone, out[:nt])
