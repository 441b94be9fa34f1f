"""Pins of the oracle's model math against things other than itself:
library routines (numpy/torch fp64), closed forms and invariants.
CPU only."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from speculative_decoding_verification_round_gb300 import synth


def test_f16_conversion_matches_numpy(orc):
    g = np.random.default_rng(1)
    x = np.concatenate([g.standard_normal(20000) * 10.0 ** g.integers(-8, 5, 20000),
                        [0.0, -0.0, 65504.0, 65520.0, 6.1e-5, 5.96e-8, 2.98e-8]])
    ours = orc.f64_to_f16_bits(x)
    ref = x.astype(np.float16).view(np.uint16)      # numpy rounds from double once
    assert np.array_equal(ours, ref)
    back = orc.f16_bits_to_f64(ref)
    assert np.array_equal(back, ref.view(np.float16).astype(np.float64))


@pytest.mark.parametrize("qtype", [4, 6, 8])
def test_unpack_round_trips_generator_ints(orc, qtype):
    g = np.random.default_rng(2)
    N, K = 48, 256
    w = synth.q_weight(g, qtype, N, K)
    # every representable int appears in the first row (exhaustive values)
    lo, hi = {4: (-8, 7), 6: (-32, 31), 8: (-128, 127)}[qtype]
    vals = np.arange(lo, hi + 1, dtype=np.int8)
    w["q"][0, :vals.size] = vals
    w["qs"], w["qh"] = synth.pack_canonical(qtype, w["q"])
    qw = orc.QWeight(qtype, w["qs"], w["qh"], w["scales"], N, K)
    deq = orc.dequant(qw)
    s = w["scales"].view(np.float16).astype(np.float32)
    expect = np.repeat(s, 32, axis=1) * w["q"].astype(np.float32)
    assert np.array_equal(deq, expect)


def test_q8_block_is_twos_complement_bytes_in_element_order(orc):
    """A q8_0 block written out by hand: byte j is element j as an int8
    (0x80 = -128, 0xff = -1, 0x7f = 127), times the block's fp16 scale."""
    blk = np.array([0x00, 0x01, 0x7f, 0x80, 0x81, 0xff, 0xfe, 0x40] + list(range(0x10, 0x28)),
                   np.uint8)
    qs = np.stack([blk, blk[::-1]]).reshape(1, 2, 32)
    scales = np.array([[0.5, -0.25]], np.float16).view(np.uint16)
    deq = orc.dequant(orc.QWeight(8, qs, None, scales, 1, 64))[0]
    first = [0, 1, 127, -128, -127, -1, -2, 64] + list(range(16, 40))
    assert deq[:32].tolist() == [0.5 * v for v in first]
    assert deq[32:].tolist() == [-0.25 * v for v in first[::-1]]


@pytest.mark.parametrize("qtype", [4, 6, 8])
def test_one_hot_activation_returns_weight_column(orc, qtype):
    g = np.random.default_rng(3)
    N, K = 40, 128
    w = synth.q_weight(g, qtype, N, K)
    qw = orc.QWeight(qtype, w["qs"], w["qh"], w["scales"], N, K)
    ks = [0, 17, 31, 32, 100, 127]
    x = np.zeros((len(ks), K), np.float64)
    for r, k in enumerate(ks):
        x[r, k] = 1.0
    y = orc.linear(qw, x.astype(np.float16).view(np.uint16))
    s = w["scales"].view(np.float16).astype(np.float32)
    for r, k in enumerate(ks):
        expect = s[:, k // 32] * w["q"][:, k].astype(np.float32)
        assert np.array_equal(y[r], expect)


@pytest.mark.parametrize("qtype,N,K,R", [(4, 64, 512, 3), (6, 80, 320, 9), (4, 16, 32, 1),
                                         (8, 48, 288, 5)])
def test_linear_matches_numpy_float64_matmul(orc, qtype, N, K, R):
    g = np.random.default_rng(4)
    w = synth.q_weight(g, qtype, N, K)
    x = synth.f16_normal(g, (R, K))
    qw = orc.QWeight(qtype, w["qs"], w["qh"], w["scales"], N, K)
    y = orc.linear(qw, x)
    wd = (np.repeat(w["scales"].view(np.float16).astype(np.float64), 32, axis=1)
          * w["q"].astype(np.float64))
    ref = x.view(np.float16).astype(np.float64) @ wd.T
    assert np.allclose(y, ref.astype(np.float32), rtol=1e-6, atol=1e-6)
    assert np.max(np.abs(y - ref) / (1 + np.abs(ref))) < 1e-6


def test_rmsnorm_matches_torch(orc):
    g = np.random.default_rng(5)
    h = (g.standard_normal((7, 96)) * 3).astype(np.float32)
    gamma = synth.norm_gammas(g, 1, 96)[0]
    out = orc.rmsnorm(h, gamma, 1e-6).view(np.float16).astype(np.float64)
    ref = F.rms_norm(torch.from_numpy(h).double(), (96,), torch.from_numpy(gamma).double(),
                     eps=1e-6)
    ref16 = ref.numpy().astype(np.float16).astype(np.float64)
    assert np.array_equal(out, ref16) or np.max(np.abs(out - ref16)) <= 2 ** -10 * np.max(np.abs(ref16))
    # scale invariance (eps negligible) and unit RMS with gamma = 1
    out2 = orc.rmsnorm(h * 8.0, gamma, 1e-6).view(np.float16)
    assert np.array_equal(out2, orc.rmsnorm(h, gamma, 1e-6).view(np.float16))
    u = orc.rmsnorm(h, np.ones(96, np.float32), 0.0).view(np.float16).astype(np.float64)
    assert np.allclose(np.sqrt(np.mean(u ** 2, axis=1)), 1.0, atol=2e-3)


def test_rope_against_complex_rotation_and_invariants(orc):
    g = np.random.default_rng(6)
    hd, theta = 128, 10000.0
    x = g.standard_normal((5, hd)).astype(np.float32)
    pos = np.array([0, 1, 17, 4095, 100000])
    out = orc.rope(x, pos, theta).view(np.float16).astype(np.float64)
    # textbook: (x_i + j x_{i+64}) * exp(j * pos * theta^(-2i/hd))
    f = theta ** (-2.0 * np.arange(hd // 2) / hd)
    z = (x[:, :hd // 2] + 1j * x[:, hd // 2:]) * np.exp(1j * pos[:, None] * f[None, :])
    ref = np.concatenate([z.real, z.imag], axis=1)
    assert np.allclose(out, ref, rtol=2e-3, atol=2e-3)
    assert np.array_equal(out[0], x[0].astype(np.float16).astype(np.float64))  # pos 0 = identity
    # relative-position property: <R(p) q, R(p') k> depends on p - p' only
    qv = g.standard_normal((1, hd)).astype(np.float32)
    kv = g.standard_normal((1, hd)).astype(np.float32)

    def dot(pq, pk):
        a = orc.rope(qv, [pq], theta).view(np.float16).astype(np.float64)
        b = orc.rope(kv, [pk], theta).view(np.float16).astype(np.float64)
        return float((a * b).sum())
    assert abs(dot(10, 3) - dot(1007, 1000)) < 0.05


def test_attention_matches_torch_sdpa(orc):
    g = np.random.default_rng(7)
    rows, nq, nkv, hd, max_ctx = 4, 8, 2, 64, 40
    n_past = 30
    q = synth.f16_normal(g, (rows, nq, hd))
    kc = synth.f16_normal(g, (nkv, max_ctx, hd))
    vc = synth.f16_normal(g, (nkv, max_ctx, hd))
    pos = np.arange(n_past, n_past + rows)
    out = orc.attention(q, kc, vc, pos).view(np.float16).astype(np.float64)
    qt = torch.from_numpy(q.view(np.float16).astype(np.float64)).permute(1, 0, 2)[None]
    kt = torch.from_numpy(kc.view(np.float16).astype(np.float64))[None]
    vt = torch.from_numpy(vc.view(np.float16).astype(np.float64))[None]
    mask = torch.arange(max_ctx)[None, :] <= torch.from_numpy(pos)[:, None]
    ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, enable_gqa=True)
    ref = ref[0].permute(1, 0, 2).numpy()
    assert np.allclose(out, ref, atol=2e-3, rtol=2e-3)


def test_swiglu_matches_torch_silu(orc):
    g = np.random.default_rng(8)
    a = (g.standard_normal(1000) * 4).astype(np.float32)
    b = (g.standard_normal(1000) * 4).astype(np.float32)
    out = orc.swiglu(a, b).view(np.float16).astype(np.float64)
    ref = (F.silu(torch.from_numpy(a).double()) * torch.from_numpy(b).double()).numpy()
    assert np.allclose(out, ref, rtol=1e-3, atol=1e-4)
    assert orc.swiglu(np.zeros(1, np.float32), np.ones(1, np.float32))[0] == 0


# --------------------------------------------------------------------------
# the full verify-round forward of a tiny decoder
# --------------------------------------------------------------------------
TINY = dict(n_layers=2, hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16, ffn=96,
            vocab=50, max_ctx=24)


def tiny_model(orc, seed=9, **over):
    cfg = dict(TINY, **over)
    g = np.random.default_rng(seed)
    L, H, F_, hd = cfg["n_layers"], cfg["hidden"], cfg["ffn"], cfg["head_dim"]
    nq, nkv, V = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["vocab"]
    mk = lambda qt, N, K: synth.q_weight(g, qt, N, K, mult=0.05)
    raw = dict(wqkv=[mk(4, (nq + 2 * nkv) * hd, H) for _ in range(L)],
               wo=[mk(4, H, nq * hd) for _ in range(L)],
               wgu=[mk(4, 2 * F_, H) for _ in range(L)],
               wd=[mk(4, H, F_) for _ in range(L)], lm=mk(6, V, H))
    Q = lambda w: orc.QWeight(w["qtype"], w["qs"], w["qh"], w["scales"], w["N"], w["K"])
    embed = synth.f16_normal(g, (V, H))
    norm_w = synth.norm_gammas(g, 2 * L + 1, H)
    m = orc.Model(L, H, nq, nkv, hd, F_, V, cfg["max_ctx"], embed, norm_w,
                  [Q(w) for w in raw["wqkv"]], [Q(w) for w in raw["wo"]],
                  [Q(w) for w in raw["wgu"]], [Q(w) for w in raw["wd"]], Q(raw["lm"]))
    return m, raw, embed, norm_w, cfg


def empty_cache(cfg, n_seq, g=None):
    shape = (cfg["n_layers"], n_seq, cfg["n_kv_heads"], cfg["max_ctx"], cfg["head_dim"])
    if g is None:
        return np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    return synth.f16_normal(g, shape), synth.f16_normal(g, shape)


def torch_forward(raw, embed, norm_w, cfg, tokens, n_past, kc, vc):
    """Library-routine composition of the same decoder in fp64 torch
    (F.rms_norm, complex-rotation RoPE, F.scaled_dot_product_attention with
    GQA, F.silu), for one sequence.  Roundings to fp16 at the same points."""
    d64 = lambda w: torch.from_numpy(np.repeat(w["scales"].view(np.float16).astype(np.float64), 32, 1)
                                     * w["q"].astype(np.float64))
    r16 = lambda t: t.to(torch.float16).to(torch.float64)
    L, H, hd = cfg["n_layers"], cfg["hidden"], cfg["head_dim"]
    nq, nkv, Fd = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["ffn"]
    nt = len(tokens)
    pos = torch.arange(n_past, n_past + nt)
    h = torch.from_numpy(embed.view(np.float16)[tokens].astype(np.float64))
    kc = torch.from_numpy(kc.view(np.float16).astype(np.float64)).clone()
    vc = torch.from_numpy(vc.view(np.float16).astype(np.float64)).clone()
    f = 10000.0 ** (-2.0 * torch.arange(hd // 2, dtype=torch.float64) / hd)
    rot = torch.polar(torch.ones(nt, hd // 2, dtype=torch.float64), pos[:, None] * f[None, :])

    def rope(x):  # x [nt][heads][hd]
        z = torch.complex(x[..., :hd // 2], x[..., hd // 2:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], -1)
    for l in range(L):
        nw = torch.from_numpy(norm_w.astype(np.float64))
        x = r16(F.rms_norm(h, (H,), nw[2 * l], eps=1e-6))
        qkv = (x @ d64(raw["wqkv"][l]).T).float().double()
        q = r16(rope(qkv[:, :nq * hd].reshape(nt, nq, hd)))
        k = r16(rope(qkv[:, nq * hd:(nq + nkv) * hd].reshape(nt, nkv, hd)))
        v = r16(qkv[:, (nq + nkv) * hd:].reshape(nt, nkv, hd))
        kc[l, 0, :, n_past:n_past + nt] = k.permute(1, 0, 2)
        vc[l, 0, :, n_past:n_past + nt] = v.permute(1, 0, 2)
        mask = torch.arange(cfg["max_ctx"])[None, :] <= pos[:, None]
        a = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], kc[l, 0][None],
                                           vc[l, 0][None], attn_mask=mask, enable_gqa=True)
        a = r16(a[0].permute(1, 0, 2).reshape(nt, nq * hd))
        h = (h + (a @ d64(raw["wo"][l]).T).float().double()).float().double()
        x = r16(F.rms_norm(h, (H,), nw[2 * l + 1], eps=1e-6))
        gu = (x @ d64(raw["wgu"][l]).T).float().double()
        s = r16(F.silu(gu[:, :Fd]) * gu[:, Fd:])
        h = (h + (s @ d64(raw["wd"][l]).T).float().double()).float().double()
    x = r16(F.rms_norm(h, (H,), torch.from_numpy(norm_w[2 * L].astype(np.float64)), eps=1e-6))
    return (x @ d64(raw["lm"]).T).float().numpy()


def test_forward_matches_library_composition(orc):
    m, raw, embed, norm_w, cfg = tiny_model(orc)
    g = np.random.default_rng(10)
    kc, vc = empty_cache(cfg, 1, g)
    tokens = np.array([[3, 7, 7, 41, 0]], np.int32)
    n_past = 11
    ref = torch_forward(raw, embed, norm_w, cfg, tokens[0], n_past, kc.copy(), vc.copy())
    logits = m.forward(tokens, [n_past], kc, vc)
    assert np.max(np.abs(logits - ref) / (1 + np.abs(ref))) < 2e-3


def test_forward_rows_equal_sequential_nt1_and_are_causal(orc):
    """Verify rows at nt = d+1 equal d+1 single-row passes at the same
    positions (the weights-once batch is only a batching of the same math),
    and a row never depends on later drafted tokens."""
    m, raw, embed, norm_w, cfg = tiny_model(orc, seed=11)
    g = np.random.default_rng(12)
    kc0, vc0 = empty_cache(cfg, 1, g)
    tokens = np.array([[5, 9, 2, 33]], np.int32)
    n_past = 6
    kc, vc = kc0.copy(), vc0.copy()
    batched = m.forward(tokens, [n_past], kc, vc)
    kc1, vc1 = kc0.copy(), vc0.copy()
    for i in range(tokens.shape[1]):
        row = m.forward(tokens[:, i:i + 1], [n_past + i], kc1, vc1)
        assert np.array_equal(row[0], batched[i])
    assert np.array_equal(kc, kc1) and np.array_equal(vc, vc1)
    # causality: changing the last draft leaves earlier rows unchanged
    t2 = tokens.copy()
    t2[0, -1] = 44
    other = m.forward(t2, [n_past], kc0.copy(), vc0.copy())
    assert np.array_equal(other[:-1], batched[:-1])
    assert not np.array_equal(other[-1], batched[-1])


def test_forward_multi_sequence_is_per_sequence(orc):
    m, raw, embed, norm_w, cfg = tiny_model(orc, seed=13)
    g = np.random.default_rng(14)
    kc, vc = empty_cache(cfg, 3, g)
    tokens = np.array([[1, 2, 3], [4, 5, 6], [7, 8, 9]], np.int32)
    n_past = [2, 9, 15]
    both = m.forward(tokens, n_past, kc.copy(), vc.copy())
    for s in range(3):
        ks, vs = np.ascontiguousarray(kc[:, s:s + 1]), np.ascontiguousarray(vc[:, s:s + 1])
        one = m.forward(tokens[s:s + 1], [n_past[s]], ks, vs)
        assert np.array_equal(one, both[3 * s:3 * s + 3])


def test_zero_layer_model_is_lm_head_of_normed_embedding(orc):
    m, raw, embed, norm_w, cfg = tiny_model(orc, seed=15, n_layers=0)
    kc, vc = empty_cache(cfg, 1)
    tokens = np.array([[4, 8]], np.int32)
    logits = m.forward(tokens, [0], kc, vc)
    x = orc.rmsnorm(embed.view(np.float16)[tokens[0]].astype(np.float32), norm_w[0], 1e-6)
    assert np.array_equal(logits, orc.linear(m.lm_head, x))
