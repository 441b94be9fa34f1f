"""Seeded synthetic inputs for the verify round.

This module only draws random numbers and lays them out in the canonical
block formats; it holds none of the verify round's arithmetic.  Both the CUDA
path and the oracle are fed from here.

Canonical block layout (the pages name 4-bit, 6-bit and 8-bit block formats,
but do not fix the bits; this is the reading used throughout):
  * Q4, blocks of 32 along K: ``qs[n][b][16]`` bytes; byte j holds element j
    in its low nibble and element j+16 in its high nibble, stored as
    ``u = q + 8`` with ``q`` in [-8, 7].
  * Q6, blocks of 32: the low 4 bits of ``u = q + 32`` in ``qs`` (same nibble
    order), the high 2 bits in ``qh[n][b][8]``: element j at bits
    ``2*(j%4)`` of byte ``j//4``; ``q`` in [-32, 31].
  * Q8 (q8_0), blocks of 32: ``qs[n][b][32]`` bytes, byte j = element j as
    a two's-complement int8, ``q`` in [-128, 127].
  * ``scales[n][b]``: fp16 bits; weight = scale * q.

Workloads (value distributions of the pages' configurations):
  * WL_LMHEAD_GREEDY   H=1024, V=32000, d=2 (nt=3), Q4 LM head.
  * WL_ACCEPT_STOCH    12 sequences, d=7, V=248320, p-logits N(0,2),
                       q = p + N(0, 0.5), T=1.
  * WL_LINEAR_SWEEP    Q4 5120x13824 and Q6 13824x5120 (N_out x K_in),
                       nt in {1,2,3,4,8,9,16}.
  * WL_DECODER8        8 layers, H=4096, 32/8 heads, hd 128, FFN 14336,
                       Q6 LM head V=151936, 4096 cached positions, nt=8.
                       Q4 linears at the sweep's scale, LM head at LM_SCALE.
  * WL_DECODER14B      40 layers, H=5120, 40/8 heads, FFN 13824, Q6 LM head
                       V=248320, 12 sequences x 512 cached positions, nt=16,
                       T=0.7.
  * WL_LINEAR_SWEEP_Q8 q8_0 5120x13824 at the same nts.
  * WL_DRAFT05B        a 0.5B-class draft: 24 layers, H=896, 14/2 heads of
                       64, FFN 4864, V=151936, Q4 weights and LM head.
"""
from __future__ import annotations

import numpy as np

Q4_SCALE = 0.01   # fp16(|N(0,1)| * 0.01)
Q6_SCALE = 0.005  # fp16(|N(0,1)| * 0.005)
Q8_SCALE = 0.000625  # fp16(|N(0,1)| * 0.000625): the Q4 weights' range at 8 bits
# The decoder workloads' Q6 LM head: fp16(|N(0,1)| * 0.0015), which gives
# logits with a standard deviation of about 3 (at the sweep's 0.005 it is
# 9-12, far peakier than a language model's)
LM_SCALE = 0.0015

WL_LMHEAD_GREEDY = dict(name="lmhead_greedy_H1024_V32000_nt3", hidden=1024,
                        vocab=32000, d=2, p_agree=0.74, seed=0)
WL_ACCEPT_STOCH = dict(name="accept_stochastic_12seq_d7_V248320", n_seq=12, d=7,
                       vocab=248320, p_std=2.0, q_noise=0.5, temperature=1.0,
                       seed=0)
WL_LINEAR_SWEEP = dict(name="linear_sweep_q4_5120x13824_q6_13824x5120",
                       mats=[(4, 5120, 13824), (6, 13824, 5120)],
                       nts=[1, 2, 3, 4, 8, 9, 16], seed=0)
WL_LINEAR_SWEEP_Q8 = dict(name="linear_sweep_q8_5120x13824",
                          mats=[(8, 5120, 13824)], nts=[1, 2, 3, 4, 8, 9, 16], seed=1)
WL_DECODER8 = dict(name="decoder8_H4096_V151936_ctx4096_nt8", n_layers=8,
                   hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
                   ffn=14336, vocab=151936, ctx=4096, n_seq=1, d=7,
                   p_agree=0.74, lm_qtype=6, lm_scale=LM_SCALE, seed=0)
# The draft of the full-round measurement: a 0.5B-class decoder with 4-bit
# weights throughout (the pages pair their 7B/14B targets with a 0.5B q4_0
# draft): 24 layers of H=896, 14 query / 2 KV heads of 64, FFN 4864, the
# target's 151936-id vocabulary.
WL_DRAFT05B = dict(name="draft05b_24L_H896_V151936", n_layers=24, hidden=896,
                   n_q_heads=14, n_kv_heads=2, head_dim=64, ffn=4864, vocab=151936,
                   ctx=4096, n_seq=1, lm_qtype=4, lm_scale=LM_SCALE, seed=5)
WL_DECODER14B = dict(name="decoder14b_40L_H5120_V248320_12seq_ctx512_nt16",
                     n_layers=40, hidden=5120, n_q_heads=40, n_kv_heads=8,
                     head_dim=128, ffn=13824, vocab=248320, ctx=512, n_seq=12,
                     d=15, temperature=0.7, q_noise=0.5, lm_qtype=6, lm_scale=LM_SCALE,
                     seed=0)


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# host (numpy) generators, for sizes the oracle handles directly
# --------------------------------------------------------------------------
QT_RANGE = {4: (-8, 7), 6: (-32, 31), 8: (-128, 127)}
QT_SCALE = {4: Q4_SCALE, 6: Q6_SCALE, 8: Q8_SCALE}


def q_ints(g: np.random.Generator, qtype: int, N: int, K: int) -> np.ndarray:
    lo, hi = QT_RANGE[qtype]
    return g.integers(lo, hi + 1, size=(N, K), dtype=np.int8)


def pack_canonical(qtype: int, q: np.ndarray):
    """ints q[N][K] -> (qs[N][K/32][16] (Q8: [32]), qh[N][K/32][8] or None)."""
    N, K = q.shape
    assert K % 32 == 0
    if qtype == 8:  # one two's-complement byte per element, in element order
        return np.ascontiguousarray(q.astype(np.int8).view(np.uint8).reshape(N, K // 32, 32)), None
    u = (q.astype(np.int16) + (8 if qtype == 4 else 32)).astype(np.uint8)
    u = u.reshape(N, K // 32, 32)
    lo = u & 0xF
    qs = (lo[:, :, :16] | (lo[:, :, 16:] << 4)).astype(np.uint8)
    if qtype == 4:
        return np.ascontiguousarray(qs), None
    h2 = (u >> 4) & 0x3                                  # [N][nb][32]
    h2 = h2.reshape(N, K // 32, 8, 4)
    qh = (h2[..., 0] | (h2[..., 1] << 2) | (h2[..., 2] << 4) | (h2[..., 3] << 6))
    return np.ascontiguousarray(qs), np.ascontiguousarray(qh.astype(np.uint8))


def scales_f16(g: np.random.Generator, N: int, K: int, mult: float) -> np.ndarray:
    s = np.abs(g.standard_normal((N, K // 32))) * mult
    return s.astype(np.float16).view(np.uint16)


def q_weight(g: np.random.Generator, qtype: int, N: int, K: int, mult=None):
    """Returns dict(qtype, N, K, q (ints), qs, qh, scales (fp16 bits))."""
    mult = QT_SCALE[qtype] if mult is None else mult
    q = q_ints(g, qtype, N, K)
    qs, qh = pack_canonical(qtype, q)
    return dict(qtype=qtype, N=N, K=K, q=q, qs=qs, qh=qh,
                scales=scales_f16(g, N, K, mult))


def f16_normal(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return (g.standard_normal(shape) * std).astype(np.float16).view(np.uint16)


def norm_gammas(g: np.random.Generator, n: int, H: int) -> np.ndarray:
    """RMSNorm gains: 1 + 0.1 N(0,1), fp32."""
    return (1.0 + 0.1 * g.standard_normal((n, H))).astype(np.float32)


def greedy_drafts(g: np.random.Generator, target_ids, vocab: int, p_agree: float):
    """Each draft equals the given target token with probability p_agree,
    else a uniform random id (which may coincide with it by chance)."""
    target_ids = np.asarray(target_ids, np.int64)
    agree = g.random(target_ids.shape) < p_agree
    rand = g.integers(0, vocab, size=target_ids.shape)
    return np.where(agree, target_ids, rand).astype(np.int32)


def stochastic_logits(g: np.random.Generator, n_seq: int, d: int, V: int,
                      p_std: float = 2.0, q_noise: float = 0.5):
    """p[n_seq][d+1][V] ~ N(0, p_std^2); q[n_seq][d][V] = p[:, :d] + N(0, q_noise^2)."""
    p = (g.standard_normal((n_seq, d + 1, V), dtype=np.float32) * p_std)
    q = p[:, :d] + g.standard_normal((n_seq, d, V), dtype=np.float32) * q_noise
    return p.astype(np.float32), q.astype(np.float32)


# --------------------------------------------------------------------------
# device (torch) generators, for the full-size workloads
# --------------------------------------------------------------------------
def torch_gen(seed: int, device):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return gen


def q_weight_torch(gen, qtype: int, N: int, K: int, device, mult=None):
    """Uniform random planes on the device: a uniform byte is two uniform
    nibbles (u uniform in [0,15] <=> q uniform in [-8,7]); uniform qh bytes
    give uniform 2-bit fields (u uniform in [0,63] for Q6); a uniform Q8
    byte is q uniform in [-128,127]."""
    import torch
    mult = QT_SCALE[qtype] if mult is None else mult
    nb = K // 32
    qs = torch.randint(0, 256, (N, nb, 32 if qtype == 8 else 16), generator=gen,
                       device=device, dtype=torch.uint8)
    qh = None
    if qtype == 6:
        qh = torch.randint(0, 256, (N, nb, 8), generator=gen, device=device,
                           dtype=torch.uint8)
    sc = (torch.randn((N, nb), generator=gen, device=device).abs_() * mult)
    sc = sc.to(torch.float16)
    return dict(qtype=qtype, N=N, K=K, qs=qs, qh=qh, scales=sc)


def f16_normal_torch(gen, shape, device, std: float = 1.0):
    import torch
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.float16)


def decoder_weights_torch(wl: dict, device, seed=None):
    """All weights of a synthetic decoder workload, generated on `device`."""
    import torch
    gen = torch_gen(wl["seed"] if seed is None else seed, device)
    L, H, F = wl["n_layers"], wl["hidden"], wl["ffn"]
    hd, nq, nkv, V = wl["head_dim"], wl["n_q_heads"], wl["n_kv_heads"], wl["vocab"]
    nqkv = (nq + 2 * nkv) * hd
    W = dict(wqkv=[], wo=[], wgu=[], wd=[])
    for _ in range(L):
        W["wqkv"].append(q_weight_torch(gen, 4, nqkv, H, device))
        W["wo"].append(q_weight_torch(gen, 4, H, nq * hd, device))
        W["wgu"].append(q_weight_torch(gen, 4, 2 * F, H, device))
        W["wd"].append(q_weight_torch(gen, 4, H, F, device))
    W["lm_head"] = q_weight_torch(gen, wl.get("lm_qtype", 6), V, H, device, mult=wl.get("lm_scale"))
    W["embed"] = f16_normal_torch(gen, (V, H), device)
    g = torch.randn((2 * L + 1, H), generator=gen, device=device)
    W["norm_w"] = (1.0 + 0.1 * g).to(torch.float32)
    return W
