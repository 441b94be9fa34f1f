"""Shared helpers of the test suite: moving synthetic inputs to the device,
building small decoders on both sides, and the tolerance of the pages'
numbers."""
import numpy as np

from speculative_decoding_verification_round_gb300 import synth

# logits: |gpu - oracle| <= 2e-3 * (1 + |oracle|)
LOGIT_RTOL = 2e-3
# greedy ids must match wherever the oracle's top-1/top-2 margin exceeds this
MARGIN = 1e-2


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref) / (1.0 + np.abs(ref)))) if ref.size else 0.0


def top2_margin(row):
    part = np.partition(np.asarray(row, np.float64), -2)[-2:]
    return float(part[1] - part[0])


def dev_weight(w, dev):
    import torch
    return dict(qtype=w["qtype"], N=w["N"], K=w["K"],
                qs=torch.from_numpy(np.ascontiguousarray(w["qs"])).to(dev),
                qh=None if w["qh"] is None else torch.from_numpy(np.ascontiguousarray(w["qh"])).to(dev),
                scales=torch.from_numpy(np.ascontiguousarray(w["scales"]).view(np.int16)).to(dev))


def host_weight(w):
    """device dict -> numpy canonical planes (for the oracle)."""
    return dict(qtype=w["qtype"], N=w["N"], K=w["K"], qs=w["qs"].cpu().numpy(),
                qh=None if w["qh"] is None else w["qh"].cpu().numpy(),
                scales=w["scales"].cpu().view(__import__("torch").int16).numpy().view(np.uint16))


def oracle_qweight(orc, w):
    return orc.QWeight(w["qtype"], w["qs"], w["qh"], w["scales"], w["N"], w["K"])


def small_decoder(g, L=2, H=256, nq=4, nkv=2, hd=64, F=128, V=512, lm_qtype=6, mult=None,
                  qtype=4):
    """Layer linears in `qtype`, the LM head in `lm_qtype`.  Block scales
    default to the workloads' (|N(0,1)| * 0.01 for Q4, * 0.005 for Q6,
    * 0.000625 for Q8)."""
    mk = lambda qt, N, K: synth.q_weight(g, qt, N, K, mult=mult)
    raw = dict(wqkv=[mk(qtype, (nq + 2 * nkv) * hd, H) for _ in range(L)],
               wo=[mk(qtype, H, nq * hd) for _ in range(L)],
               wgu=[mk(qtype, 2 * F, H) for _ in range(L)],
               wd=[mk(qtype, H, F) for _ in range(L)], lm_head=mk(lm_qtype, V, H))
    raw["embed"] = synth.f16_normal(g, (V, H))
    raw["norm_w"] = synth.norm_gammas(g, 2 * L + 1, H)
    cfg = dict(n_layers=L, hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=hd, ffn=F, vocab=V)
    return cfg, raw


def to_device_model(sv, cfg, raw, dev, max_ctx, max_nt, max_seqs):
    import torch
    W = dict(wqkv=[dev_weight(w, dev) for w in raw["wqkv"]],
             wo=[dev_weight(w, dev) for w in raw["wo"]],
             wgu=[dev_weight(w, dev) for w in raw["wgu"]],
             wd=[dev_weight(w, dev) for w in raw["wd"]],
             lm_head=dev_weight(raw["lm_head"], dev),
             embed=torch.from_numpy(raw["embed"].view(np.int16)).to(dev),
             norm_w=torch.from_numpy(raw["norm_w"]).to(dev))
    desc = dict(cfg, max_ctx=max_ctx, max_nt=max_nt, max_seqs=max_seqs)
    return sv.Model(desc, W)


def to_oracle_model(orc, cfg, raw, max_ctx):
    Q = lambda w: oracle_qweight(orc, w)
    return orc.Model(cfg["n_layers"], cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"],
                     cfg["head_dim"], cfg["ffn"], cfg["vocab"], max_ctx, raw["embed"],
                     raw["norm_w"], [Q(w) for w in raw["wqkv"]], [Q(w) for w in raw["wo"]],
                     [Q(w) for w in raw["wgu"]], [Q(w) for w in raw["wd"]], Q(raw["lm_head"]))


def ill_conditioned_rows(om, tokens, n_past, kc, vc, ref, thresh):
    """Rows whose logits the ORACLE ITSELF cannot pin to the tolerance: the
    oracle's pass is repeated with every cached K element of layer 0 moved
    by one fp16 unit in the last place (fp16-level noise of the size that
    differently ordered, equally correct arithmetic leaves), and a row whose
    logits then move by more than `thresh` relative to 1 + |logit| is
    reported.  Such rows exist in the synthetic decoders: their hidden
    states collapse onto a shared direction, and a row whose coefficient on
    it is near zero flips with any rounding.  Returns (mask, per-row move)."""
    kp = kc.copy()
    kp[0] += 1  # one ulp (toward larger magnitude) on every element of layer 0
    out = om.forward(tokens, n_past, kp, vc.copy())
    move = np.array([rel_err(out[r], ref[r]) for r in range(ref.shape[0])])
    return move > thresh, move
