"""Benchmark of the verify round on one GB300 (or N replicas).

Step = one full greedy verify round (spec_verify_round) of the synthetic
8-layer decoder: H=4096, 32 q / 8 kv heads of 128, SwiGLU FFN 14336, Q4
linears, Q6 LM head over V=151936, 4096 cached positions, nt = 8 (anchor +
7 drafts).  Drafts follow the target's own greedy chain with probability 0.74
per position; they are recorded by an untimed pass of the same chain, and
the timed steps replay that chain from the same starting state (every step
recomputes the whole target pass: nothing is cached between steps).

Printed JSON line: value = emitted tokens per second of the rounds (accepted
drafts + the one correction/bonus token per round), plus the verify-round
latency, the weight-stream bandwidth of the verify GEMM against the HBM
roofline, the nt sweep of the linear layers, the end-to-end number through
host buffers, and the oracle's CPU rate.

--impl reference times the CPU oracle (the plain fp64 reference of the same
round) on the host cores, on the same workload and metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verify-round µs at nt=1..16; weight-stream HBM GB/s vs peak; accepted tok/s"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# --------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)
# --------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path=None):
        import tempfile
        self.gpu = gpu_index
        self.proc = None
        self.start_line = 0
        self.path = path or os.path.join(tempfile.gettempdir(),
                                         f"spec_verify_clocks_rank{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            # the first sample takes a while: start timing only once it is there
            t0 = time.time()
            while time.time() - t0 < 5.0 and self.proc.poll() is None and self._lines() == 0:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        self.start_line = self._lines()
        return self

    def _lines(self) -> int:
        try:
            with open(self.path) as f:
                return sum(1 for _ in f)
        except OSError:
            return 0

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows, before = [], []
        for n, line in enumerate(open(self.path)):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                (rows if n >= self.start_line else before).append(parts)
        if not rows and before:
            rows = before[-1:]  # the timed region was shorter than the sampling interval
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------------------
# the workload
# --------------------------------------------------------------------------
# HBM bytes per weight of each block format: the integers plus one fp16
# scale per 32
WEIGHT_BYTES = {4: 0.5625, 6: 0.8125, 8: 1.0625}


def build_model(sv, synth, wl, dev, max_ctx):
    W = synth.decoder_weights_torch(wl, dev)
    desc = dict(n_layers=wl["n_layers"], hidden=wl["hidden"], n_q_heads=wl["n_q_heads"],
                n_kv_heads=wl["n_kv_heads"], head_dim=wl["head_dim"], ffn=wl["ffn"],
                vocab=wl["vocab"], max_ctx=max_ctx, max_nt=sv.SPEC_MAX_NT, max_seqs=wl["n_seq"])
    return sv.Model(desc, W), W


def fill_context(sv, synth, m, wl, dev, seed=1):
    import torch
    gen = synth.torch_gen(seed, dev)
    for l in range(wl["n_layers"]):
        for s in range(wl["n_seq"]):
            k = synth.f16_normal_torch(gen, (wl["n_kv_heads"], wl["ctx"], wl["head_dim"]), dev)
            v = synth.f16_normal_torch(gen, (wl["n_kv_heads"], wl["ctx"], wl["head_dim"]), dev)
            sv.spec_kv_fill(m, l, s, 0, wl["ctx"], k.view(torch.int16), v.view(torch.int16))
    torch.cuda.synchronize()


def record_chain(sv, synth, m, wl, dev, n_rounds, anchor, rng):
    """Untimed: run the speculative chain once, drafting from the target's
    own greedy continuation (nt = 1 passes from a saved state) with
    agreement probability p per position.  Returns the per-round drafts."""
    import torch
    d, V = wl["d"], wl["vocab"]
    sid = torch.zeros(1, dtype=torch.int32, device=dev)
    n_acc = torch.zeros(1, dtype=torch.int32, device=dev)
    em = torch.zeros((1, d + 1), dtype=torch.int32, device=dev)
    em1 = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    sv.spec_state_set(m, [0], n_past=[wl["ctx"]], emit_idx=[0], anchor=[anchor])
    drafts = []
    for _ in range(n_rounds):
        n_past, ei, anc = sv.spec_state_get(m, [0])
        chain, tok = [], anc[0]
        for i in range(d):
            sv.spec_state_set(m, [0], n_past=[n_past[0] + i], anchor=[tok])
            sv.spec_verify_round(m, 1, sid, None, 0, n_acc=n_acc, emitted=em1)
            true_next = int(em1.item())
            tok = true_next if rng.random() < wl["p_agree"] else int(rng.integers(0, V))
            chain.append(tok)
        sv.spec_state_set(m, [0], n_past=n_past, emit_idx=ei, anchor=anc)
        dr = torch.tensor([chain], dtype=torch.int32, device=dev)
        sv.spec_verify_round(m, 1, sid, dr, d, n_acc=n_acc, emitted=em)
        drafts.append(chain)
    assert sv.spec_error_check(m) == 0
    return drafts


class L2Flush:
    """Evicts L2 by READING a buffer twice the L2 size (a write would leave
    dirty lines whose write-back the next kernel would pay for)."""

    def __init__(self, dev):
        import torch
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.buf = torch.ones(max(2 * l2, 64 << 20) // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.buf.amax()


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "linear_q_traffic_decoder8_nt8.json")
LINEAR_SRC = os.path.join(ROOT, "speculative_decoding_verification_round_gb300", "csrc", "linear.cu")


def measured_traffic(shapes):
    """DRAM bytes per verify-GEMM launch over one round's launch mix, from the
    committed ncu record of these shapes -- or None when the record is
    missing, lacks a shape, or was taken on a different linear.cu."""
    import hashlib
    try:
        rec = json.load(open(TRAFFIC_RECORD))
        sha = hashlib.sha256(open(LINEAR_SRC, "rb").read()).hexdigest()
    except (OSError, ValueError):
        return None
    if rec.get("linear_cu_sha256") != sha:
        return None
    total, n = 0.0, 0
    for qt, N, K, count in shapes:
        b = rec.get("dram_bytes_per_launch", {}).get(f"{qt}:{N}:{K}")
        if b is None:
            return None
        total += b * count
        n += count
    return total / n


def time_dominant_kernel(sv, synth, wl, dev, hbm_peak, reps=20):
    """The verify GEMM at the decoder's shapes, nt = 8, timed alone with CUDA
    events on its stream; L2 flushed between launches.  Returns the achieved
    weight-stream GB/s over one round's mix of launches (8 x [qkv, o,
    gate/up, down] + the LM head)."""
    import torch
    H, F, hd, nq, nkv, V = (wl["hidden"], wl["ffn"], wl["head_dim"], wl["n_q_heads"],
                            wl["n_kv_heads"], wl["vocab"])
    shapes = [(4, (nq + 2 * nkv) * hd, H, wl["n_layers"]), (4, H, nq * hd, wl["n_layers"]),
              (4, 2 * F, H, wl["n_layers"]), (4, H, F, wl["n_layers"]), (6, V, H, 1)]
    gen = synth.torch_gen(5, dev)
    st = torch.cuda.current_stream()
    flush = L2Flush(dev)
    nt = wl["d"] + 1
    total_bytes, total_s, per = 0.0, 0.0, []
    for qt, N, K, count in shapes:
        w = synth.q_weight_torch(gen, qt, N, K, dev)
        qm = sv.QMat(w, max_rows=16)
        x = synth.f16_normal_torch(gen, (nt, K), dev).view(torch.int16)
        y = torch.empty((nt, N), dtype=torch.float32, device=dev)
        nbytes = N * K * WEIGHT_BYTES[qt] + nt * K * 2 + nt * N * 4
        times = []
        for i in range(reps + 3):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            sv.spec_linear_q(qm, x, nt, y, st)
            e1.record(st)
            e1.synchronize()
            if i >= 3:
                times.append(e0.elapsed_time(e1) * 1e-3)
        t = statistics.median(times)
        per.append({"qtype": qt, "N": N, "K": K, "us": t * 1e6, "gbs": nbytes / t / 1e9})
        total_bytes += nbytes * count
        total_s += t * count
        qm.close()
        del w
    gbs = total_bytes / total_s / 1e9
    return gbs, per, total_bytes / (4 * wl["n_layers"] + 1), measured_traffic(shapes)


ROUND_SWEEP_NTS = (1, 2, 3, 4, 8, 9, 16)
ROUND_SWEEP_GROUP = 10


def round_sweep(sv, m, wl, dev, groups=5):
    """Greedy verify rounds of the workload's model at each nt (d = nt - 1
    random drafts, graphs replayed): the state is reset before each group of
    ROUND_SWEEP_GROUP back-to-back rounds; median over groups of the mean
    round time (us), and the worst nt = 9..16 round over the nt = 1 round."""
    import torch
    rng = np.random.default_rng(7)
    sid = torch.zeros(1, dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream()
    us = {}
    for nt in ROUND_SWEEP_NTS:
        d = nt - 1
        dr = torch.from_numpy(rng.integers(0, wl["vocab"], (1, max(d, 1))).astype(np.int32)).to(dev)
        n_acc = torch.zeros(1, dtype=torch.int32, device=dev)
        em = torch.zeros((1, nt), dtype=torch.int32, device=dev)
        times = []
        for grp in range(groups + 1):
            sv.spec_state_set(m, [0], n_past=[wl["ctx"]], emit_idx=[0], anchor=[1234])
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(ROUND_SWEEP_GROUP):
                sv.spec_verify_round(m, 1, sid, dr if d else None, d, n_acc=n_acc, emitted=em)
            e1.record(st)
            e1.synchronize()
            if grp > 0:  # the first group captures the graph and warms up
                times.append(e0.elapsed_time(e1) * 1e3 / ROUND_SWEEP_GROUP)
        us[str(nt)] = round(statistics.median(times), 2)
    worst = max(us[str(n)] for n in ROUND_SWEEP_NTS if n >= 9)
    return {"us": us, "nt9_16_over_nt1": round(worst / us["1"], 3)}


def greedy_continuation(sv, m, wl, dev, d, rng, sid, n_acc, em1, p_agree):
    """Untimed: the target's own greedy continuation of sequence 0 for d
    positions (nt = 1 passes from a saved state, restored after), each
    position kept with probability p_agree, else a random id -- the drafts
    of one round at depth d."""
    n_past, ei, anc = sv.spec_state_get(m, [0])
    chain, tok = [], anc[0]
    for i in range(d):
        sv.spec_state_set(m, [0], n_past=[n_past[0] + i], anchor=[tok])
        sv.spec_verify_round(m, 1, sid, None, 0, n_acc=n_acc, emitted=em1)
        true_next = int(em1.item())
        tok = true_next if rng.random() < p_agree else int(rng.integers(0, wl["vocab"]))
        chain.append(tok)
    sv.spec_state_set(m, [0], n_past=n_past, emit_idx=ei, anchor=anc)
    return chain


ADAPTIVE_ROUNDS = 64
# (name, per-position draft agreement, deepest depth the controller may pick):
# the workload's agreement with the controller's default cap of 7, and a
# near-perfect drafter allowed the full 16-row verify block
ADAPTIVE_CASES = (("p0.74_dmax7", None, 7), ("p0.95_dmax15", 0.95, 15))


def adaptive_depth_run(sv, m, wl, dev, rounds=ADAPTIVE_ROUNDS):
    """The adaptive draft-depth controller in the loop: each round's depth
    comes from the controller, its drafts from the target's own greedy chain
    (agreement p_agree per position), and the round's CUDA-event time plus
    its accept count go back to the controller.  The same loop at the fixed
    depth 7 runs beside it.  Reported per case: emitted tokens per second of
    verify time, the depths chosen, and the controller's host time per call
    (median, through the Python binding)."""
    import torch
    sid = torch.zeros(1, dtype=torch.int32, device=dev)
    n_acc = torch.zeros(1, dtype=torch.int32, device=dev)
    em1 = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream()
    # capture every depth's graph first, so that no timed round pays for it
    for d in range(sv.SPEC_MAX_NT):
        em = torch.zeros((1, d + 1), dtype=torch.int32, device=dev)
        dr = torch.zeros((1, d), dtype=torch.int32, device=dev) if d else None
        sv.spec_state_set(m, [0], n_past=[wl["ctx"]], emit_idx=[0], anchor=[1234])
        sv.spec_verify_round(m, 1, sid, dr, d, n_acc=n_acc, emitted=em)
    torch.cuda.synchronize()
    out = {"rounds": rounds}
    for name, p_agree, d_max in ADAPTIVE_CASES:
        p_agree = wl["p_agree"] if p_agree is None else p_agree
        case = {"p_agree": p_agree, "d_max": d_max}
        for mode in ("adaptive", "static7"):
            rng = np.random.default_rng(11)
            sv.spec_state_set(m, [0], n_past=[wl["ctx"]], emit_idx=[0], anchor=[1234])
            ctl = sv.DepthController(d_max=d_max) if mode == "adaptive" else None
            tokens, secs, ctl_t, hist = 0, 0.0, [], {}
            for _ in range(rounds):
                d = ctl.next_depth() if ctl is not None else 7
                chain = greedy_continuation(sv, m, wl, dev, d, rng, sid, n_acc, em1, p_agree)
                dr = torch.tensor([chain], dtype=torch.int32, device=dev) if d else None
                em = torch.zeros((1, d + 1), dtype=torch.int32, device=dev)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                sv.spec_verify_round(m, 1, sid, dr, d, n_acc=n_acc, emitted=em)
                e1.record(st)
                e1.synchronize()
                t = e0.elapsed_time(e1) * 1e-3
                a = int(n_acc.item())
                tokens += a + 1
                secs += t
                hist[str(d)] = hist.get(str(d), 0) + 1
                if ctl is not None:
                    t0 = time.perf_counter()
                    ctl.observe(d, [a], t)
                    ctl_t.append(time.perf_counter() - t0)
            case[mode] = {"tok_per_s": round(tokens / secs, 1), "depths": hist}
            if ctl is not None:
                case[mode]["controller_us_per_call"] = round(statistics.median(ctl_t) * 1e6, 2)
                ctl.close()
        out[name] = case
    return out


FULL_ROUND_DRAFT_LAYERS = (6, 24)
FULL_ROUND_REPS = 24


def full_round_run(sv, synth, m, wl, dev, max_ctx, rounds=ADAPTIVE_ROUNDS):
    """Whole rounds with the draft phase timed in ("Speculative Decoding
    (D5-R) -- Plan", section 3: d sequential nt = 1 draft forwards, then one
    nt = d + 1 target forward).  The draft is a 0.5B-class decoder on the same
    engine: each draft forward is its graph-replayed d = 0 round, whose greedy
    commit makes its token the next forward's input, all on the device.  Its
    random-weight tokens are computed and dropped: the target verifies drafts
    from its own greedy chain at agreement p_agree (synthetic acceptance), so
    only the draft's cost enters.  Two draft depths: 6 layers (a quarter of
    the 0.5B's 24, as the 8-layer target is a quarter-depth 32-layer model)
    and the full 24.  Per depth d = 0..7: median round time and draft time per
    token, emitted tokens per second as measured and as expected from the
    agreement (E(d) over the median round time; the best static depth is
    chosen on the latter); then the adaptive controller with d_min = 0
    (d = 0 is plain decoding) on these round times."""
    import torch
    st = torch.cuda.current_stream()
    sid = torch.zeros(1, dtype=torch.int32, device=dev)
    n_acc = torch.zeros(1, dtype=torch.int32, device=dev)
    dn = torch.zeros(1, dtype=torch.int32, device=dev)
    dem = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    em1 = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    out = {"draft_shape": synth.WL_DRAFT05B["name"], "p_agree": wl["p_agree"]}
    for n_layers in FULL_ROUND_DRAFT_LAYERS:
        dwl = dict(synth.WL_DRAFT05B, n_layers=n_layers)
        dm, W = build_model(sv, synth, dwl, dev, max_ctx)
        del W
        fill_context(sv, synth, dm, dwl, dev, seed=7)

        def one_round(d, rng):
            sv.spec_state_set(m, [0], n_past=[wl["ctx"]], emit_idx=[0], anchor=[1234])
            sv.spec_state_set(dm, [0], n_past=[wl["ctx"]], emit_idx=[0], anchor=[1234])
            chain = greedy_continuation(sv, m, wl, dev, d, rng, sid, n_acc, em1, wl["p_agree"])
            dr = torch.tensor([chain], dtype=torch.int32, device=dev) if d else None
            em = torch.zeros((1, d + 1), dtype=torch.int32, device=dev)
            torch.cuda.synchronize()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(st)
            for _ in range(d):
                sv.spec_verify_round(dm, 1, sid, None, 0, n_acc=dn, emitted=dem)
            ev[1].record(st)
            sv.spec_verify_round(m, 1, sid, dr, d, n_acc=n_acc, emitted=em)
            ev[2].record(st)
            ev[2].synchronize()
            return (ev[0].elapsed_time(ev[2]) * 1e-3, ev[0].elapsed_time(ev[1]) * 1e-3,
                    int(n_acc.item()))

        rng = np.random.default_rng(13)
        for d in range(8):  # graphs and first-touch work outside the timed rounds
            one_round(d, rng)
        per_d, draft_tok = {}, []
        for d in range(8):
            rng = np.random.default_rng(17 + d)
            ts, toks = [], 0
            for _ in range(FULL_ROUND_REPS):
                t, td, a = one_round(d, rng)
                ts.append(t)
                toks += a + 1
                if d:
                    draft_tok.append(td / d)
            # drafts agree independently with probability p per position:
            # E(d) = (1 - p^(d+1)) / (1 - p) tokens a round, noise-free
            p = wl["p_agree"]
            e_tok = (1.0 - p ** (d + 1)) / (1.0 - p)
            t_med = statistics.median(ts)
            per_d[str(d)] = {"round_us": round(t_med * 1e6, 1),
                             "tok_per_s": round(toks / sum(ts), 1),
                             "expected_tok_per_s": round(e_tok / t_med, 1)}
        best = max(per_d, key=lambda k: per_d[k]["expected_tok_per_s"])
        leg = {"draft_us_per_token": round(statistics.median(draft_tok) * 1e6, 1),
               "by_depth": per_d, "best_static_d": int(best),
               "best_over_plain_decode": round(per_d[best]["expected_tok_per_s"] /
                                               per_d["0"]["expected_tok_per_s"], 3)}
        rng = np.random.default_rng(11)
        ctl = sv.DepthController(d_min=0, d_max=7)
        toks, secs, hist = 0, 0.0, {}
        for _ in range(rounds):
            d = ctl.next_depth()
            t, _, a = one_round(d, rng)
            toks += a + 1
            secs += t
            hist[str(d)] = hist.get(str(d), 0) + 1
            ctl.observe(d, [a], t)
        ctl.close()
        leg["adaptive"] = {"tok_per_s": round(toks / secs, 1), "depths": hist, "rounds": rounds}
        out[f"draft{n_layers}L"] = leg
        assert sv.spec_error_check(dm) == 0
        dm.close()
    return out


def nt_sweep(sv, synth, dev, reps=20, wl=None):
    """The linear-layer sweep: Q4 5120x13824 and Q6 13824x5120 (or the
    given workload's matrices) at each nt, L2 flushed between launches
    (verify-GEMM microseconds and GB/s)."""
    import torch
    wl = synth.WL_LINEAR_SWEEP if wl is None else wl
    gen = synth.torch_gen(wl["seed"], dev)
    st = torch.cuda.current_stream()
    flush = L2Flush(dev)
    out = {}
    for qt, N, K in wl["mats"]:
        w = synth.q_weight_torch(gen, qt, N, K, dev)
        qm = sv.QMat(w, max_rows=16)
        x = synth.f16_normal_torch(gen, (16, K), dev).view(torch.int16)
        y = torch.empty((16, N), dtype=torch.float32, device=dev)
        wbytes = N * K * WEIGHT_BYTES[qt]
        row = {}
        for nt in wl["nts"]:
            times = []
            for i in range(reps + 3):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                sv.spec_linear_q(qm, x, nt, y, st)
                e1.record(st)
                e1.synchronize()
                if i >= 3:
                    times.append(e0.elapsed_time(e1) * 1e-3)
            t = statistics.median(times)
            row[str(nt)] = {"us": round(t * 1e6, 2), "gbs": round(wbytes / t / 1e9, 1)}
        out[f"q{qt}_{N}x{K}"] = row
        qm.close()
    return out


def run_ours(args):
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    from speculative_decoding_verification_round_gb300 import synth
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(ws, "nccl")
    wl = dict(synth.WL_DECODER8)
    d, V = wl["d"], wl["vocab"]
    max_ctx = wl["ctx"] + max(8 * (args.warmup + args.steps + 4),
                              sv.SPEC_MAX_NT * ROUND_SWEEP_GROUP, sv.SPEC_MAX_NT * (ADAPTIVE_ROUNDS + 2)) + 64
    hbm_peak, peak_kind = peaks()
    m, W = build_model(sv, synth, wl, dev, max_ctx)
    del W
    torch.cuda.empty_cache()
    fill_context(sv, synth, m, wl, dev, seed=1 + rank)
    rng = np.random.default_rng(wl["seed"] + rank)
    anchor = 1234
    n_rounds = args.warmup + args.steps
    drafts = record_chain(sv, synth, m, wl, dev, n_rounds, anchor, rng)
    sid = torch.zeros(1, dtype=torch.int32, device=dev)
    dr_dev = [torch.tensor([c], dtype=torch.int32, device=dev) for c in drafts]
    n_acc = torch.zeros((n_rounds, 1), dtype=torch.int32, device=dev)
    em = torch.zeros((n_rounds, 1, d + 1), dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream()
    # replay: warm-up rounds, then exactly K timed rounds
    sv.spec_state_set(m, [0], n_past=[wl["ctx"]], emit_idx=[0], anchor=[anchor])
    for j in range(args.warmup):
        sv.spec_verify_round(m, 1, sid, dr_dev[j], d, n_acc=n_acc[j], emitted=em[j])
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local, args.clocks_csv) as clk:
        torch.cuda.nvtx.range_push("timed")
        e0.record(st)
        for j in range(args.warmup, n_rounds):
            sv.spec_verify_round(m, 1, sid, dr_dev[j], d, n_acc=n_acc[j], emitted=em[j])
        e1.record(st)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    barrier(dist)
    torch.cuda.synchronize()
    assert sv.spec_error_check(m) == 0
    elapsed = e0.elapsed_time(e1) * 1e-3
    emitted_tokens = int((n_acc[args.warmup:].cpu().numpy() + 1).sum())
    t_max = max_over_ranks(dist, elapsed, dev)
    tokens_all = sum_over_ranks(dist, emitted_tokens, dev)
    ms_per_step = t_max / args.steps * 1e3

    # end to end through host buffers: spec_verify_round_host takes the
    # drafts from host memory (copied into the model's mapped pinned staging,
    # which the round's kernels read and write in place: one graph launch)
    # and returns (n_acc, emitted) in host memory, every step
    sv.spec_state_set(m, [0], n_past=[wl["ctx"]], emit_idx=[0], anchor=[anchor])
    h_drafts = [np.array([c], dtype=np.int32) for c in drafts]
    h_sid = np.zeros(1, dtype=np.int32)
    h_acc = np.empty(1, dtype=np.int32)
    h_em = np.empty((1, d + 1), dtype=np.int32)
    e2e_tok = 0
    for j in range(args.warmup):
        sv.spec_verify_round_host(m, 1, h_sid, h_drafts[j], d, n_acc=h_acc, emitted=h_em)
    torch.cuda.synchronize()
    barrier(dist)
    t0 = time.perf_counter()
    for j in range(args.warmup, n_rounds):
        sv.spec_verify_round_host(m, 1, h_sid, h_drafts[j], d, n_acc=h_acc, emitted=h_em)
        e2e_tok += int(h_acc[0]) + 1
    t_e2e = max_over_ranks(dist, time.perf_counter() - t0, dev)
    e2e_all = sum_over_ranks(dist, e2e_tok, dev)

    line = None
    if rank == 0:
        gbs, per, bytes_per_launch, traffic = time_dominant_kernel(sv, synth, wl, dev, hbm_peak)
        sweep = nt_sweep(sv, synth, dev) if not args.no_sweep else None
        sweep_q8 = nt_sweep(sv, synth, dev, wl=synth.WL_LINEAR_SWEEP_Q8) if not args.no_sweep else None
        rsweep = round_sweep(sv, m, wl, dev) if not args.no_sweep else None
        adaptive = adaptive_depth_run(sv, m, wl, dev) if not args.no_sweep else None
        full_round = full_round_run(sv, synth, m, wl, dev, max_ctx) if not args.no_sweep else None
        n_layers = wl["n_layers"]
        # embed (with the first norm), 8 per layer but the first layer's
        # norm, final norm + LM head, fused accept + commit
        launches_per_round = 1 + 8 * n_layers - 1 + 2 + 1
        weight_bytes = sum(p["N"] * p["K"] * WEIGHT_BYTES[p["qtype"]] *
                           (n_layers if p["qtype"] == 4 else 1) for p in per)
        kv_bytes = n_layers * wl["n_kv_heads"] * (wl["ctx"] + d) * wl["head_dim"] * 2 * 2
        round_s = ms_per_step * 1e-3
        line = {
            "metric": METRIC,
            "value": round(tokens_all / t_max, 2),
            "unit": "tok/s",
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f16",
            "precision": "Q4/Q6 block ints exact in f16, f16 activations, f32 accumulate",
            "data": "synthetic (seeded N(0,1) activations and KV, uniform block ints, random-init weights)",
            "config": {"workload": wl["name"], "n_layers": n_layers, "hidden": wl["hidden"],
                       "heads": f"{wl['n_q_heads']}/{wl['n_kv_heads']}x{wl['head_dim']}",
                       "ffn": wl["ffn"], "vocab": V, "context": wl["ctx"], "nt": d + 1,
                       "n_seq": wl["n_seq"], "p_agree": wl["p_agree"], "graphs": True,
                       "l2": "inputs larger than L2 (1.49 GB of weights per round)",
                       "parallelism": f"replicas x{ws}"},
            "verify_round_us": round(round_s * 1e6, 2),
            "emitted_tokens_per_round": round(tokens_all / ws / args.steps, 3),
            "round_bytes": {"weights": weight_bytes, "kv": kv_bytes,
                            "gbs": round((weight_bytes + kv_bytes) / round_s / 1e9, 1),
                            "frac_of_hbm": round((weight_bytes + kv_bytes) / round_s / 1e9 / hbm_peak, 4)},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "traffic": None if traffic is None else round(traffic),
                         "kernel": "linear_q_kernel (verify GEMM), nt=8, one round's launch mix",
                         "algorithmic_bytes_per_launch": round(bytes_per_launch),
                         "peak_kind": peak_kind, "per_shape": per},
            "sweep": sweep,
            "sweep_q8": sweep_q8,
            "round_sweep": rsweep,
            "adaptive_depth": adaptive,
            "full_round": full_round,
            "e2e": {"value": round(e2e_all / t_e2e, 2), "unit": "tok/s",
                    "api": "spec_verify_round_host (host arrays, mapped pinned staging)",
                    "h2d_bytes_per_step": 4 * (1 + d), "d2h_bytes_per_step": 4 * (2 + d)},
            "gpu_launches": launches_per_round * args.steps,
            "clocks": clk.summary(),
        }
        if ws == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(W=None, wl=wl, drafts=drafts[:1], anchor=anchor,
                                                m=m, sv=sv, dev=dev)
    m.close()
    if line is not None:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


# --------------------------------------------------------------------------
# the CPU oracle on the same workload
# --------------------------------------------------------------------------
def oracle_model_host(wl, dev_or_cpu="cpu"):
    """The decoder's canonical weights on the host, generated by the same
    seeded generator (on the GPU when there is one)."""
    import torch
    import oracle
    from speculative_decoding_verification_round_gb300 import synth
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    W = synth.decoder_weights_torch(wl, gen_dev)
    def hw(w):
        return oracle.QWeight(w["qtype"], w["qs"].cpu().numpy(),
                              None if w["qh"] is None else w["qh"].cpu().numpy(),
                              w["scales"].cpu().view(torch.int16).numpy().view(np.uint16),
                              w["N"], w["K"])
    om = oracle.Model(wl["n_layers"], wl["hidden"], wl["n_q_heads"], wl["n_kv_heads"],
                      wl["head_dim"], wl["ffn"], wl["vocab"], wl["ctx"] + 64,
                      W["embed"].cpu().view(torch.int16).numpy().view(np.uint16),
                      W["norm_w"].cpu().numpy(), [hw(w) for w in W["wqkv"]],
                      [hw(w) for w in W["wo"]], [hw(w) for w in W["wgu"]],
                      [hw(w) for w in W["wd"]], hw(W["lm_head"]))
    del W
    return om


def oracle_context(wl, seed=1):
    import torch
    from speculative_decoding_verification_round_gb300 import synth
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    gen = synth.torch_gen(seed, gen_dev)
    L, nkv, hd, ctx = wl["n_layers"], wl["n_kv_heads"], wl["head_dim"], wl["ctx"]
    kc = np.zeros((L, 1, nkv, ctx + 64, hd), np.uint16)
    vc = np.zeros_like(kc)
    for l in range(L):
        k = synth.f16_normal_torch(gen, (nkv, ctx, hd), gen_dev)
        v = synth.f16_normal_torch(gen, (nkv, ctx, hd), gen_dev)
        kc[l, 0, :, :ctx] = k.cpu().view(torch.int16).numpy().view(np.uint16)
        vc[l, 0, :, :ctx] = v.cpu().view(torch.int16).numpy().view(np.uint16)
    return kc, vc


def oracle_round(orc, om, kc, vc, wl, anchor, draft):
    tokens = np.array([[anchor] + list(draft)], np.int32)
    logits = om.forward(tokens, [wl["ctx"]], kc, vc)
    am = np.array([[orc.argmax(r) for r in logits]], np.int32)
    n_acc, em = orc.accept_greedy(am, np.array([draft], np.int32))
    return int(n_acc[0]) + 1


def cpu_baseline(W, wl, drafts, anchor, m=None, sv=None, dev=None):
    import oracle
    oracle.build()
    om = oracle_model_host(wl)
    kc, vc = oracle_context(wl)
    t0 = time.perf_counter()
    toks = oracle_round(oracle, om, kc, vc, wl, anchor, drafts[0])
    t = time.perf_counter() - t0
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {"value": round(toks / t, 4), "unit": "tok/s", "cores": cores, "kind": "oracle",
            "sample": f"one full verify round of {wl['name']} (nt={wl['d'] + 1}, all "
                      f"{wl['n_layers']} layers + LM head, fp64), {t:.1f} s"}


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    from speculative_decoding_verification_round_gb300 import synth
    oracle.build()
    wl = dict(synth.WL_DECODER8)
    om = oracle_model_host(wl)
    kc0, vc0 = oracle_context(wl)
    rng = np.random.default_rng(wl["seed"])
    anchor = 1234
    draft = [int(x) for x in rng.integers(0, wl["vocab"], wl["d"])]
    for _ in range(args.warmup):
        oracle_round(oracle, om, kc0.copy(), vc0.copy(), wl, anchor, draft)
    t0 = time.perf_counter()
    toks = 0
    for _ in range(args.steps):
        toks += oracle_round(oracle, om, kc0.copy(), vc0.copy(), wl, anchor, draft)
    t = time.perf_counter() - t0
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    val = toks / t
    sample = (f"{args.steps} full verify rounds of {wl['name']} on the CPU oracle "
              f"(fp64, all layers + LM head)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "tok/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl["name"], "nt": wl["d"] + 1},
        "cpu_baseline": {"value": round(val, 4), "unit": "tok/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(val, 4), "unit": "tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


def linear_only(spec: str, nt: int = 8, reps: int = 3):
    """Profiling driver: spec_linear_q at nt on packed synthetic matrices,
    `spec` = 'QT:N:K,QT:N:K,...', each launched `reps` times."""
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    from speculative_decoding_verification_round_gb300 import synth
    dev = torch.device("cuda:0")
    gen = synth.torch_gen(3, dev)
    for item in spec.split(","):
        qt, N, K = (int(v) for v in item.split(":"))
        w = synth.q_weight_torch(gen, qt, N, K, dev)
        qm = sv.QMat(w, max_rows=16)
        x = synth.f16_normal_torch(gen, (nt, K), dev).view(torch.int16)
        y = torch.empty((nt, N), dtype=torch.float32, device=dev)
        for _ in range(reps):
            sv.spec_linear_q(qm, x, nt, y)
        torch.cuda.synchronize()
        qm.close()
        del w
    print("linear-only ok")


def draft_only(n_layers: int, warm: int = 3, reps: int = 3):
    """Profiling driver: nt = 1 forwards (graph-replayed d = 0 rounds) of the
    0.5B-class draft at `n_layers` layers and a 4096-position context; the
    last `reps` run inside the NVTX range "draft"."""
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    from speculative_decoding_verification_round_gb300 import synth
    dev = torch.device("cuda:0")
    wl = dict(synth.WL_DRAFT05B, n_layers=n_layers)
    dm, W = build_model(sv, synth, wl, dev, wl["ctx"] + 64)
    del W
    fill_context(sv, synth, dm, wl, dev, seed=7)
    sid = torch.zeros(1, dtype=torch.int32, device=dev)
    n_acc = torch.zeros(1, dtype=torch.int32, device=dev)
    em = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    sv.spec_state_set(dm, [0], n_past=[wl["ctx"]], emit_idx=[0], anchor=[1234])
    for _ in range(warm):
        sv.spec_verify_round(dm, 1, sid, None, 0, n_acc=n_acc, emitted=em)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("draft")
    for _ in range(reps):
        sv.spec_verify_round(dm, 1, sid, None, 0, n_acc=n_acc, emitted=em)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    assert sv.spec_error_check(dm) == 0
    dm.close()
    print("draft-only ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--linear-only", default=None,
                    help="profiling driver: QT:N:K[,QT:N:K...] verify-GEMM launches only")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the raw nvidia-smi clock samples in this file")
    ap.add_argument("--draft-only", type=int, default=None, metavar="LAYERS",
                    help="profiling driver: nt = 1 forwards of the 0.5B-class draft")
    args = ap.parse_args()
    if args.linear_only:
        linear_only(args.linear_only)
        return
    if args.draft_only:
        draft_only(args.draft_only)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        # each oracle step is a full fp64 round (seconds of CPU work): bound
        # the run to a few minutes
        args.steps = min(args.steps, 5)
        args.warmup = min(args.warmup, 3)
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
