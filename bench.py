"""Benchmark of the verify round on one GB300 (or N replicas).

Step = one verify round of the batched 14B-shaped workload: a 40-layer
decoder (H 5120, 40 query / 8 KV heads of 128, SwiGLU FFN 13824, Q4 linears,
Q6 LM head over V = 248320), 12 sequences with 512 cached positions each,
nt = 16 rows per sequence (anchor + 15 drafts: 192 rows in one weights-once
target pass), strict rejection sampling at T = 0.7.  The draft logits come
from a noisy-target drafter: the target's own nt = 1 logits along the draft
chain plus N(0, 0.5) noise, each draft sampled from them.  The drafter runs
untimed while the rounds are recorded; the timed steps replay the recorded
rounds from the same starting state, and every step recomputes the whole
target pass, the accept and the commit.

Printed JSON line: value = emitted tokens per second over the 12 sequences
(accepted drafts + one correction or bonus token per sequence and round);
the verify-round latency with graphs and with raw launches; the verify GEMM
measured inside the round (CUDA events around each launch) against the
tensor and HBM rooflines; the end-to-end rate through host buffers; the
oracle's CPU rate; and compact legs for the other workloads (LM-head greedy
round, standalone stochastic accept, linear sweep, 8-layer greedy decoder).

--impl reference times the CPU oracle (the plain fp64 reference) on the
same workload: each step is a bounded sample (one sequence, a 2-layer slice
of the 40 layers plus the LM head), scaled to the full round.
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
    """(HBM GB/s, sustained bf16 TFLOP/s, burst bf16 TFLOP/s, kind)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops_sustained"]), float(p["bf16_tflops"]),
                "measured")
    except Exception:
        return 6800.0, 1700.0, 1900.0, "fallback"


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
def smi_id(local: int) -> str:
    """The id nvidia-smi knows this process's CUDA device by: its PCI bus id
    (CUDA_VISIBLE_DEVICES may renumber devices, nvidia-smi does not), else
    its UUID, else the CUDA index."""
    import torch
    p = torch.cuda.get_device_properties(local)
    try:
        return f"{int(p.pci_domain_id):08X}:{int(p.pci_bus_id):02X}:{int(p.pci_device_id):02X}.0"
    except Exception:
        pass
    try:
        u = str(p.uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(local)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu, path=None):
        """gpu: what nvidia-smi --id takes (a PCI bus id, a UUID or an index)."""
        import tempfile
        self.gpu = gpu
        self.proc = None
        self.start_line = 0
        tag = "".join(ch if ch.isalnum() else "_" for ch in str(gpu))
        self.path = path or os.path.join(tempfile.gettempdir(),
                                         f"spec_verify_clocks_{tag}.csv")

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
    """The workload's decoder with random-init weights (generated on the
    device, repacked by the library; the canonical planes are dropped)."""
    import torch
    W = synth.decoder_weights_torch(wl, dev)
    desc = dict(n_layers=wl["n_layers"], hidden=wl["hidden"], n_q_heads=wl["n_q_heads"],
                n_kv_heads=wl["n_kv_heads"], head_dim=wl["head_dim"], ffn=wl["ffn"],
                vocab=wl["vocab"], max_ctx=max_ctx, max_nt=sv.SPEC_MAX_NT, max_seqs=wl["n_seq"])
    m = sv.Model(desc, W)
    del W
    torch.cuda.empty_cache()
    return m


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


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "tc_linear_traffic_decoder14b_r192.json")
GEMM_SRC = os.path.join(ROOT, "speculative_decoding_verification_round_gb300", "csrc", "tcgemm.cu")


def measured_traffic(shapes):
    """DRAM bytes per verify-GEMM launch over a launch mix, from the committed
    ncu record (profiles/, command inside) -- or None when the record is
    missing, lacks a shape, or was taken on a different kernel source (the
    record's source_sha256 against GEMM_SRC).  shapes: (qtype, N, K,
    launches[, rows]); a record key is "QT:N:K" or "QT:N:K:R"."""
    import hashlib
    try:
        rec = json.load(open(TRAFFIC_RECORD))
        sha = hashlib.sha256(open(GEMM_SRC, "rb").read()).hexdigest()
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256") != sha:
        return None
    total, n = 0.0, 0
    for sh in shapes:
        qt, N, K, count = sh[:4]
        key = f"{qt}:{N}:{K}" + (f":{sh[4]}" if len(sh) > 4 else "")
        b = rec.get("dram_bytes_per_launch", {}).get(key)
        if b is None:
            return None
        total += b * count
        n += count
    return total / n


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
        dm = build_model(sv, synth, dwl, dev, max_ctx)
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


# --------------------------------------------------------------------------
# the batched stochastic workload (the step)
# --------------------------------------------------------------------------
def state0_of(wl):
    n = wl["n_seq"]
    return (list(range(n)), [wl["ctx"]] * n, [1000 * s for s in range(n)],
            [(7919 * s + 1234) % wl["vocab"] for s in range(n)])


def set_state(sv, m, st):
    slots, n_past, ei, anc = st
    sv.spec_state_set(m, slots, n_past=n_past, emit_idx=ei, anchor=anc)


def record_stochastic(sv, synth, m, wl, dev, n_rounds, seed):
    """Untimed: the speculative chain of all sequences, with the noisy-target
    drafter.  Draft step i of a round: an nt = 1 target pass at the draft
    position (a greedy d = 0 round with logits, state restored afterwards),
    draft logits = those logits + N(0, q_noise), the draft sampled from
    softmax(draft logits / T) (Gumbel-max on the device).  Then the round
    itself (it commits).  Returns [(drafts [n_seq][d], q [n_seq][d][V])]."""
    import torch
    n_seq, d, V, T = wl["n_seq"], wl["d"], wl["vocab"], wl["temperature"]
    slots = list(range(n_seq))
    sid = torch.arange(n_seq, dtype=torch.int32, device=dev)
    gen = synth.torch_gen(seed, dev)
    lg1 = torch.empty((n_seq, V), dtype=torch.float32, device=dev)
    na1 = torch.empty(n_seq, dtype=torch.int32, device=dev)
    em1 = torch.empty((n_seq, 1), dtype=torch.int32, device=dev)
    n_acc = torch.empty(n_seq, dtype=torch.int32, device=dev)
    em = torch.empty((n_seq, d + 1), dtype=torch.int32, device=dev)
    rounds = []
    for _ in range(n_rounds):
        n_past, ei, anc = sv.spec_state_get(m, slots)
        tok = list(anc)
        qs = torch.empty((n_seq, d, V), dtype=torch.float32, device=dev)
        dr = torch.empty((n_seq, d), dtype=torch.int32, device=dev)
        for i in range(d):
            sv.spec_state_set(m, slots, n_past=[p + i for p in n_past], anchor=tok)
            sv.spec_verify_round(m, n_seq, sid, None, 0, n_acc=na1, emitted=em1, logits_out=lg1)
            q_i = qs[:, i]
            q_i.copy_(lg1)
            q_i.add_(torch.randn((n_seq, V), generator=gen, device=dev), alpha=wl["q_noise"])
            u = torch.rand((n_seq, V), generator=gen, device=dev)
            x = torch.argmax(q_i / T - torch.log(-torch.log(u)), dim=1).to(torch.int32)
            dr[:, i] = x
            tok = x.tolist()
        sv.spec_state_set(m, slots, n_past=n_past, emit_idx=ei, anchor=anc)
        sv.spec_verify_round(m, n_seq, sid, dr, d, qs, False, T, seed, n_acc, em)
        rounds.append((dr, qs))
    assert sv.spec_error_check(m) == 0
    return rounds


def replay(sv, m, wl, dev, rounds, st0, warmup, steps, seed, clk=None):
    """Warm-up rounds, then exactly `steps` rounds between two CUDA events
    (device time); returns (seconds, n_acc [steps][n_seq] on the host)."""
    import torch
    n_seq, d, T = wl["n_seq"], wl["d"], wl["temperature"]
    sid = torch.arange(n_seq, dtype=torch.int32, device=dev)
    n_acc = torch.zeros((warmup + steps, n_seq), dtype=torch.int32, device=dev)
    em = torch.zeros((warmup + steps, n_seq, d + 1), dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream()
    set_state(sv, m, st0)
    for j in range(warmup):
        dr, qs = rounds[j]
        sv.spec_verify_round(m, n_seq, sid, dr, d, qs, False, T, seed, n_acc[j], em[j])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clk is not None:
        clk.__enter__()
    try:
        if clk is not None:  # the headline's timed steps: NVTX range "timed" for launch lists
            torch.cuda.nvtx.range_push("timed")
        e0.record(st)
        for j in range(warmup, warmup + steps):
            dr, qs = rounds[j]
            sv.spec_verify_round(m, n_seq, sid, dr, d, qs, False, T, seed, n_acc[j], em[j])
        e1.record(st)
        torch.cuda.synchronize()
        if clk is not None:
            torch.cuda.nvtx.range_pop()
    finally:
        if clk is not None:
            clk.__exit__(None, None, None)
    assert sv.spec_error_check(m) == 0
    return e0.elapsed_time(e1) * 1e-3, n_acc[warmup:].cpu().numpy()


def in_round_kernels(sv, m, wl, dev, rounds, st0, warmup, steps, seed):
    """The round's kernels timed inside real rounds (spec_model_profile: raw
    launches, a CUDA event before and after each GEMM / attention launch),
    per kernel class: us per launch, achieved TFLOP/s and GB/s."""
    set_state(sv, m, st0)
    m.profile(True)
    import torch
    n_seq, d, T = wl["n_seq"], wl["d"], wl["temperature"]
    sid = torch.arange(n_seq, dtype=torch.int32, device=dev)
    n_acc = torch.zeros(n_seq, dtype=torch.int32, device=dev)
    em = torch.zeros((n_seq, d + 1), dtype=torch.int32, device=dev)
    for j in range(warmup + steps):
        if j == warmup:
            m.profile(True)  # totals of the timed rounds only
        dr, qs = rounds[j]
        sv.spec_verify_round(m, n_seq, sid, dr, d, qs, False, T, seed, n_acc, em)
    names = {"qkv": sv.SPEC_PROF_QKV, "o": sv.SPEC_PROF_O, "gate_up": sv.SPEC_PROF_GATE_UP,
             "down": sv.SPEC_PROF_DOWN, "lm_head": sv.SPEC_PROF_LM_HEAD,
             "all_gemms": sv.SPEC_PROF_ALL_GEMMS, "attention": sv.SPEC_PROF_ATTN}
    out = {}
    for k, kind in names.items():
        r = m.profile_read(kind)
        n = max(r["launches"], 1)
        out[k] = dict(launches=r["launches"], seconds=r["seconds"],
                      us_per_launch=r["seconds"] / n * 1e6,
                      tflops=r["flops"] / r["seconds"] / 1e12 if r["seconds"] else 0.0,
                      gbs=r["bytes"] / r["seconds"] / 1e9 if r["seconds"] else 0.0,
                      bytes_per_launch=r["bytes"] / n, flops_per_launch=r["flops"] / n)
    m.profile(False)
    assert sv.spec_error_check(m) == 0
    return out


def e2e_host(sv, m, wl, dev, rounds, st0, warmup, steps, seed):
    """The same rounds through spec_verify_round_host: sequence ids and drafts
    from host memory, the draft logits from pinned host memory (copied to the
    device inside the call), n_acc and emitted back in host memory, every
    step.  Returns (tokens, wall seconds, h2d bytes, d2h bytes per step)."""
    import torch
    n_seq, d, V, T = wl["n_seq"], wl["d"], wl["vocab"], wl["temperature"]
    h_sid = np.arange(n_seq, dtype=np.int32)
    h_dr = [dr.cpu().numpy() for dr, _ in rounds[:warmup + steps]]
    h_q = []
    for _, qs in rounds[:warmup + steps]:
        t = torch.empty(qs.shape, dtype=torch.float32, pin_memory=True)
        t.copy_(qs)
        h_q.append(t)
    h_acc = np.empty(n_seq, np.int32)
    h_em = np.empty((n_seq, d + 1), np.int32)
    set_state(sv, m, st0)
    for j in range(warmup):
        sv.spec_verify_round_host(m, n_seq, h_sid, h_dr[j], d, h_q[j], False, T, seed,
                                  n_acc=h_acc, emitted=h_em)
    torch.cuda.synchronize()
    toks = 0
    t0 = time.perf_counter()
    for j in range(warmup, warmup + steps):
        sv.spec_verify_round_host(m, n_seq, h_sid, h_dr[j], d, h_q[j], False, T, seed,
                                  n_acc=h_acc, emitted=h_em)
        toks += int((h_acc + 1).sum())
    t = time.perf_counter() - t0
    assert sv.spec_error_check(m) == 0
    h2d = 4 * n_seq + 4 * n_seq * d + 4 * n_seq * d * V
    d2h = 4 * n_seq + 4 * n_seq * (d + 1)
    return toks, t, h2d, d2h


# --------------------------------------------------------------------------
# the other workloads (compact legs)
# --------------------------------------------------------------------------
def lmhead_leg(sv, synth, dev, hbm_peak, reps=50):
    """H 1024, V 32000, d 2: the LM head (Q4, fused argmax, no logits) and the
    greedy accept of drafts that agree with the target argmax w.p. 0.74; L2
    flushed between rounds (18 MB of weights fit in L2)."""
    import torch
    wl = synth.WL_LMHEAD_GREEDY
    H, V, d = wl["hidden"], wl["vocab"], wl["d"]
    g = np.random.default_rng(wl["seed"])
    w = synth.q_weight(g, 4, V, H)
    x = synth.f16_normal(g, (d + 1, H))
    dw = dict(qtype=4, N=V, K=H, qs=torch.from_numpy(w["qs"]).to(dev), qh=None,
              scales=torch.from_numpy(w["scales"].view(np.int16)).to(dev))
    m = sv.Model(dict(n_layers=0, hidden=H, vocab=V, max_nt=d + 1, max_seqs=1),
                 dict(lm_head=dw, norm_w=torch.ones((1, H), dtype=torch.float32, device=dev)))
    xd = torch.from_numpy(x.view(np.int16)).to(dev)
    am = torch.empty(d + 1, dtype=torch.int32, device=dev)
    sv.spec_lm_head(m, xd, d + 1, None, am)
    dr_h = synth.greedy_drafts(g, am.cpu().numpy()[:d], V, wl["p_agree"])[None, :]
    dr = torch.from_numpy(dr_h).to(dev)
    n_acc = torch.empty(1, dtype=torch.int32, device=dev)
    em = torch.empty((1, d + 1), dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    st = torch.cuda.current_stream()
    times = []
    for i in range(reps + 3):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        sv.spec_lm_head(m, xd, d + 1, None, am)
        sv.spec_accept_greedy(am.view(1, d + 1), dr, 1, d, n_acc, em)
        e1.record(st)
        e1.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1) * 1e-3)
    assert sv.spec_error_check(m) == 0
    t = statistics.median(times)
    nbytes = V * H * WEIGHT_BYTES[4] + (d + 1) * H * 2
    m.close()
    leg = {"us": round(t * 1e6, 2), "gbs": round(nbytes / t / 1e9, 1),
           "frac_hbm": round(nbytes / t / 1e9 / hbm_peak, 3), "n_acc": int(n_acc.item()),
           "l2": "flushed"}
    return leg, dict(w=w, x=x, draft=dr_h)


def accept_leg(sv, synth, dev, hbm_peak, reps=20):
    """12 sequences, d 7, V 248320: the standalone strict rejection sampler
    on p-logits N(0, 2) and draft logits p + N(0, 0.5), T 1, drafts sampled
    from the draft logits; L2 flushed between calls."""
    import torch
    wl = synth.WL_ACCEPT_STOCH
    n_seq, d, V, T = wl["n_seq"], wl["d"], wl["vocab"], wl["temperature"]
    g = np.random.default_rng(wl["seed"])
    p, q = synth.stochastic_logits(g, n_seq, d, V, wl["p_std"], wl["q_noise"])
    pd, qd = torch.from_numpy(p).to(dev), torch.from_numpy(q).to(dev)
    gen = synth.torch_gen(wl["seed"], dev)
    u = torch.rand(qd.shape, generator=gen, device=dev)
    dr = torch.argmax(qd / T - torch.log(-torch.log(u)), dim=2).to(torch.int32)
    sid_h = (np.arange(n_seq) * 3 + 1).astype(np.int32)
    sid = torch.from_numpy(sid_h).to(dev)
    ei0 = torch.arange(n_seq, dtype=torch.int64, device=dev) * 1000
    ei = ei0.clone()
    n_acc = torch.empty(n_seq, dtype=torch.int32, device=dev)
    em = torch.empty((n_seq, d + 1), dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    st = torch.cuda.current_stream()
    times = []
    for i in range(reps + 3):
        flush()
        ei.copy_(ei0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        sv.spec_accept_stochastic(pd, qd, dr, n_seq, d, V, T, 0x5EED, sid, ei, n_acc, em)
        e1.record(st)
        e1.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1) * 1e-3)
    assert sv.spec_error_check(None) == 0
    t = statistics.median(times)
    dense = 4.0 * V * n_seq * (2 * d + 1)
    leg = {"us": round(t * 1e6, 2), "gbs_dense": round(dense / t / 1e9, 1),
           "frac_hbm": round(dense / t / 1e9 / hbm_peak, 3),
           "mean_accepted": round(float(n_acc.float().mean().item()), 3), "l2": "flushed"}
    return leg, dict(p=p, q=q, draft=dr.cpu().numpy(), seq_ids=sid_h,
                     emit_idx=(np.arange(n_seq) * 1000).astype(np.uint64), T=T)


def decoder8_leg(sv, synth, dev, args, hbm_peak):
    """The 8-layer H 4096 decoder, greedy, nt 8, 4096 cached positions, drafts
    on the target's greedy chain w.p. 0.74: rounds graph-replayed and
    raw-launched, and the round time at each nt."""
    import torch
    wl = dict(synth.WL_DECODER8)
    d = wl["d"]
    rounds = 20
    max_ctx = wl["ctx"] + max(8 * (rounds + 4), sv.SPEC_MAX_NT * ROUND_SWEEP_GROUP,
                              sv.SPEC_MAX_NT * (ADAPTIVE_ROUNDS + 2)) + 64
    m = build_model(sv, synth, wl, dev, max_ctx)
    fill_context(sv, synth, m, wl, dev, seed=1)
    rng = np.random.default_rng(wl["seed"])
    anchor = 1234
    drafts = record_chain(sv, synth, m, wl, dev, rounds + 3, anchor, rng)
    sid = torch.zeros(1, dtype=torch.int32, device=dev)
    dr_dev = [torch.tensor([c], dtype=torch.int32, device=dev) for c in drafts]
    n_acc = torch.zeros((rounds + 3, 1), dtype=torch.int32, device=dev)
    em = torch.zeros((rounds + 3, 1, d + 1), dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream()
    leg = {}
    for graphs in (True, False):
        m.set_graphs(graphs)
        sv.spec_state_set(m, [0], n_past=[wl["ctx"]], emit_idx=[0], anchor=[anchor])
        for j in range(3):
            sv.spec_verify_round(m, 1, sid, dr_dev[j], d, n_acc=n_acc[j], emitted=em[j])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for j in range(3, rounds + 3):
            sv.spec_verify_round(m, 1, sid, dr_dev[j], d, n_acc=n_acc[j], emitted=em[j])
        e1.record(st)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) * 1e-3 / rounds
        toks = int((n_acc[3:].cpu().numpy() + 1).sum())
        key = "graph" if graphs else "raw"
        leg[f"round_us_{key}"] = round(t * 1e6, 2)
        leg[f"tok_s_{key}"] = round(toks / (t * rounds), 1)
    m.set_graphs(True)
    assert sv.spec_error_check(m) == 0
    wbytes = (wl["n_layers"] * ((wl["n_q_heads"] + 2 * wl["n_kv_heads"]) * wl["head_dim"] * wl["hidden"]
                                + wl["hidden"] * wl["n_q_heads"] * wl["head_dim"]
                                + 3 * wl["ffn"] * wl["hidden"]) * WEIGHT_BYTES[4]
              + wl["vocab"] * wl["hidden"] * WEIGHT_BYTES[6])
    kv = wl["n_layers"] * wl["n_kv_heads"] * (wl["ctx"] + d) * wl["head_dim"] * 4
    leg["round_frac_hbm"] = round((wbytes + kv) / (leg["round_us_graph"] * 1e-6) / 1e9 / hbm_peak, 3)
    if not args.no_legs:
        rs = round_sweep(sv, m, wl, dev)
        leg["round_sweep_us"] = rs["us"]
        leg["nt9_16_over_nt1"] = rs["nt9_16_over_nt1"]
    extras = {}
    if args.extras:
        extras["adaptive_depth"] = adaptive_depth_run(sv, m, wl, dev)
        extras["full_round"] = full_round_run(sv, synth, m, wl, dev, max_ctx)
    m.close()
    return leg, extras, drafts[3], anchor


def compact_sweep(sw):
    out = {}
    for name, row in sw.items():
        nts = sorted(row, key=int)
        out[name] = {"us": {k: row[k]["us"] for k in nts}, "gbs_nt8": row.get("8", {}).get("gbs"),
                     "nt16_over_nt1": round(row["16"]["us"] / row["1"]["us"], 3)}
    return out


# --------------------------------------------------------------------------
# the CPU oracle (cpu_baseline leg and the reference arm)
# --------------------------------------------------------------------------
def oracle_model_host(wl):
    """The decoder's canonical weights on the host, from the same seeded
    generator (run on the GPU when there is one)."""
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


SLICE_LAYERS = 2


class OracleSlice:
    """The oracle on a bounded sample of the batched workload: ONE sequence
    through a 2-layer slice of the 40 layers plus the LM head, nt 16, and the
    stochastic accept; drafts from the noisy-target drafter (the oracle's own
    nt = 1 passes + N(0, 0.5), sampled by the harness sampler), built once.
    A full round is estimated as n_seq x (n_layers / 2 x t(2 layers) +
    t(LM head) + t(accept))."""

    def __init__(self, wl, seed=99):
        import oracle
        oracle.build()
        self.o = oracle
        self.wl = wl
        sl = dict(wl, n_layers=SLICE_LAYERS)
        self.om = oracle_model_host(sl)
        self.kc, self.vc = oracle_context(sl, seed=2)
        d, V, T, ctx = wl["d"], wl["vocab"], wl["temperature"], wl["ctx"]
        g = np.random.default_rng(seed)
        self.anchor = int(g.integers(0, V))
        self.seed = seed
        kco, vco = self.kc.copy(), self.vc.copy()
        tok = self.anchor
        self.q = np.zeros((1, d, V), np.float32)
        self.draft = np.zeros((1, d), np.int32)
        for i in range(d):
            p_i = self.om.forward(np.array([[tok]], np.int32), [ctx + i], kco, vco)[0]
            self.q[0, i] = p_i + (g.standard_normal(V) * wl["q_noise"]).astype(np.float32)
            W, S = oracle.row_weights(self.q[0, i], T)
            U = oracle.uniforms(seed, i, 0, 1)
            tok = oracle.weight_pick(W, S, int(U[0]))
            self.draft[0, i] = tok
        # the LM head alone, to split the slice's time
        x = np.zeros((d + 1, wl["hidden"]), np.uint16)
        t0 = time.perf_counter()
        oracle.linear(self.om.lm_head, x)
        self.t_lm = time.perf_counter() - t0

    def step(self):
        """One sample: returns (emitted tokens of the sequence, seconds of the
        sample, estimated seconds of a full round)."""
        wl, o = self.wl, self.o
        d, T = wl["d"], wl["temperature"]
        tokens = np.concatenate([[[self.anchor]], self.draft], 1).astype(np.int32)
        t0 = time.perf_counter()
        lg = self.om.forward(tokens, [wl["ctx"]], self.kc.copy(), self.vc.copy())
        t1 = time.perf_counter()
        n_acc, _, _ = o.accept_stochastic(lg.reshape(1, d + 1, -1), self.q, self.draft, T,
                                          self.seed, [0], [0])
        t2 = time.perf_counter()
        t_layers = max(t1 - t0 - self.t_lm, 0.0)
        full = wl["n_seq"] * (wl["n_layers"] / SLICE_LAYERS * t_layers + self.t_lm + (t2 - t1))
        return int(n_acc[0]) + 1, t2 - t0, full


def cores_used():
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def cpu_baseline(wl5, tokens_per_round, legs_in):
    """The oracle as it stands, timed on the host cores: the headline as a
    scaled 2-layer slice, and each leg's own workload."""
    import oracle
    sl = OracleSlice(wl5)
    _, t_sample, t_round = sl.step()
    out = {"value": round(tokens_per_round / t_round, 4), "unit": "tok/s", "cores": cores_used(),
           "kind": "oracle",
           "sample": (f"one sequence of {wl5['name']}: a {SLICE_LAYERS}-layer slice + LM head, "
                      f"nt {wl5['d'] + 1}, fp64, + the stochastic accept ({t_sample:.1f} s); "
                      f"scaled to the full round ({wl5['n_seq']} sequences x "
                      f"{wl5['n_layers']} layers: {t_round:.1f} s); tokens per round "
                      f"{tokens_per_round:.2f} from the GPU rounds of the same workload")}
    per = {}
    if "lmhead" in legs_in:
        a = legs_in["lmhead"]
        qw = oracle.QWeight(4, a["w"]["qs"], None, a["w"]["scales"], a["w"]["N"], a["w"]["K"])
        t0 = time.perf_counter()
        lg = oracle.linear(qw, a["x"])
        am = np.array([[oracle.argmax(r) for r in lg]], np.int32)
        oracle.accept_greedy(am, a["draft"])
        per["lmhead_greedy_us"] = round((time.perf_counter() - t0) * 1e6, 1)
    if "accept" in legs_in:
        a = legs_in["accept"]
        t0 = time.perf_counter()
        oracle.accept_stochastic(a["p"], a["q"], a["draft"], a["T"], 0x5EED, a["seq_ids"],
                                 a["emit_idx"])
        per["accept_stochastic_us"] = round((time.perf_counter() - t0) * 1e6, 1)
    if "decoder8" in legs_in:
        a = legs_in["decoder8"]
        wl = a["wl"]
        om = oracle_model_host(wl)
        kc, vc = oracle_context(wl)
        tokens = np.array([[a["anchor"]] + list(a["draft"])], np.int32)
        t0 = time.perf_counter()
        lg = om.forward(tokens, [wl["ctx"]], kc, vc)
        am = np.array([[oracle.argmax(r) for r in lg]], np.int32)
        n_acc, _ = oracle.accept_greedy(am, np.array([a["draft"]], np.int32))
        per["decoder8_round_us"] = round((time.perf_counter() - t0) * 1e6, 1)
    out["per_workload"] = per
    return out


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    from speculative_decoding_verification_round_gb300 import synth
    wl = dict(synth.WL_DECODER14B)
    sl = OracleSlice(wl)
    for _ in range(args.warmup):
        sl.step()
    toks, t_samples, t_full = 0, 0.0, 0.0
    for _ in range(args.steps):
        tk, ts, tf = sl.step()
        toks += tk * wl["n_seq"]
        t_samples += ts
        t_full += tf
    val = toks / t_full
    sample = (f"{args.steps} samples, each one sequence through a {SLICE_LAYERS}-layer slice "
              f"of {wl['name']} + LM head + the stochastic accept on the CPU oracle (fp64); "
              f"{t_samples:.1f} s in all, scaled to full rounds of {wl['n_seq']} sequences x "
              f"{wl['n_layers']} layers; tokens per round = {wl['n_seq']} x the sample's "
              f"emitted count")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(val, 5), "unit": "tok/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_full / args.steps * 1e3, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl["name"], "n_seq": wl["n_seq"], "nt": wl["d"] + 1,
                   "temperature": wl["temperature"]},
        "cpu_baseline": {"value": round(val, 5), "unit": "tok/s", "cores": cores_used(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(val, 5), "unit": "tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------
def run_ours(args):
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    from speculative_decoding_verification_round_gb300 import synth
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(ws, "nccl")
    hbm_peak, tc_sustained, tc_burst, peak_kind = peaks()
    wl = dict(synth.WL_DECODER14B)
    n_seq, d, V, T = wl["n_seq"], wl["d"], wl["vocab"], wl["temperature"]
    seed = 0x5EED + rank
    n_rounds = args.warmup + args.steps
    max_ctx = wl["ctx"] + (d + 1) * (n_rounds + 2) + 64
    m = build_model(sv, synth, wl, dev, max_ctx)
    fill_context(sv, synth, m, wl, dev, seed=2 + rank)
    st0 = state0_of(wl)
    set_state(sv, m, st0)
    rounds = record_stochastic(sv, synth, m, wl, dev, n_rounds, seed)

    # the timed steps: graph-replayed rounds
    barrier(dist)
    torch.cuda.synchronize()
    clk = ClockSampler(smi_id(local), args.clocks_csv)
    elapsed, n_acc = replay(sv, m, wl, dev, rounds, st0, args.warmup, args.steps, seed, clk)
    barrier(dist)
    torch.cuda.synchronize()
    emitted = int((n_acc + 1).sum())
    t_max = max_over_ranks(dist, elapsed, dev)
    tokens_all = sum_over_ranks(dist, emitted, dev)
    ms_per_step = t_max / args.steps * 1e3

    # end to end through host buffers (every rank: same work, max time)
    e2e_tok, t_e2e, h2d, d2h = e2e_host(sv, m, wl, dev, rounds, st0, args.warmup, args.steps, seed)
    t_e2e = max_over_ranks(dist, t_e2e, dev)
    e2e_all = sum_over_ranks(dist, e2e_tok, dev)

    line = None
    if rank == 0:
        # the same rounds launched kernel by kernel, then timed per kernel class
        m.set_graphs(False)
        t_raw, _ = replay(sv, m, wl, dev, rounds, st0, args.warmup, args.steps, seed)
        m.set_graphs(True)
        kern = in_round_kernels(sv, m, wl, dev, rounds, st0, min(args.warmup, 3),
                                min(args.steps, 5), seed)
        R = n_seq * (d + 1)
        gem = kern["all_gemms"]
        tflops = gem["tflops"]
        n_layers = wl["n_layers"]
        shapes = [(4, (wl["n_q_heads"] + 2 * wl["n_kv_heads"]) * wl["head_dim"], wl["hidden"], n_layers, R),
                  (4, wl["hidden"], wl["n_q_heads"] * wl["head_dim"], n_layers, R),
                  (4, 2 * wl["ffn"], wl["hidden"], n_layers, R),
                  (4, wl["hidden"], wl["ffn"], n_layers, R), (6, V, wl["hidden"], 1, R)]
        traffic = measured_traffic(shapes)
        weight_bytes = sum(N * K * WEIGHT_BYTES[qt] * c for qt, N, K, c, _ in shapes)
        kv_bytes = n_layers * n_seq * wl["n_kv_heads"] * (wl["ctx"] + d + 1) * wl["head_dim"] * 4
        round_s = ms_per_step * 1e-3
        gemm_us_step = gem["seconds"] / max(min(args.steps, 5), 1) * 1e6
        del rounds
        torch.cuda.empty_cache()
        m.close()
        torch.cuda.empty_cache()
        legs, legs_in, extras = {}, {}, {}
        if not args.no_legs:
            legs["lmhead_greedy_H1024_V32000_nt3"], legs_in["lmhead"] = lmhead_leg(sv, synth, dev, hbm_peak)
            legs["accept_stochastic_12seq_d7_V248320"], legs_in["accept"] = accept_leg(sv, synth, dev, hbm_peak)
            legs["linear_sweep"] = compact_sweep(nt_sweep(sv, synth, dev))
            dec8, extras, dr8, anc8 = decoder8_leg(sv, synth, dev, args, hbm_peak)
            legs["decoder8_H4096_V151936_ctx4096_nt8"] = dec8
            legs_in["decoder8"] = dict(wl=dict(synth.WL_DECODER8), draft=dr8, anchor=anc8)
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
            "precision": "Q4/Q6 block ints, f16 activations, f32 accumulate; integer-weight sampler",
            "data": "synthetic (seeded N(0,1) activations and KV, uniform block ints, random-init "
                    "weights; draft logits = target nt=1 logits + N(0,0.5))",
            "config": {"workload": wl["name"], "n_layers": n_layers, "hidden": wl["hidden"],
                       "heads": f"{wl['n_q_heads']}/{wl['n_kv_heads']}x{wl['head_dim']}",
                       "ffn": wl["ffn"], "vocab": V, "context": wl["ctx"], "n_seq": n_seq,
                       "nt": d + 1, "rows": R, "temperature": T, "mode": "stochastic",
                       "drafter": "noisy target (target nt=1 logits + N(0,0.5)), untimed",
                       "graphs": True,
                       "l2": "inputs larger than L2 (7.2 GB of weights per round)",
                       "parallelism": f"replicas x{ws}"},
            "verify_round_us": round(round_s * 1e6, 1),
            "verify_round_us_raw_launch": round(t_raw / args.steps * 1e6, 1),
            "emitted_tokens_per_round": round(tokens_all / ws / args.steps, 3),
            "round_bytes": {"weights": weight_bytes, "kv": kv_bytes,
                            "gbs": round((weight_bytes + kv_bytes) / round_s / 1e9, 1),
                            "frac_of_hbm": round((weight_bytes + kv_bytes) / round_s / 1e9 / hbm_peak, 4)},
            "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": tc_sustained,
                         "unit": "TFLOP/s", "frac": round(tflops / tc_sustained, 4),
                         "traffic": None if traffic is None else round(traffic),
                         "kernel": f"verify GEMM (all {4 * n_layers + 1} launches of a round, "
                                   f"{R} rows), timed inside raw-launched rounds",
                         "algorithmic_flops_per_launch": round(gem["flops_per_launch"]),
                         "algorithmic_bytes_per_launch": round(gem["bytes_per_launch"]),
                         "hbm_gbs": round(gem["gbs"], 1), "hbm_peak": hbm_peak,
                         "hbm_frac": round(gem["gbs"] / hbm_peak, 4),
                         "gemm_us_per_step": round(gemm_us_step, 1),
                         "peak_kind": f"{peak_kind} bf16 sustained (fp16 = bf16 rate)"},
            "kernels_in_round": {k: {"us_per_launch": round(v["us_per_launch"], 2),
                                     "tflops": round(v["tflops"], 1), "gbs": round(v["gbs"], 1)}
                                 for k, v in kern.items()},
            "e2e": {"value": round(e2e_all / t_e2e, 2), "unit": "tok/s",
                    "api": "spec_verify_round_host (ids and drafts from host arrays, draft "
                           "logits from pinned host memory, outputs to host arrays)",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            # embed + 8 per layer (the first norm inside embed) + final norm and
            # LM head + row max, row sum, decide, resample + commit
            "gpu_launches": (1 + 8 * n_layers - 1 + 2 + 5) * args.steps,
            "clocks": clk.summary(),
        }
        if extras:
            line.update(extras)
        if ws == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl, tokens_all / args.steps, legs_in)
        line["workloads"] = legs  # last: the compact legs end the line
    else:
        m.close()
    if line is not None:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


# --------------------------------------------------------------------------
# profiling drivers (no JSON line)
# --------------------------------------------------------------------------
def linear_only(spec: str, nt: int = 8, reps: int = 3, tc: bool = False):
    """spec_linear_q (or, with tc, spec_linear_q_tc) at nt rows on packed
    synthetic matrices, `spec` = 'QT:N:K,QT:N:K,...', each launched `reps`
    times."""
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    from speculative_decoding_verification_round_gb300 import synth
    dev = torch.device("cuda:0")
    gen = synth.torch_gen(3, dev)
    for item in spec.split(","):
        qt, N, K = (int(v) for v in item.split(":"))
        w = synth.q_weight_torch(gen, qt, N, K, dev)
        qm = sv.QMat(w, max_rows=max(nt, 16))
        x = synth.f16_normal_torch(gen, (nt, K), dev).view(torch.int16)
        y = torch.empty((nt, N), dtype=torch.float32, device=dev)
        for _ in range(reps):
            (sv.spec_linear_q_tc if tc else sv.spec_linear_q)(qm, x, nt, y)
        torch.cuda.synchronize()
        assert sv.spec_error_check(None) == 0
        qm.close()
        del w
    print("linear-only ok")


def round_only(n_layers: int, warm: int = 2, reps: int = 2):
    """Stochastic rounds of the batched workload at `n_layers` layers (the
    last `reps` inside the NVTX range "rounds"), for launch lists."""
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    from speculative_decoding_verification_round_gb300 import synth
    dev = torch.device("cuda:0")
    wl = dict(synth.WL_DECODER14B, n_layers=n_layers)
    n = warm + reps
    m = build_model(sv, synth, wl, dev, wl["ctx"] + (wl["d"] + 1) * (n + 2) + 64)
    fill_context(sv, synth, m, wl, dev, seed=2)
    st0 = state0_of(wl)
    set_state(sv, m, st0)
    rounds = record_stochastic(sv, synth, m, wl, dev, n, 0x5EED)
    set_state(sv, m, st0)
    sid = torch.arange(wl["n_seq"], dtype=torch.int32, device=dev)
    n_acc = torch.zeros(wl["n_seq"], dtype=torch.int32, device=dev)
    em = torch.zeros((wl["n_seq"], wl["d"] + 1), dtype=torch.int32, device=dev)
    for j in range(n):
        if j == warm:
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_push("rounds")
        dr, qs = rounds[j]
        sv.spec_verify_round(m, wl["n_seq"], sid, dr, wl["d"], qs, False, wl["temperature"],
                             0x5EED, n_acc, em)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    assert sv.spec_error_check(m) == 0
    m.close()
    print("round-only ok")


def decoder8_only(warm: int = 3, reps: int = 3):
    """Greedy nt = 8 rounds of the 8-layer H 4096 decoder (graph-replayed,
    drafts on the target's greedy chain); the last `reps` run inside the
    NVTX range "rounds", for launch lists."""
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    from speculative_decoding_verification_round_gb300 import synth
    dev = torch.device("cuda:0")
    wl = dict(synth.WL_DECODER8)
    d, n = wl["d"], warm + reps
    m = build_model(sv, synth, wl, dev, wl["ctx"] + 8 * (n + 4) + 64)
    fill_context(sv, synth, m, wl, dev, seed=1)
    anchor = 1234
    drafts = record_chain(sv, synth, m, wl, dev, n, anchor, np.random.default_rng(wl["seed"]))
    sid = torch.zeros(1, dtype=torch.int32, device=dev)
    n_acc = torch.zeros(1, dtype=torch.int32, device=dev)
    em = torch.zeros((1, d + 1), dtype=torch.int32, device=dev)
    sv.spec_state_set(m, [0], n_past=[wl["ctx"]], emit_idx=[0], anchor=[anchor])
    for j in range(n):
        if j == warm:
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_push("rounds")
        dr = torch.tensor([drafts[j]], dtype=torch.int32, device=dev)
        sv.spec_verify_round(m, 1, sid, dr, d, n_acc=n_acc, emitted=em)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    assert sv.spec_error_check(m) == 0
    m.close()
    print("decoder8-only ok")


def draft_only(n_layers: int, warm: int = 3, reps: int = 3):
    """nt = 1 forwards (graph-replayed d = 0 rounds) of the 0.5B-class draft
    at `n_layers` layers and a 4096-position context; the last `reps` run
    inside the NVTX range "draft"."""
    import torch
    import speculative_decoding_verification_round_gb300 as sv
    from speculative_decoding_verification_round_gb300 import synth
    dev = torch.device("cuda:0")
    wl = dict(synth.WL_DRAFT05B, n_layers=n_layers)
    dm = build_model(sv, synth, wl, dev, wl["ctx"] + 64)
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
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-legs", action="store_true",
                    help="only the headline workload (no LM-head, accept, sweep, decoder-8 legs)")
    ap.add_argument("--extras", action="store_true",
                    help="also the adaptive-depth and full-round (with draft) legs on decoder-8")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the raw nvidia-smi clock samples in this file")
    ap.add_argument("--linear-only", default=None,
                    help="profiling driver: QT:N:K[,QT:N:K...] verify-GEMM launches only")
    ap.add_argument("--linear-rows", type=int, default=8, help="rows of --linear-only")
    ap.add_argument("--linear-tc", action="store_true",
                    help="--linear-only on the tensor-core GEMM of multi-sequence rounds")
    ap.add_argument("--round-only", type=int, default=None, metavar="LAYERS",
                    help="profiling driver: stochastic rounds of the batched workload")
    ap.add_argument("--decoder8-only", action="store_true",
                    help="profiling driver: greedy nt=8 rounds of the 8-layer decoder (NVTX 'rounds')")
    ap.add_argument("--draft-only", type=int, default=None, metavar="LAYERS",
                    help="profiling driver: nt = 1 forwards of the 0.5B-class draft")
    args = ap.parse_args()
    if args.linear_only:
        linear_only(args.linear_only, nt=args.linear_rows, tc=args.linear_tc)
        return
    if args.round_only:
        round_only(args.round_only)
        return
    if args.decoder8_only:
        decoder8_only()
        return
    if args.draft_only:
        draft_only(args.draft_only)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
