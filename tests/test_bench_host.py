"""Host-side logic of bench.py that the measurement contract rests on: the
clock summary taken from nvidia-smi samples (only samples inside the timed
region count; throttle reasons are reported) and the DRAM-traffic record
(used only while it was taken on the current verify-GEMM source).  CPU only."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def sample(mhz, mx=2070, hw="Not Active", thermal="Not Active", power="Not Active"):
    return f"0, {mhz}, {mx}, 900.0, 0x0, {hw}, {thermal}, Not Active, {power}\n"


def sampler_with(tmp_path, before, during):
    path = tmp_path / "clocks.csv"
    path.write_text("".join(before + during))
    c = bench.ClockSampler(0, str(path))
    c.proc = object()           # as if nvidia-smi had been started
    c.start_line = len(before)  # lines present when the timed region began
    return c


def test_only_samples_inside_the_timed_region_count(tmp_path):
    c = sampler_with(tmp_path, [sample(345), sample(345)],
                     [sample(2070), sample(2055), sample(2070, power="Active")])
    s = c.summary()
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_throttle_reasons_are_reported(tmp_path):
    c = sampler_with(tmp_path, [], [sample(1500, hw="Active"), sample(1490, thermal="Active")])
    s = c.summary()
    assert s["sm_mhz"] == 1495
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_a_region_shorter_than_the_interval_takes_the_last_sample(tmp_path):
    c = sampler_with(tmp_path, [sample(2000), sample(2070)], [])
    s = c.summary()
    assert s["sm_mhz"] == 2070 and s["samples"] == 1


def test_no_sampler_reports_unsampled():
    c = bench.ClockSampler(0, "/nonexistent/clocks.csv")
    assert c.summary()["reasons"] == ["unsampled"]


def test_traffic_record_is_used_only_for_its_source(tmp_path, monkeypatch):
    src = tmp_path / "tcgemm.cu"
    src.write_text("// kernel v1\n")
    rec = tmp_path / "traffic.json"
    rec.write_text(json.dumps({
        "source_sha256": hashlib.sha256(src.read_bytes()).hexdigest(),
        "dram_bytes_per_launch": {"4:64:128": 100, "6:32:64": 400}}))
    monkeypatch.setattr(bench, "TRAFFIC_RECORD", str(rec))
    monkeypatch.setattr(bench, "GEMM_SRC", str(src))
    # per launch over the mix: (3 x 100 + 1 x 400) / 4
    assert bench.measured_traffic([(4, 64, 128, 3), (6, 32, 64, 1)]) == pytest.approx(175.0)
    assert bench.measured_traffic([(4, 64, 128, 1), (8, 16, 32, 1)]) is None  # shape not captured
    assert bench.measured_traffic([(4, 64, 128, 1, 192)]) is None             # rows not captured
    src.write_text("// kernel v2\n")
    assert bench.measured_traffic([(4, 64, 128, 3)]) is None                  # source changed


def test_committed_traffic_record_shows_no_re_reads():
    """The record under profiles/: every captured shape moved its packed
    weight bytes once (within 10%, plus the activation rows it reads and the
    outputs it writes).  A record older than the kernel's source is not used
    by the bench (traffic null) and is not judged here."""
    if not os.path.exists(bench.TRAFFIC_RECORD):
        pytest.skip("no traffic record for the bench's workload: the bench reports traffic null")
    rec = json.load(open(bench.TRAFFIC_RECORD))
    sha = hashlib.sha256(open(bench.GEMM_SRC, "rb").read()).hexdigest()
    if rec["source_sha256"] != sha:
        pytest.skip("the record predates the kernel source: the bench reports traffic null")
    for key, b in rec["dram_bytes_per_launch"].items():
        f = list(map(int, key.split(":")))
        qt, N, K = f[:3]
        R = f[3] if len(f) > 3 else 0
        w = N * K * bench.WEIGHT_BYTES[qt]
        io = R * K * 2 + R * N * 4  # fp16 activations in, fp32 outputs out
        assert 0.98 * w <= b <= 1.10 * (w + io), key  # no re-reads
