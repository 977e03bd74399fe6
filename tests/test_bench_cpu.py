"""Host logic of bench.py that needs no GPU: byte counts, peaks, clock records, defaults."""

import json
import sys

import pytest

import bench
from kernelized_causal_self_gb300 import inputs


def test_algorithmic_bytes_per_token_head():
    w = inputs.WORKLOADS[bench.MAIN]
    assert (w.D, w.M) == (64, 64)
    assert bench.fwd_bytes(w) == 512              # q, k, v read + out written, bf16
    assert bench.bwd_bytes(w) == 1280             # q, k, v, dout bf16 + dq, dk, dv float32
    d = inputs.WORKLOADS["decode_s256h8d64_prefill1024_steps3072"]
    assert bench.decode_bytes(d) == 2 * 64 * 64 * 4 + 2 * 64 * 4 + 4 * 64 * 2
    assert bench.extend_bytes(d, 64) == 64 * 512 + 2 * 64 * 64 * 4 + 2 * 64 * 4


def test_peaks_measured_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6800.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6672.2, "bf16_tflops": 1917.6}))
    p = bench.load_peaks()
    assert p["source"] == "measured" and p["hbm_gbs"] == 6672.2


def test_clock_record_parsing(tmp_path):
    log = tmp_path / "clocks.csv"
    log.write_text(
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
        "0, 2055, 2070, 1385.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
        "0, 2070, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
        "garbage line\n")
    c = bench.Clocks(0)
    c.path = str(log)
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    c2 = bench.Clocks(0)
    c2.path = str(tmp_path / "empty.csv")
    (tmp_path / "empty.csv").write_text("")
    assert c2.summary() is None


def test_default_run_meets_the_timing_rules(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert a.gpus == 1 and a.impl == "ours"
    assert a.warmup >= 3 and a.steps >= 1


def test_kernel_revision_is_stable():
    r = bench.kernel_revision()
    assert r == bench.kernel_revision() and len(r) == 16
    int(r, 16)


@pytest.mark.parametrize("world", [1])
def test_single_process_needs_no_process_group(world, monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup(None) == (1, 0, 0)
    bench.barrier(world)  # no process group: a no-op
