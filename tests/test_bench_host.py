"""Host-side logic of bench.py without a GPU: the max-over-ranks timing and the
barrier under a 2-rank gloo group, and the reference arm's JSON line."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    m = bench.max_over_ranks(1.5 + rank, w, torch.device("cpu"))
    out[rank] = m
    dist.destroy_process_group()


def test_max_over_ranks_under_gloo():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_clock_summary_reads_median_max_and_active_reasons():
    """The clocks record beside every bench line: the median SM clock under
    sampling, the highest maximum seen, and every throttle reason reported
    Active at least once; lines that do not parse are skipped."""
    bench = _bench()
    cs = bench.ClockSampler(0)
    cs.out = "\n".join([
        "2070, 2070, 900.5, Not Active, Not Active, Not Active, Not Active",
        "1980, 2070, 1390.0, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 1200.0, Not Active, Not Active, Not Active, Not Active",
        "[N/A], 2070, 10.0, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ])
    s = cs.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    cs.out = "1500, 2070, 1400.0, Active, Not Active, Active, Not Active"
    assert cs.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    cs.out = ""
    assert cs.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_traffic_is_reported_only_for_the_sources_it_was_captured_on(monkeypatch):
    """roofline.traffic comes from one ncu capture; it is reported only while
    the kernel's sources hash to the digest stored with it, else null."""
    bench = _bench()
    stored = bench.BWD_TRAFFIC["dense_4k"]
    monkeypatch.setattr(bench, "kernel_digest", lambda: stored["digest"])
    assert bench.bwd_traffic("dense_4k") == stored["bytes"]
    assert bench.bwd_traffic("dense_64k") is None
    monkeypatch.setattr(bench, "kernel_digest", lambda: "0" * 16)
    assert bench.bwd_traffic("dense_4k") is None


def test_kernel_digest_covers_its_sources(tmp_path, monkeypatch):
    """The digest changes when any of the kernel's sources changes."""
    bench = _bench()
    src = tmp_path / "associative_affine_scan_gb300" / "csrc"
    src.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES:
        (src / name).write_bytes(b"x")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d0 = bench.kernel_digest()
    for name in bench.KERNEL_SOURCES:
        (src / name).write_bytes(b"y")
        assert bench.kernel_digest() != d0
        (src / name).write_bytes(b"x")
    assert bench.kernel_digest() == d0


def test_peaks_fall_back_when_the_measured_file_is_absent(tmp_path, monkeypatch):
    bench = _bench()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (6800.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6790.0}))
    assert bench.measured_peaks() == (6790.0, "measured")
