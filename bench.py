"""Benchmark of libscan's hot path: one step = scan_fwd + scan_bwd of the scalar
scan on the dense [B=8, C=1536, T=4096] fp32 workload (synthetic, seeded).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dense_4k|dense_64k] [--no-rows]

Prints one JSON line (rank 0). `value` is whole-job scan elements/s of the
fwd+bwd step with inputs resident in HBM (CUDA events on the launching stream,
L2 flushed between steps); `e2e` is the same metric through the C ABI's
host-buffer step (scan_step_host: pinned host inputs and results, the copies
pipelined with the scans over row pieces), host<->device copies inside the
timed region. `rows` times every other workload the same way (the 64K-step
dense rows, the packed bidirectional bf16 rows, the 4x4 block form, the log
space, the outer-product state), fwd and bwd, each against the measured copy
peak and against the library's own copy kernels (`copy`).
`--impl reference` times the fp64 CPU oracle on the host cores instead.
Under torchrun (N > 1) every rank scans its own copy of the workload (weak
scaling, no collective on the data path); the step time is the max over ranks.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "scan elements/s and achieved HBM GB/s (fwd, fwd+bwd) at B=8 C=1536 T=4K–64K"
UNIT = "elem/s"
# fp32 algorithmic bytes per element: fwd reads a, x and writes h; bwd reads a,
# h, dh and writes da, dx (h0 / dh0 are per row, < 0.1 %)
FWD_BYTES = 12
BWD_BYTES = 20
# the pages' figure for this workload: "associative_scan_triton" README,
# kernel-level Fwd+Bwd table, seqlen 4096: 0.602 ms on an H100 (fp32 inferred)
PAGES_FWD_BWD_MS = {"dense_4k": 0.602, "dense_64k": 9.212}
# dram__bytes_read.sum + dram__bytes_write.sum per launch of the backward
# kernel on dense_4k, from an ncu capture, with the digest of the sources that
# build that kernel and choose its launch shape at the time of the capture.
# When the sources differ from the digest the figure no longer describes the
# kernel that runs, and the line reports traffic as null.
BWD_TRAFFIC = {"dense_4k": {"bytes": 961830912, "digest": "4caca3090d8f5eda"}}
KERNEL_SOURCES = ("scan_scalar.cuh", "scan_internal.h", "scan_scalar_bwd_f32.cu", "scan_api.cu")
L2_FLUSH_BYTES = 256 << 20
COPY_BYTES = 1 << 30  # per direction, for the copy-ceiling kernels


def kernel_digest() -> str:
    """sha256 over the sources of the dense scalar kernels and their planner."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "associative_affine_scan_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def bwd_traffic(workload: str):
    t = BWD_TRAFFIC.get(workload)
    if not t or t["bytes"] is None or t["digest"] != kernel_digest():
        return None
    return t["bytes"]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def __enter__(self):
        sel = []
        try:
            uuid = torch.cuda.get_device_properties(self.dev).uuid
            sel = ["-i", f"GPU-{uuid}"]
        except Exception:
            sel = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for line in (getattr(self, "out", "") or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def make_workload(name: str, rank: int):
    from associative_affine_scan_gb300 import workloads
    if name == "dense_4k":
        return workloads.dense_4k(seed=rank)
    if name == "dense_64k":
        return workloads.dense_64k(seed=rank)
    raise ValueError(name)


def run_ours(args, world, rank, local):
    import associative_affine_scan_gb300 as scan
    if not os.path.exists(scan.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    w = make_workload(args.workload, rank)
    B, C, T = w.a.shape
    n = B * C * T
    a, x, dh = (t.to(dev) for t in (w.a, w.x, w.dh))
    h0 = w.h0.to(dev) if w.h0 is not None else None
    h = torch.empty_like(a)
    da, dx = torch.empty_like(a), torch.empty_like(a)
    dh0 = torch.empty(B, C, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    # The two C-ABI calls are captured once into CUDA graphs on a dedicated
    # stream and replayed, so the host-side marshalling of the binding does
    # not leave the GPU idle inside the timed events (each replay launches the
    # same single kernel the direct call launches).
    gs = torch.cuda.Stream(dev)
    gs.wait_stream(stream)
    with torch.cuda.stream(gs):
        for _ in range(args.warmup):
            flush.zero_()
            scan.scan_fwd(a, x, h0, out=h)
            scan.scan_bwd(a, h, dh, h0, out=(da, dx, dh0))
    torch.cuda.synchronize()
    if scan.scan_get_device_status(dev, gs) != scan.SCAN_OK:
        raise RuntimeError("device status not OK after warm-up")
    g_fwd, g_bwd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_fwd, stream=gs):
        scan.scan_fwd(a, x, h0, out=h)
    with torch.cuda.graph(g_bwd, stream=gs):
        scan.scan_bwd(a, h, dh, h0, out=(da, dx, dh0))
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        with torch.cuda.stream(gs):
            for i in range(args.steps):
                flush.zero_()  # L2 flush between timed steps, outside the event pair
                ev[i][0].record(gs)
                g_fwd.replay()
                ev[i][1].record(gs)
                g_bwd.replay()
                ev[i][2].record(gs)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    barrier(world)
    status = scan.scan_get_device_status(dev, gs)
    if status != scan.SCAN_OK:
        raise RuntimeError(f"device status {scan.scan_status_string(status)}")
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    step_ms = [f + b for f, b in zip(fwd_ms, bwd_ms)]
    ms_local = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(ms_local, world, dev)
    fwd_avg = max_over_ranks(sum(fwd_ms) / len(fwd_ms), world, dev)
    bwd_avg = max_over_ranks(sum(bwd_ms) / len(bwd_ms), world, dev)
    clocks = clk.summary()

    # ---- end to end through the same calls with pinned host buffers ----
    ha, hx, hdh = (t.pin_memory() for t in (w.a, w.x, w.dh))
    hh0 = w.h0.pin_memory() if w.h0 is not None else None
    out_h = torch.empty(a.shape, dtype=torch.float32).pin_memory()
    out_da, out_dx = (torch.empty(a.shape, dtype=torch.float32).pin_memory() for _ in range(2))
    out_dh0 = torch.empty(B, C, dtype=torch.float32).pin_memory()
    bytes_in = sum(t.numel() * t.element_size() for t in (ha, hx, hdh) + ((hh0,) if hh0 is not None else ()))
    bytes_out = sum(t.numel() * t.element_size() for t in (out_h, out_da, out_dx, out_dh0))

    # one library call per step: the library pipelines the copies in, the two
    # scans and the copies out over row pieces
    def e2e_step():
        scan.scan_step_host(ha, hx, hdh, hh0, out=(out_h, out_da, out_dx, out_dh0),
                            device=(a, x, h0, dh, h, da, dx, dh0))

    e2e_steps = max(3, min(args.steps, 10))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)

    # the other carry schemes on the same step (the planner chose stationary)
    variants = {}
    if not args.no_rows:
        for name, var in (("lookback", scan.SCAN_VARIANT_LOOKBACK),
                          ("stream", scan.SCAN_VARIANT_STREAM)):
            o = {"variant": var}
            vf = time_calls(lambda: scan.scan_fwd(a, x, h0, out=h, opts=o), args.steps, 3, flush,
                            stream)
            vb = time_calls(lambda: scan.scan_bwd(a, h, dh, h0, out=(da, dx, dh0), opts=o),
                            args.steps, 3, flush, stream)
            variants[name] = {"fwd_ms": vf, "bwd_ms": vb, "step_ms": vf + vb}
        if scan.scan_get_device_status(dev, stream) != scan.SCAN_OK:
            raise RuntimeError("device status not OK after the variant timings")

    extra, copy = {}, None
    if not args.no_rows:
        del a, x, dh, h, da, dx, dh0, flush
        torch.cuda.empty_cache()
        copy = measure_copy(dev, scan, max(3, min(args.steps, 10)))
        extra = measure_rows(args, dev, scan, ceiling=copy["ceiling_gbs"])

    spread = {"step_median_ms": float(np.median(step_ms)), "step_min_ms": min(step_ms),
              "fwd_median_ms": float(np.median(fwd_ms)), "fwd_min_ms": min(fwd_ms),
              "bwd_median_ms": float(np.median(bwd_ms)), "bwd_min_ms": min(bwd_ms)}
    return dict(n=n, B=B, C=C, T=T, ms=ms, fwd_ms=fwd_avg, bwd_ms=bwd_avg, wall=wall,
                clocks=clocks, e2e_ms=e2e_ms, bytes_in=bytes_in, bytes_out=bytes_out,
                w=w, extra=extra, copy=copy, spread=spread, variants=variants)


def time_calls(fn, steps, warmup, flush, stream):
    """Mean device time of fn (a few C-ABI calls): warm up, capture fn once into a
    CUDA graph on a dedicated stream, then time `steps` replays with CUDA events on
    that stream, the L2 flushed before each (outside the event pair)."""
    gs = torch.cuda.Stream(flush.device)
    gs.wait_stream(stream)
    with torch.cuda.stream(gs):
        for _ in range(warmup):
            flush.zero_()
            fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        fn()
    torch.cuda.synchronize()
    total = 0.0
    with torch.cuda.stream(gs):
        for _ in range(steps):
            flush.zero_()
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(gs)
            graph.replay()
            e.record(gs)
            torch.cuda.synchronize()
            total += s.elapsed_time(e)
    return total / steps


ROWS = ("dense_64k", "packed_bidir", "affine_4x4", "log_4k", "gdn_4k", "rglru_4k")


def measure_rows(args, dev, scan, names=ROWS, small=False, ceiling=None):
    """Throughput of every other workload, fwd and bwd, each timed alone (graph
    replays, L2 flushed between them); each workload is freed before the next.

    small: the packed row with 12 sequences instead of 64 (same 2 x 2048 rows,
    2.5 GB on the device), the size used for full ncu captures.
    ceiling: the library's copy ceiling in GB/s; each row's GB/s is also given
    as a fraction of it."""
    from associative_affine_scan_gb300 import workloads
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    steps, warm = max(1, min(args.steps, 10)), 3
    out = {}
    peak, _ = measured_peaks()
    runners = {
        "dense_64k": lambda: _row_dense(scan, workloads, dev, steps, warm, flush, stream),
        "packed_bidir": lambda: _row_packed(scan, workloads, dev, steps, warm, flush, stream,
                                            small),
        "affine_4x4": lambda: _row_affine(scan, workloads, dev, steps, warm, flush, stream),
        "log_4k": lambda: _row_log(scan, workloads, dev, steps, warm, flush, stream),
        "gdn_4k": lambda: _row_gdn(scan, workloads, dev, steps, warm, flush, stream),
        "rglru_4k": lambda: _row_rglru(scan, workloads, dev, steps, warm, flush, stream),
    }
    for name in names:
        try:
            r = runners[name]()
        except Exception as e:  # reported, not fatal: the other rows still print
            out[name] = {"error": f"{type(e).__name__}: {e}"}
            continue
        finally:
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
        for d in ("fwd", "bwd"):
            r[d + "_frac"] = r[d + "_gbs"] / peak
            if ceiling:
                r[d + "_frac_of_copy_kernel"] = r[d + "_gbs"] / ceiling
        tot_bytes = r["fwd_gbs"] * r["fwd_ms"] + r["bwd_gbs"] * r["bwd_ms"]
        r["fwd_bwd_gbs"] = tot_bytes / (r["fwd_ms"] + r["bwd_ms"])
        r["fwd_bwd_frac"] = r["fwd_bwd_gbs"] / peak
        out[name] = r
    return out


def _row_dense(scan, workloads, dev, steps, warm, flush, stream):
    # the 8 x 1536 x 65536 fp32 rows: 12 bytes per element forward, 20 backward
    w = workloads.dense_64k(seed=0)
    a, x, dh = w.a.to(dev), w.x.to(dev), w.dh.to(dev)
    del w
    h = scan.scan_fwd(a, x)
    n = a.numel()
    f_ms = time_calls(lambda: scan.scan_fwd(a, x, out=h), steps, warm, flush, stream)
    g = scan.scan_bwd(a, h, dh)
    b_ms = time_calls(lambda: scan.scan_bwd(a, h, dh, out=g), steps, warm, flush, stream)
    return {"elems": n, "fwd_ms": f_ms, "bwd_ms": b_ms,
            "fwd_gbs": n * FWD_BYTES / f_ms / 1e6, "bwd_gbs": n * BWD_BYTES / b_ms / 1e6,
            "fwd_bwd_elem_per_s": n / (f_ms + b_ms) * 1e3}


def measure_copy(dev, scan, steps):
    """GB/s (read + write) of the library's two copy kernels over COPY_BYTES,
    timed like the scan rows."""
    src = torch.empty(COPY_BYTES // 4, dtype=torch.float32, device=dev).uniform_()
    dst = torch.empty_like(src)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = {"bytes_per_direction": COPY_BYTES}
    peak, _ = measured_peaks()
    for name, mode in (("vec", scan.SCAN_COPY_VEC), ("tma", scan.SCAN_COPY_TMA)):
        ms = time_calls(lambda: scan.scan_copy(src, dst, mode, status=status), steps, 3, flush,
                        stream)
        gbs = 2 * COPY_BYTES / ms / 1e6
        out[name] = {"ms": ms, "gbs": gbs, "frac": gbs / peak}
    torch.cuda.synchronize()
    if int(status.item()) != 0 or not torch.equal(src, dst):
        raise RuntimeError("copy kernels: status or contents wrong")
    out["ceiling_gbs"] = max(out["vec"]["gbs"], out["tma"]["gbs"])
    del src, dst
    torch.cuda.empty_cache()
    return out


def _row_gdn(scan, workloads, dev, steps, warm, flush, stream):
    # per (head, step): fwd reads alpha, b, c (S each), v (D) and writes o (D)
    # plus an S x D checkpoint every 32 steps; bwd reads alpha, b, c, v, dout
    # and the checkpoints and writes dalpha, db, dc (S side: 16 S bytes) and
    # dv (D side: v, dout, dv, 12 D bytes)
    w = workloads.gdn_4k(seed=0)
    alpha, b, v, c, dout = (t.to(dev) for t in (w.alpha, w.b, w.v, w.c, w.dout))
    S, D = b.shape[-1], v.shape[-1]
    ws = torch.empty(scan.gdn_workspace_bytes(*alpha.shape, S, D), dtype=torch.uint8, device=dev)
    o, ck = scan.gdn_fwd(alpha, b, v, c, workspace=ws)
    n = alpha.numel()
    f_bytes = n * (4 + 8 * S + 8 * D) + ck.numel() * 4
    b_bytes = n * (8 + 16 * S + 12 * D) + ck.numel() * 4
    f_ms = time_calls(lambda: scan.gdn_fwd(alpha, b, v, c, checkpoints=ck, out=o, workspace=ws),
                      steps, warm, flush, stream)
    g = scan.gdn_bwd(alpha, b, v, c, ck, dout, workspace=ws)
    b_ms = time_calls(lambda: scan.gdn_bwd(alpha, b, v, c, ck, dout, out=g, workspace=ws), steps,
                      warm, flush, stream)
    return {"head_steps": n, "fwd_ms": f_ms, "bwd_ms": b_ms,
            "fwd_gbs": f_bytes / f_ms / 1e6, "bwd_gbs": b_bytes / b_ms / 1e6}


def _row_packed(scan, workloads, dev, steps, warm, flush, stream, small):
    w = workloads.packed_bidir(seed=0, n_seqs=12 if small else 64)
    af, xf, ar, xr, cu, dhf, dhr = (t.to(dev) for t in (w.af, w.xf, w.ar, w.xr, w.cu_seqlens,
                                                         w.dhf, w.dhr))
    hf, hr = scan.scan_bidir_fwd(af, xf, ar, xr, None, None, cu)
    n = 2 * af.numel()
    f_ms = time_calls(lambda: scan.scan_bidir_fwd(af, xf, ar, xr, None, None, cu, out=(hf, hr)),
                      steps, warm, flush, stream)
    g = scan.scan_bidir_bwd(af, hf, dhf, ar, hr, dhr, None, None, cu)
    b_ms = time_calls(lambda: scan.scan_bidir_bwd(af, hf, dhf, ar, hr, dhr, None, None, cu, out=g),
                      steps, warm, flush, stream)
    return {"elems": n, "sum_len": int(w.cu_seqlens[-1]), "fwd_ms": f_ms, "bwd_ms": b_ms,
            "fwd_gbs": n * 8 / f_ms / 1e6, "bwd_gbs": n * 14 / b_ms / 1e6,
            "fwd_bwd_elem_per_s": n / (f_ms + b_ms) * 1e3}


def _row_log(scan, workloads, dev, steps, warm, flush, stream):
    # log space: fwd reads log a, log x and writes h (12 B/elem); bwd reads
    # log a, log x, h, dh and writes d log a, d log x (24 B/elem)
    w = workloads.log_4k(seed=0)
    la, lx, ldh = w.log_a.to(dev), w.log_x.to(dev), w.dh.to(dev)
    hl = scan.scan_log_fwd(la, lx)
    n = la.numel()
    l_ms = time_calls(lambda: scan.scan_log_fwd(la, lx, out=hl), steps, warm, flush, stream)
    gl = scan.scan_log_bwd(la, lx, hl, ldh)
    lb_ms = time_calls(lambda: scan.scan_log_bwd(la, lx, hl, ldh, out=gl), steps, warm, flush,
                       stream)
    return {"elems": n, "fwd_ms": l_ms, "bwd_ms": lb_ms,
            "fwd_gbs": n * 12 / l_ms / 1e6, "bwd_gbs": n * 24 / lb_ms / 1e6}


def _row_rglru(scan, workloads, dev, steps, warm, flush, stream):
    # RG-LRU: fwd reads x, gate_a, gate_x and writes h (16 B/elem); bwd reads
    # x, gate_a, gate_x, h, dh and writes dx, dgate_a, dgate_x (32 B/elem);
    # segment_pos (4 B per (b, t), shared by the channels) and a_param are
    # below 0.1 % and not counted
    w = workloads.rglru_4k(seed=0)
    x, ga, gx, ap, dh, seg = (t.to(dev) for t in (w.x, w.gate_a, w.gate_x, w.a_param, w.dh,
                                                 w.segment_pos))
    h = scan.rglru_fwd(x, ga, gx, ap, seg)
    n = x.numel()
    f_ms = time_calls(lambda: scan.rglru_fwd(x, ga, gx, ap, seg, out=h), steps, warm, flush,
                      stream)
    g = scan.rglru_bwd(x, ga, gx, ap, h, dh, seg)
    b_ms = time_calls(lambda: scan.rglru_bwd(x, ga, gx, ap, h, dh, seg, out=g), steps, warm,
                      flush, stream)
    return {"elems": n, "fwd_ms": f_ms, "bwd_ms": b_ms,
            "fwd_gbs": n * 16 / f_ms / 1e6, "bwd_gbs": n * 32 / b_ms / 1e6}


def _row_affine(scan, workloads, dev, steps, warm, flush, stream):
    # per (b, t, n) block: fwd reads A, B and writes H (3 x 64 bytes); bwd reads
    # A, H, dH and writes dA, dB (5 x 64 bytes)
    w = workloads.affine_4x4(seed=0)
    A, Bm, dH = w.A.to(dev), w.Bm.to(dev), w.dH.to(dev)
    H = scan.affine_scan_fwd(A, Bm)
    nb = w.n_blocks
    f_ms = time_calls(lambda: scan.affine_scan_fwd(A, Bm, out=H), steps, warm, flush, stream)
    g = scan.affine_scan_bwd(A, H, dH)
    b_ms = time_calls(lambda: scan.affine_scan_bwd(A, H, dH, out=g), steps, warm, flush, stream)
    return {"blocks": nb, "fwd_ms": f_ms, "bwd_ms": b_ms,
            "fwd_gbs": nb * 192 / f_ms / 1e6, "bwd_gbs": nb * 320 / b_ms / 1e6}


def oracle_fwd_bwd(w, rows, threads=1):
    """The fp64 oracle on `rows` rows of the workload (fwd then bwd); with
    threads > 1 the rows are split into that many slices run at once (the
    oracle is C called through ctypes, which releases the GIL)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    B, C, T = w.a.shape
    a = w.a.reshape(B * C, T)[:rows].double().numpy()[None]
    x = w.x.reshape(B * C, T)[:rows].double().numpy()[None]
    dh = w.dh.reshape(B * C, T)[:rows].double().numpy()[None]
    h0 = w.h0.reshape(B * C)[:rows].double().numpy()[None] if w.h0 is not None else None
    threads = max(1, min(threads, rows))
    cuts = [rows * i // threads for i in range(threads + 1)]

    def part(i):
        r0, r1 = cuts[i], cuts[i + 1]
        hp = None if h0 is None else h0[:, r0:r1]
        oracle.scan_fwd(a[:, r0:r1], x[:, r0:r1], hp)
        oracle.scan_bwd(a[:, r0:r1], x[:, r0:r1], dh[:, r0:r1], hp)

    t0 = time.perf_counter()
    if threads == 1:
        part(0)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(part, range(threads)))
    return time.perf_counter() - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _timed_passes(w, rows, threads, budget_s):
    """Repeat oracle passes over `rows` rows until about budget_s seconds of
    wall time have run; returns (passes, seconds)."""
    first = oracle_fwd_bwd(w, rows, threads)
    passes = max(1, int(budget_s / max(first, 1e-9)))
    dt = sum(oracle_fwd_bwd(w, rows, threads) for _ in range(passes))
    return passes, dt


def cpu_baseline(w, cpu_s: float = 8.0, all_core_cpu_s: float = 24.0):
    """Oracle elements/s on bounded samples of whole rows of the workload:
    single-threaded (about cpu_s seconds of CPU work) and with the rows split
    over every host core (about all_core_cpu_s seconds of CPU work). The
    reported value is the all-core one."""
    B, C, T = w.a.shape
    rows = B * C
    probe = min(rows, 64)
    per_row = oracle_fwd_bwd(w, probe) / probe
    take1 = int(max(1, min(rows, cpu_s / max(per_row, 1e-9))))
    p1, dt1 = _timed_passes(w, take1, 1, cpu_s)
    cores = host_cores()
    taken = int(max(1, min(rows, all_core_cpu_s / max(per_row, 1e-9))))
    pn, dtn = _timed_passes(w, taken, cores, all_core_cpu_s / cores)
    return {"value": pn * taken * T / dtn, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{pn} passes over {taken} of {rows} rows x T={T} (fwd+bwd, fp64), rows "
                      f"split over {cores} threads, {dtn:.2f} s",
            "single_thread": {"value": p1 * take1 * T / dt1, "cores": 1,
                              "sample": f"{p1} passes over {take1} rows, {dt1:.2f} s"}}


def run_reference(args, world, rank):
    """The reference arm: the fp64 CPU oracle, as it stands, on the host cores."""
    if rank != 0:
        return None
    w = make_workload(args.workload, 0)
    B, C, T = w.a.shape
    rows = B * C
    probe = min(rows, 32)
    per_row = oracle_fwd_bwd(w, probe) / probe
    cores = host_cores()
    # each step: as many rows as the host's cores finish in ~4 s, so the whole
    # run ends in minutes
    take = int(max(1, min(rows, cores * 4.0 / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        oracle_fwd_bwd(w, max(1, take // 8), cores)
    times = [oracle_fwd_bwd(w, take, cores) for _ in range(args.steps)]
    dt = sum(times) / len(times)
    value = take * T / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "C": C, "T": T,
                   "step": "oracle scan fwd + bwd on a bounded row sample"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{take} of {rows} rows x T={T} per step (fwd+bwd, fp64), "
                                   f"split over {cores} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="dense_4k", choices=["dense_4k", "dense_64k"])
    ap.add_argument("--no-rows", action="store_true",
                    help="skip the other workloads and the copy kernels (the headline step only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--row", choices=ROWS + ("copy",),
                    help="time only this form (fwd and bwd, --steps timed calls each) and print "
                         "its figures; the command the ncu captures of that form use ('copy': "
                         "the two copy-ceiling kernels)")
    ap.add_argument("--small", action="store_true",
                    help="with --row packed_bidir: 12 sequences instead of 64 (ncu capture size)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()

    if args.row:
        import associative_affine_scan_gb300 as scan
        if not os.path.exists(scan.LIB_PATH):
            import __graft_entry__
            __graft_entry__.build()
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        if args.row == "copy":
            out = measure_copy(dev, scan, args.steps)
            if rank == 0:
                print(json.dumps({"row": "copy", **out}), flush=True)
            return
        rows = measure_rows(args, dev, scan, names=(args.row,), small=args.small)
        if rank == 0:
            print(json.dumps({"row": args.row, "small": args.small, **rows[args.row]}), flush=True)
        return

    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    r = run_ours(args, world, rank, local)
    if rank != 0:
        barrier(world)
        return
    peak, peak_kind = measured_peaks()
    n_total = r["n"] * world
    value = n_total / (r["ms"] * 1e-3)
    bwd_gbs = r["n"] * BWD_BYTES / (r["bwd_ms"] * 1e-3) / 1e9
    fwd_gbs = r["n"] * FWD_BYTES / (r["fwd_ms"] * 1e-3) / 1e9
    step_gbs = r["n"] * (FWD_BYTES + BWD_BYTES) / (r["ms"] * 1e-3) / 1e9
    pages_ms = PAGES_FWD_BWD_MS.get(args.workload)
    vs = value / (r["n"] / (pages_ms * 1e-3)) if pages_ms else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": vs, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "B": r["B"], "C": r["C"], "T": r["T"],
                   "step": "scan_fwd + scan_bwd (fp32)", "l2": "flushed (256 MB write) between "
                   "timed steps; per-step working set 1.2 GB > L2"},
        "gbs": step_gbs,
        "fwd": {"ms": r["fwd_ms"], "elem_per_s": r["n"] / (r["fwd_ms"] * 1e-3), "gbs": fwd_gbs,
                "frac": fwd_gbs / peak},
        "bwd": {"ms": r["bwd_ms"], "elem_per_s": r["n"] / (r["bwd_ms"] * 1e-3), "gbs": bwd_gbs,
                "frac": bwd_gbs / peak},
        "roofline": {"bound": "hbm", "kernel": "scalar_scan_kernel_r72 (backward)",
                     "achieved": bwd_gbs, "peak": peak, "unit": "GB/s", "frac": bwd_gbs / peak,
                     "peak_source": peak_kind,
                     "traffic": bwd_traffic(args.workload), "kernel_digest": kernel_digest()},
        "e2e": {"value": n_total / (r["e2e_ms"] * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": r["bytes_in"], "d2h_bytes_per_step": r["bytes_out"]},
        "gpu_launches": 2 * args.steps,
        "clocks": r["clocks"],
        "wall_s": r["wall"],
        "baseline_context": {"ms": pages_ms, "hardware": "H100 80GB",
                             "source": "associative_scan_triton README, kernel-level Fwd+Bwd"},
    }
    line["timing_spread"] = r["spread"]  # this rank's median and minimum over the timed steps
    if r["variants"]:
        line["variants"] = dict(
            {"stationary (planner)": {"fwd_ms": r["fwd_ms"], "bwd_ms": r["bwd_ms"],
                                      "step_ms": r["ms"]}}, **r["variants"])
    if r["copy"]:
        line["copy"] = r["copy"]
        line["roofline"]["frac_of_copy_kernel"] = bwd_gbs / r["copy"]["ceiling_gbs"]
    if r["extra"]:
        line["rows"] = r["extra"]
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(r["w"])
    print(json.dumps(line), flush=True)
    barrier(world)


if __name__ == "__main__":
    main()
