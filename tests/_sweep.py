"""Exhaustive comparison of full-size GPU results with the fp64 oracle.

The full-size workloads (up to 805 M elements) are checked batch by batch: a
batch of rows, channels or lanes is copied to the host, the oracle computes
the same batch in fp64, and each named output's error is reduced to its
maximum. Batches run on a thread pool with one thread per host core: the
oracle is C called through ctypes and numpy's large-array operations both
release Python's lock, so the batches run on separate cores while host memory
stays bounded by (threads x batch size).
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np


def host_threads() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(n, 32))


def as_f64(t):
    if hasattr(t, "detach"):
        return t.detach().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def max_rel(got, ref, scale=None) -> float:
    """max |got - ref| / max(1, |ref|[, scale]) over all elements."""
    got = as_f64(got)
    ref = np.asarray(ref, dtype=np.float64)
    if got.size == 0:
        return 0.0
    den = np.maximum(1.0, np.abs(ref))
    if scale is not None:
        den = np.maximum(den, scale)
    return float(np.max(np.abs(got - ref) / den))


def worst(a: float, b: float) -> float:
    """The larger of two errors; NaN if either is NaN (Python's max would
    drop a NaN that is not its first argument)."""
    if a != a or b != b:
        return float("nan")
    return max(a, b)


def batches(n: int, size: int):
    return [(i, min(n, i + size)) for i in range(0, n, size)]


def sweep(n: int, size: int, check) -> dict:
    """Run check(i0, i1) -> {name: error} over [0, n) in batches of `size`
    on the host cores; returns the maximum of each name over all batches,
    plus "batches" (how many ran) and "items" (n)."""
    parts = batches(n, size)
    with ThreadPoolExecutor(max_workers=host_threads()) as ex:
        results = list(ex.map(lambda ab: check(*ab), parts))
    out: dict = {}
    for r in results:
        for k, v in r.items():
            out[k] = worst(out.get(k, 0.0), v)
    out["batches"] = len(parts)
    out["items"] = n
    return out
