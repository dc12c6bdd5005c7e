"""Streams a full-size workload's GPU results through the CPU oracle.

The GPU computes the whole workload first.  Then this helper walks the
elements in block-aligned slices: the calling thread copies each slice's
inputs and GPU outputs to the host, and a pool of host threads (one per
core) runs the unchanged, single-threaded oracle on the slice and compares
bit for bit.  Every block is an independent oracle problem given its global
element index (the Philox counter), so a slice needs nothing from outside
it.  The oracle's C functions release the GIL; so do numpy's comparisons.
No oracle input comes from the CUDA path: each slice's oracle starts from
its own state (zero error buffers) and carries that state across steps.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np


def host_threads() -> int:
    if hasattr(os, "sched_getaffinity"):
        return max(1, len(os.sched_getaffinity(0)))
    return os.cpu_count() or 1


def slices(n: int, step: int):
    """[lo, hi) bounds covering [0, n) in pieces of `step` elements (the last shorter)."""
    return [(lo, min(lo + step, n)) for lo in range(0, n, step)]


def run(bounds, fetch, check, threads: int | None = None) -> int:
    """fetch(lo, hi) on this thread, then check(lo, hi, data) on the pool.
    At most threads + 4 fetched slices are held at once.  Returns the number
    of elements checked; re-raises the first failure."""
    threads = threads or host_threads()
    limit = threads + 4
    checked = 0
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        pending = {}
        for lo, hi in bounds:
            pending[ex.submit(check, lo, hi, fetch(lo, hi))] = hi - lo
            if len(pending) >= limit:
                done, _ = cf.wait(pending, return_when=cf.FIRST_COMPLETED)
                for f in done:
                    f.result()
                    checked += pending.pop(f)
        for f in cf.as_completed(list(pending)):
            f.result()
            checked += pending[f]
    return checked


def same_bits(a: np.ndarray, b: np.ndarray) -> bool:
    """Byte-for-byte equality of two arrays (any dtypes, same byte length)."""
    a = np.ascontiguousarray(a).view(np.uint8)
    b = np.ascontiguousarray(b).view(np.uint8)
    return a.shape == b.shape and bool(np.array_equal(a, b))
