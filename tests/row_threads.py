"""Evaluate a per-row function over row chunks in several threads.

The oracle's C functions compute every row on its own and are called through
ctypes, which releases the GIL for the duration of the call, so row chunks run
in parallel threads and concatenate to exactly the single-call result. Used to
gate full-size launches on every row in seconds rather than minutes.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np


def host_threads() -> int:
    """Cores this process may run on (its affinity mask)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _concat(parts):
    if parts[0] is None:
        return None
    return np.concatenate(parts, axis=0)


def map_rows(fn, *row_arrays, threads=None, min_rows=64):
    """fn(*chunks) over contiguous row chunks of row_arrays (same row count);
    returns what fn(*row_arrays) would: an array, or a tuple of arrays (or
    None entries), concatenated along rows."""
    M = row_arrays[0].shape[0]
    n = min(threads or host_threads(), max(1, M // min_rows))
    if n <= 1:
        return fn(*row_arrays)
    bounds = [(M * i // n, M * (i + 1) // n) for i in range(n)]
    with ThreadPoolExecutor(max_workers=n) as ex:
        parts = list(ex.map(lambda ab: fn(*(a[ab[0]:ab[1]] for a in row_arrays)), bounds))
    if isinstance(parts[0], tuple):
        return tuple(_concat([p[k] for p in parts]) for k in range(len(parts[0])))
    return _concat(parts)
