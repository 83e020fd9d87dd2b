"""Evaluating the oracle's attention over host threads (oracle; test infrastructure).

No arithmetic of the method lives here: the rows asked for are grouped by request, a
request's rows are cut into pieces of about equal cost, each piece is handed to the unchanged
``paged_attention`` on those rows, and the calls run on a thread pool, longest first (numpy
releases the GIL inside its loops).  The result of a request's rows does not depend on the
other requests of the batch ("one mixed step equals each request alone"), nor a row's on the
other rows asked for; the oracle's tests pin both.
"""
from __future__ import annotations

import math

import numpy as np

from .attention import paged_attention


def _openblas_thread_setters():
    """(get, set) of the OpenBLAS that numpy loaded, or None: the oracle's per-request calls run
    in threads, and a BLAS that also spawns threads per call oversubscribes the cores."""
    import ctypes
    import glob
    import os

    paths = glob.glob(os.path.join(os.path.dirname(np.__file__), os.pardir, "numpy.libs",
                                   "*openblas*"))
    try:
        with open("/proc/self/maps") as f:
            paths += sorted({ln.split()[-1] for ln in f if "openblas" in ln and "/" in ln})
    except OSError:
        pass
    for path in paths:
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for pre, suf in (("scipy_openblas_", "64_"), ("scipy_openblas_", ""), ("openblas_", "64_"),
                         ("openblas_", "")):
            get = getattr(lib, f"{pre}get_num_threads{suf}", None)
            put = getattr(lib, f"{pre}set_num_threads{suf}", None)
            if get is not None and put is not None:
                get.restype = ctypes.c_int
                put.argtypes = [ctypes.c_int]
                return get, put
    return None


def oracle_attention_threads(q64, hist_k, hist_v, k64, v64, qsl, seq_lens, R, rows,
                             workers=None):
    """The oracle's attention for the flat rows ``rows``: oracle calls on one request's own rows
    each (a mixed step gives each request what it gets alone, a pinned property of the oracle),
    a long request's rows cut into several calls so that the work (rows x keys) spreads over
    every host thread instead of waiting on the few longest requests.  Falls back to one call
    over the whole batch when BLAS cannot be pinned to one thread per call."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    qsl = np.asarray(qsl)
    rows = np.asarray(sorted(set(int(r) for r in rows)), np.int64)
    owner = np.searchsorted(qsl[1:R + 1], rows, side="right")
    blas = _openblas_thread_setters()
    workers = workers or max(1, min(32, len(os.sched_getaffinity(0))))
    if blas is None or workers == 1:
        return paged_attention(q64, hist_k, hist_v, k64, v64, qsl[:R + 1], seq_lens[:R], R,
                               rows=rows.tolist())
    out = np.full_like(q64, np.nan)
    out[int(qsl[R]):] = 0.0

    def one(task):  # rows `sel` of request i, alone (no other request or row changes them)
        _, i, sel = task
        s, e = int(qsl[i]), int(qsl[i + 1])
        res = paged_attention(q64[s:e], [hist_k[i]], [hist_v[i]], k64[s:e], v64[s:e],
                              [0, e - s], [int(seq_lens[i])], 1, rows=(sel - s).tolist())
        out[sel] = res[sel - s]

    # pieces of about a quarter of one thread's share of the rows x keys, longest first
    groups = [(i, rows[owner == i]) for i in np.unique(owner).tolist()]
    total = sum(len(sel) * max(1, int(seq_lens[i])) for i, sel in groups)
    share = max(1.0, total / (4 * workers))
    tasks = []
    for i, sel in groups:
        cost = len(sel) * max(1, int(seq_lens[i]))
        for part in np.array_split(sel, max(1, min(len(sel), math.ceil(cost / share)))):
            tasks.append((len(part) * max(1, int(seq_lens[i])), i, part))
    tasks.sort(key=lambda t: -t[0])
    get, put = blas
    before = get()
    put(1)
    try:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(one, tasks))
    finally:
        put(before)
    return out
