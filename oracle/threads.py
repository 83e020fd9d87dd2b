"""Evaluating the oracle's attention over host threads (oracle; test infrastructure).

No arithmetic of the method lives here: the rows asked for are grouped by request, each
request is handed to the unchanged ``paged_attention`` on its own rows, and the calls run on a
thread pool (numpy releases the GIL inside its loops).  The result of a request's rows does
not depend on the other requests of the batch, a property the oracle's tests pin ("one mixed
step equals each request alone").
"""
from __future__ import annotations

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
    """The oracle's attention for the flat rows ``rows``: one oracle call per request that has
    any, on that request's own rows (a mixed step gives each request what it gets alone, a pinned
    property of the oracle), spread over host threads (numpy releases the GIL inside its loops).
    Falls back to one call over the whole batch when BLAS cannot be pinned to one thread per
    call."""
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

    def one(i):  # request i alone (the oracle's result for a request does not depend on others)
        s, e = int(qsl[i]), int(qsl[i + 1])
        sel = rows[owner == i]
        res = paged_attention(q64[s:e], [hist_k[i]], [hist_v[i]], k64[s:e], v64[s:e],
                              [0, e - s], [int(seq_lens[i])], 1, rows=(sel - s).tolist())
        out[sel] = res[sel - s]

    get, put = blas
    before = get()
    put(1)
    try:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(one, np.unique(owner).tolist()))
    finally:
        put(before)
    return out
