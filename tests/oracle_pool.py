"""Every-element comparison of a full-size CUDA result with the FP64 oracle,
one (batch or sequence, query head) per task, spread over the host cores.

The pool is started with the "spawn" method (a child forked from a process
that has used the GPU can hang).  Each worker runs single-threaded BLAS and
computes its head's oracle rows in chunks (bounded memory), then compares
them with the GPU rows it was handed and returns only the error figures.
Test infrastructure: only tests/ and the benchmark's correctness gate use it.
"""

from __future__ import annotations

import multiprocessing as mp
import os
from contextlib import contextmanager

import numpy as np

ROW_CHUNK = 1024
_THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _compare_head(task):
    """task = (key, q [Lq, D], k [Lk, D], v [Lk, D], o_gpu [Lq, D], lse_gpu [Lq], rows or None, kw).
    Returns (key, max|dO|, max|dlse|, |O_ref| at the worst element, row of the worst element)."""
    import oracle
    key, q, k, v, go, gl, rows, kw = task
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    worst_o = worst_l = 0.0
    at_o, at_row = 0.0, -1
    for c0 in range(0, len(rows), ROW_CHUNK):
        r = rows[c0:c0 + ROW_CHUNK]
        ro, rl = oracle.attention_rows(q, k, v, r, **kw)
        g_o = go[c0:c0 + ROW_CHUNK]
        g_l = gl[c0:c0 + ROW_CHUNK]
        err = np.abs(g_o - ro)
        if err.size and float(err.max()) > worst_o:
            i = np.unravel_index(int(err.argmax()), err.shape)
            worst_o, at_o, at_row = float(err[i]), float(abs(ro[i])), int(r[i[0]])
        fin = np.isfinite(rl)
        # rows without an eligible key must give exactly O = 0 and lse = -inf
        if not np.array_equal(np.isfinite(g_l), fin):
            return key, float("inf"), float("inf"), 0.0, -1
        if (~fin).any() and (np.any(g_o[~fin] != 0.0) or np.any(g_l[~fin] != -np.inf)):
            return key, float("inf"), float("inf"), 0.0, -1
        if fin.any():
            worst_l = max(worst_l, float(np.max(np.abs(g_l[fin] - rl[fin]))))
    return key, worst_o, worst_l, at_o, at_row


@contextmanager
def spawn_pool(workers=None):
    workers = workers or len(os.sched_getaffinity(0))
    saved = {v: os.environ.get(v) for v in _THREAD_VARS}
    for v in _THREAD_VARS:
        os.environ[v] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers) as pool:
            yield pool
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old


def _f64(t):
    return t.float().double().numpy()


def head_tasks(w, inp, o, lse, rows_of=None):
    """Tasks for every (batch or sequence, query head) of a workload.  o, lse
    are CPU tensors in the workload's layout ([B,H,N,D] view or packed
    [T,H,D] / [H,T]).  rows_of(L) may pick the rows to compare (default all)."""
    group = w.Hq // w.Hkv
    kw = dict(causal=w.causal, scale=w.scale, window_left=w.window_left, window_right=w.window_right,
              num_global=w.num_global)
    if w.layout == "varlen":
        cu = inp["cu_seqlens"].tolist()
        cuk = inp["cu_seqlens_k"].tolist() if "cu_seqlens_k" in inp else cu
        for s in range(len(cu) - 1):
            t0, t1, k0, k1 = cu[s], cu[s + 1], cuk[s], cuk[s + 1]
            if t1 == t0:
                continue
            rows = None if rows_of is None else rows_of(t1 - t0)
            sel = slice(None) if rows is None else rows
            for h in range(w.Hq):
                hk = h // group
                yield ((s, h), _f64(inp["q"][t0:t1, h]), _f64(inp["k"][k0:k1, hk]), _f64(inp["v"][k0:k1, hk]),
                       _f64(o[t0:t1, h][sel]), _f64(lse[h, t0:t1][sel]), rows, kw)
    else:
        for b in range(w.B):
            rows = None if rows_of is None else rows_of(w.N)
            sel = slice(None) if rows is None else rows
            for h in range(w.Hq):
                hk = h // group
                yield ((b, h), _f64(inp["q"][b, h]), _f64(inp["k"][b, hk]), _f64(inp["v"][b, hk]),
                       _f64(o[b, h][sel]), _f64(lse[b, h][sel]), rows, kw)


def compare_workload(w, inp, o, lse, rows_of=None, pool=None):
    """Max |dO| and |dlse| over every compared element, with where the worst
    O error sits.  Returns a dict."""
    tasks = head_tasks(w, inp, o, lse, rows_of)
    if pool is None:
        with spawn_pool() as p:
            results = list(p.imap_unordered(_compare_head, tasks, chunksize=1))
    else:
        results = list(pool.imap_unordered(_compare_head, tasks, chunksize=1))
    worst = max(results, key=lambda r: r[1])
    return {"max_abs_dO": max(r[1] for r in results), "max_abs_dlse": max(r[2] for r in results),
            "worst_head": list(worst[0]), "worst_row": worst[4], "abs_O_ref_at_worst": worst[3],
            "heads": len(results)}


def stratified_rows(L, edge=256, tile=128):
    """The first and last `edge` rows of a sequence and both rows at every
    `tile`-row boundary."""
    rows = set(range(min(edge, L))) | set(range(max(0, L - edge), L))
    for b in range(tile, L, tile):
        rows.update((b - 1, b))
    return np.array(sorted(rows), dtype=np.int64)
