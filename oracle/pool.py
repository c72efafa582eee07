"""Run the attention oracle over a process pool (all host cores).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``.  This module holds no
arithmetic of its own: it cuts the output into (head, block of query rows)
units and evaluates each with ``attention.attention_rows`` exactly as it
stands, in worker processes.  Every output element goes through the same
float64 steps as in one process; only the library matmul's internal summation
order may differ with its thread count (differences of about 1e-15).

The pool uses the ``spawn`` start method (safe after the parent process has
initialised CUDA) and one BLAS thread per worker; Q, K and V travel once,
through shared memory.
"""

from __future__ import annotations

import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np

_W: dict = {}


def host_cores() -> int:
    return len(os.sched_getaffinity(0))


def _init(names, shapes, scale):
    try:
        from threadpoolctl import threadpool_limits
        threadpool_limits(1)
    except Exception:
        pass
    _W["shm"] = [shared_memory.SharedMemory(name=n) for n in names]
    _W["arr"] = [np.ndarray(s, dtype=np.float64, buffer=m.buf) for s, m in zip(shapes, _W["shm"])]
    _W["scale"] = scale


def _unit(args):
    from . import attention
    h, rows = args
    q, k, v = _W["arr"]
    return h, rows, attention.attention_rows(q, k, v, _W["scale"], rows, heads=[h])[:, 0, :]


def attention_rows_parallel(q, k, v, scale: float, rows=None, workers: int | None = None,
                            rows_per_unit: int = 1170) -> np.ndarray:
    """``attention.attention_rows(q, k, v, scale, rows)`` for every head, on a
    spawn pool of ``workers`` processes (default: all host cores).  Returns
    [len(rows)][H][D] float64."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    H, D = q.shape[1], q.shape[2]
    out = np.empty((len(rows), H, D), dtype=np.float64)
    units = [(h, rows[i:i + rows_per_unit]) for h in range(H)
             for i in range(0, len(rows), rows_per_unit)]
    workers = max(1, min(workers or host_cores(), len(units)))
    shms = []
    try:
        for a in (q, k, v):
            m = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            np.ndarray(a.shape, dtype=np.float64, buffer=m.buf)[...] = a
            shms.append(m)
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers, initializer=_init,
                      initargs=([m.name for m in shms], [q.shape, k.shape, v.shape], float(scale))) as pool:
            pos = {int(r): i for i, r in enumerate(rows)}
            for h, rs, o in pool.imap_unordered(_unit, units):
                out[[pos[int(r)] for r in rs], h, :] = o
    finally:
        for m in shms:
            m.close()
            m.unlink()
    return out
