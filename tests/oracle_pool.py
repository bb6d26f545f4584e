"""The float64 oracle run in worker processes, one head (or one packed
sequence's head) per task, for the full-output parity tests.

Workers are started with the "spawn" method, so none of them inherits the
parent's CUDA context; each imports only NumPy and the oracle.  A task's
inputs arrive as float32 arrays (exact copies of the bf16 device inputs) and
are converted exactly to float64 by the oracle itself.  Rows are evaluated in
blocks of query rows (each row of the definition depends only on its own
query), which bounds a worker's memory to a few blocks of the score matrix.
"""
from __future__ import annotations

import contextlib
import multiprocessing
import os

import numpy as np

ROW_BLOCK = 2048
_THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def head_ref(task):
    """task = (q, k, v, scale, causal): one head's [N, D] arrays.  Returns the
    oracle's O [N, D] and LSE [N] for every query row."""
    from oracle import attention as ora
    q, k, v, scale, causal = task
    q, k, v = ora.to_f64(q), ora.to_f64(k), ora.to_f64(v)
    n = q.shape[0]
    O = np.empty((n, q.shape[1]))
    L = np.empty(n)
    for r0 in range(0, n, ROW_BLOCK):
        rows = np.arange(r0, min(n, r0 + ROW_BLOCK))
        O[rows], L[rows] = ora.attention_head_ref(q, k, v, scale, causal, rows=rows)
    return O, L


def workers() -> int:
    n = os.cpu_count() or 2
    return max(1, min(8, n // 2))


@contextlib.contextmanager
def pool(processes=None):
    """A spawn-context pool whose workers use two BLAS threads each."""
    processes = processes or workers()
    saved = {k: os.environ.get(k) for k in _THREAD_VARS}
    for k in _THREAD_VARS:
        os.environ[k] = "2"
    try:
        ctx = multiprocessing.get_context("spawn")
        p = ctx.Pool(processes=processes)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    try:
        yield p
    finally:
        p.close()
        p.join()
