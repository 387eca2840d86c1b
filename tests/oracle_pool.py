"""A spawn-started process pool for the oracle's per-expert rows on K3-sized layers.

Test infrastructure. Each worker regenerates the expert it is asked for from the seeded host
generator and runs oracle.expert_rows on it, so only the z rows and the expert outputs cross
process boundaries. Workers start with single-threaded BLAS (one process per core). The pool
is started with "spawn" (never forked after the GPU was touched)."""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import oracle
import synth

_POOL = None


def _warm(i):
    return i


def _rows_task(d, seed, e, z_bits, actq):
    return oracle.expert_rows(d, synth.host_expert(d, seed, e), z_bits, actq)


def pool() -> ProcessPoolExecutor:
    global _POOL
    if _POOL is None:
        n = os.cpu_count() or 8
        keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
        saved = {k: os.environ.get(k) for k in keys}
        os.environ.update({k: "1" for k in keys})
        try:
            _POOL = ProcessPoolExecutor(n, mp_context=mp.get_context("spawn"))
            list(_POOL.map(_warm, range(4 * n)))  # every worker starts now, with this environment
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
    return _POOL


def rows_fn(d, seed, actq):
    """rows_fn for oracle.Layer.forward_np: expert e's rows for z rows, computed in the pool."""
    p = pool()
    return lambda e, z_rows: p.submit(_rows_task, d, seed, int(e), z_rows, actq).result()


def workers() -> int:
    return os.cpu_count() or 8
