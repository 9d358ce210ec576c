"""A spawn-started process pool that runs oracle functions for the full-size
parity checks (test infrastructure).

Each job is one q head (or one q head's key-column tail) handed to the
oracle as it stands; the pool only spreads independent heads over the host's
cores.  The pool is started with `spawn`, never `fork`, because the parent
has already used the GPU.  BLAS threads per worker are set so that workers x
threads matches the cores this process may use.
"""
import multiprocessing as mp
import os

import numpy as np

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def head_fwd_bwd(job):
    """Forward and backward of one q head against its kv head: q, do [S, D];
    k, v [S, D].  Returns O, LSE, dQ of the head and its contribution to the
    kv head's dK, dV (the caller sums the G heads of a group)."""
    import oracle
    q, k, v, do, cu, causal = job
    o, lse = oracle.attn_fwd(q[None], k[None], v[None], cu, causal)
    dq, dk, dv = oracle.attn_bwd(q[None], k[None], v[None], do[None], cu, causal)
    return o[0], lse[0], dq[0], dk[0], dv[0]


def head_rows(job):
    """O, LSE and dQ of selected rows of one q head (oracle.attn_rows)."""
    import oracle
    q_rows, k, v, do_rows, rows, cu, causal = job
    return oracle.attn_rows(q_rows, k, v, do_rows, rows, cu, causal)


def head_kv_tail(job):
    """One q head's contribution to dK, dV of key columns [j0, S)
    (oracle.attn_kv_tail); q and dO are given for rows >= j0 only."""
    import oracle
    q_tail, k, v, do_tail, j0, cu, causal, row_block = job
    k, v = k.astype(np.float64), v.astype(np.float64)   # once, not per row block
    S, D = k.shape
    q = np.zeros((1, S, D), dtype=q_tail.dtype)      # rows < j0 are never read
    do = np.zeros((1, S, D), dtype=do_tail.dtype)
    q[0, j0:] = q_tail
    do[0, j0:] = do_tail
    return oracle.attn_kv_tail(q, k, v, do, j0, cu, causal, row_block=row_block)


def run(fn, jobs, max_workers=None):
    """pool.map(fn, jobs) over spawn-started workers, results in job order."""
    if not jobs:
        return []
    cores = len(os.sched_getaffinity(0))
    n = max(1, min(len(jobs), cores, max_workers or cores))
    threads = max(1, cores // n)
    saved = {k: os.environ.get(k) for k in _THREAD_VARS}
    os.environ.update({k: str(threads) for k in _THREAD_VARS})
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            return pool.map(fn, jobs, chunksize=1)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
