"""The oracle's per-head work for the sampled key rows of a long workload,
spread over the host's cores: one (batch, head) slice per task, in worker
processes started with `spawn` (a process forked after CUDA has been
initialised in the parent can hang; a spawned one starts clean).

dK_j and dV_j sum over every query row, so each slice needs the oracle's own
lse and D of all its rows (`oracle.row_stats`) before `oracle.backward_key_rows`
can give the sampled key rows.  Test infrastructure only."""
import multiprocessing as mp
import os

import numpy as np

import oracle


def _key_rows_of_slice(task):
    q, k, v, do, scale, cols, kw = task
    lse, dd = oracle.row_stats(q, k, v, do, scale, rows_per_group=512, **kw)
    dk, dv = oracle.backward_key_rows(q, k, v, do, scale, cols, lse, dd, **kw)
    return lse[0, 0], dk[0, 0], dv[0, 0]


def key_rows_every_head(q, k, v, do, scale, cols, causal=False, kv_len=None, block_mask=None,
                        workers=None):
    """dK and dV of the key rows `cols` [B,H,C] of every (batch, head), and
    the oracle's lse of every query row [B,H,N].  No dropout: its counter
    names the head, which a one-slice task cannot carry."""
    B, H, N, d = q.shape
    tasks = []
    for b in range(B):
        kw = dict(causal=causal, block_mask=block_mask,
                  kv_len=None if kv_len is None else np.asarray(kv_len)[b:b + 1])
        for h in range(H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            tasks.append((np.ascontiguousarray(q[sl]), np.ascontiguousarray(k[sl]),
                          np.ascontiguousarray(v[sl]), np.ascontiguousarray(do[sl]), scale,
                          np.ascontiguousarray(cols[sl]), kw))
    n = workers or max(1, min(len(tasks), os.cpu_count() or 1))
    # one BLAS thread per worker: the workers themselves fill the cores
    saved = {key: os.environ.get(key) for key in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS")}
    os.environ.update(OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1")
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            out = pool.map(_key_rows_of_slice, tasks, chunksize=1)
    finally:
        for key, val in saved.items():
            if val is None:
                os.environ.pop(key, None)
            else:
                os.environ[key] = val
    lse = np.stack([o[0] for o in out]).reshape(B, H, N)
    dk = np.stack([o[1] for o in out]).reshape(B, H, -1, d)
    dv = np.stack([o[2] for o in out]).reshape(B, H, -1, d)
    return lse, dk, dv
