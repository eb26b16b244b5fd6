"""The float64 oracle's dK of selected keys, spread over worker processes.

At the largest workloads one head has 64K-128K query rows, and the gradient
of a key in the first key tile sums over every one of them.  The oracle
(oracle.backward_dk_keys) computes that in minutes on one core; this helper
splits the query rows into blocks and runs the oracle on each block in a
``spawn`` process pool (never forked: a process forked after the first GPU
call can hang), then adds the blocks' contributions.  It adds no arithmetic
of its own beyond that sum.

Why a row block is an exact sub-problem: with the bottom-right causal
reading (query i sees key j iff j <= i + (NK - NQ)), the rows [r0, r1) of
the full problem see only keys [0, r1 + NK - NQ).  The sub-problem with
those rows and those keys has NQ' = r1 - r0 and NK' = r1 + NK - NQ, so its
own offset NK' - NQ' = r0 + NK - NQ reproduces every row's visible set.
Keys that no row of a block sees get no contribution from it.  Without a
causal mask every block keeps all keys.  tests/test_oracle_pool.py checks
the decomposition against one direct oracle call.
"""

import multiprocessing as mp
import os
import tempfile

import numpy as np

_ARR = {}


def _init(paths, threads):
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = str(threads)
    for name, path in paths.items():
        _ARR[name] = np.load(path, mmap_mode="r")


def _block(task):
    import oracle
    r0, r1, scale, causal, mode, scale2 = task
    q1, k1, q2, k2, dkl, keys = (_ARR[n] for n in ("q1", "k1", "q2", "k2", "dkl", "keys"))
    nq, nk = q1.shape[0], k1.shape[0]
    kmax = min(nk, r1 + nk - nq) if causal else nk
    sel = np.nonzero(keys < kmax)[0]
    out = np.zeros((keys.shape[0], (q2 if mode == oracle.MODE_P2 else q1).shape[1]))
    if sel.shape[0] == 0:
        return out
    part = oracle.backward_dk_keys(np.asarray(q1[r0:r1]), np.asarray(k1[:kmax]), np.asarray(q2[r0:r1]),
                                   np.asarray(k2[:kmax]), scale, causal, np.asarray(dkl[r0:r1]), mode,
                                   np.asarray(keys[sel]), row_block=128, scale2=scale2)
    out[sel] = part
    return out


def dk_keys_pooled(q1, k1, q2, k2, scale, causal, dkl, mode, keys, scale2=None, rows_per_task=1024,
                   workers=None):
    """oracle.backward_dk_keys(q1, k1, q2, k2, scale, causal, dkl, mode, keys)
    for one head ([N, d] float64 arrays), computed block by block in a spawn
    pool.  Returns float64 [len(keys), d_g]."""
    keys = np.asarray(keys)
    nq, nk = q1.shape[0], k1.shape[0]
    first = max(0, int(keys.min()) - (nk - nq)) if causal else 0  # rows before it see none of the keys
    tasks = [(r0, min(nq, r0 + rows_per_task), scale, causal, mode, scale2)
             for r0 in range(first - first % rows_per_task, nq, rows_per_task)]
    workers = workers or max(1, min(len(tasks), len(os.sched_getaffinity(0))))
    with tempfile.TemporaryDirectory() as tmp:
        paths = {}
        for name, a in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2), ("dkl", dkl), ("keys", keys)):
            paths[name] = os.path.join(tmp, name + ".npy")
            np.save(paths[name], np.ascontiguousarray(a))
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers, initializer=_init, initargs=(paths, 1)) as pool:
            parts = pool.map(_block, tasks, chunksize=1)
    return np.sum(parts, axis=0)
