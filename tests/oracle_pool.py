"""Runs the fp64 oracle's backward over token ranges in a pool of processes (spawned, so
no CUDA context is inherited), for the checks at the full 64k-token batch that the oracle
would take minutes to finish on one core.  The fp64 hidden and head matrices live in
shared memory (one copy for all workers); each worker calls oracle.head_backward on its
token range and returns its partial sums of the selected dW rows, which the caller adds
in range order.  No tests here."""
import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np

_W = {}


def _attach(name, shape):
    shm = shared_memory.SharedMemory(name=name)
    _W.setdefault("shm", []).append(shm)
    return np.ndarray(shape, dtype=np.float64, buffer=shm.buf)


def _init(xname, xshape, wname, wshape, small, op, dloss, vrows):
    _W["inputs"] = dict(small, hidden=_attach(xname, xshape), W=_attach(wname, wshape))
    _W["op"], _W["dloss"], _W["vrows"] = op, dloss, vrows


def _work(rng):
    import oracle
    t0, t1 = rng
    _, dW, bnd = oracle.head_backward(_W["inputs"], _W["op"], _W["dloss"], rows=np.arange(t0, t1), chunk=64,
                                      want_dX=False, want_bounds=True, vrows=_W["vrows"])
    return t0, dW, bnd["W"], bnd["zW"]


def dW_rows(inputs: dict, op, dloss, vrows, workers=None, span=1024, timeout_s=1800):
    """Selected rows of the oracle's dW over the whole batch, with their bounds (the
    oracle's head_backward, split by token ranges of `span` and summed in range order).
    Raises if the pool has not finished within timeout_s (a pool whose workers cannot
    start would otherwise wait forever)."""
    workers = workers or max(1, min(32, os.cpu_count() or 1))
    X = np.ascontiguousarray(inputs["hidden"], dtype=np.float64)
    W = np.ascontiguousarray(inputs["W"], dtype=np.float64)
    shms = []
    try:
        views = []
        for a in (X, W):
            shm = shared_memory.SharedMemory(create=True, size=a.nbytes)
            shms.append(shm)
            v = np.ndarray(a.shape, dtype=np.float64, buffer=shm.buf)
            v[...] = a
            views.append(v)
        small = {k: v for k, v in inputs.items() if k not in ("hidden", "W")}
        N = X.shape[0]
        ranges = [(t, min(N, t + span)) for t in range(0, N, span)]
        env = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in env:
            os.environ[k] = "1"             # one BLAS thread per worker process
        try:
            ctx = mp.get_context("spawn")
            with ctx.Pool(workers, initializer=_init,
                          initargs=(shms[0].name, X.shape, shms[1].name, W.shape, small, op,
                                    np.asarray(dloss, np.float64), np.asarray(vrows, np.int64))) as pool:
                parts = sorted(pool.map_async(_work, ranges, chunksize=1).get(timeout_s), key=lambda r: r[0])
        finally:
            for k, v in env.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        dW = np.zeros((len(vrows), X.shape[1]))
        bW = np.zeros_like(dW)
        zW = np.zeros_like(dW)
        for _, d, b, z in parts:
            dW += d
            bW += b
            zW += z
        return dW, {"W": bW, "zW": zW}
    finally:
        for shm in shms:
            shm.close()
            shm.unlink()
