"""Run the row oracle over many query rows on all host cores.

The rows are independent, so they are split over a process pool (``spawn``: a
pool forked after CUDA initialisation can hang).  Each worker memory-maps the
key/value head from a temporary .npy file instead of receiving a copy, and runs
its BLAS on one thread: one process per core already fills the machine, and a
BLAS thread pool per process oversubscribes it (cores x cores threads), which was
more than 20x slower.
"""

import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np

_K = _V = None
_BLAS_THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _init(kpath, vpath):
    global _K, _V
    _K = np.load(kpath, mmap_mode="r")
    _V = np.load(vpath, mmap_mode="r")


def _work(args):
    import oracle
    q_rows, q_pos, causal, scale = args
    return oracle.attention_rows(q_rows, _K, _V, q_positions=q_pos, causal=causal, scale=scale)


def attention_rows_parallel(q_rows, q_pos, k_head, v_head, causal, scale=None, workers=None, chunk=64):
    """oracle.attention_rows over natural-order keys, rows spread over processes."""
    q_rows = np.asarray(q_rows, np.float64)
    q_pos = np.asarray(q_pos, np.int64)
    n = q_rows.shape[0]
    workers = workers or min(16, os.cpu_count() or 1)
    tmp = tempfile.mkdtemp(prefix="ra_oracle_")
    try:
        kpath, vpath = os.path.join(tmp, "k.npy"), os.path.join(tmp, "v.npy")
        np.save(kpath, np.asarray(k_head, np.float32))
        np.save(vpath, np.asarray(v_head, np.float32))
        order = np.argsort(q_pos, kind="stable")
        # interleave sorted rows so every task has a similar key range
        tasks, idx = [], []
        n_tasks = max(1, min(workers * 4, (n + chunk - 1) // chunk))
        for t in range(n_tasks):
            sel = order[t::n_tasks]
            if sel.size:
                tasks.append((q_rows[sel], q_pos[sel], causal, scale))
                idx.append(sel)
        ctx = mp.get_context("spawn")
        # spawned workers read the BLAS thread count from the environment at start-up
        saved = {name: os.environ.get(name) for name in _BLAS_THREAD_VARS}
        os.environ.update({name: "1" for name in _BLAS_THREAD_VARS})
        try:
            with ctx.Pool(workers, initializer=_init, initargs=(kpath, vpath)) as pool:
                res = pool.map(_work, tasks)
        finally:
            for name, val in saved.items():
                if val is None:
                    os.environ.pop(name, None)
                else:
                    os.environ[name] = val
        out = np.zeros((n, q_rows.shape[1]))
        lse = np.full(n, -np.inf)
        for sel, (o, l) in zip(idx, res):
            out[sel] = o
            lse[sel] = l
        return out, lse
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


# ------------------------------------------------------- whole heads in full --

_Q = _O = _L = None


def _init_heads(qpath, kpath, vpath, opath, lpath):
    global _Q, _K, _V, _O, _L
    _Q = np.load(qpath, mmap_mode="r")
    _K = np.load(kpath, mmap_mode="r")
    _V = np.load(vpath, mmap_mode="r")
    _O = np.load(opath, mmap_mode="r+")
    _L = np.load(lpath, mmap_mode="r+")


def _work_heads(args):
    import oracle
    b, h, r0, r1, group, causal, scale, chunk = args
    g = h // group
    o, lse = oracle.attention_rows(_Q[b, h, r0:r1], _K[b, g], _V[b, g],
                                   q_positions=np.arange(r0, r1, dtype=np.int64), causal=causal,
                                   scale=scale, chunk=chunk)
    _O[b, h, r0:r1] = o
    _L[b, h, r0:r1] = lse
    return r1 - r0


def full_attention_parallel(q, k, v, causal, scale=None, workers=None, rows_per_task=1024, chunk=256):
    """oracle.attention_rows over EVERY row of every (batch, query head), spread over processes.

    q [B, Hq, S, d], k/v [B, Hkv, S, d] in natural order (numpy, any float dtype).
    The inputs go to float64 .npy files that the workers memory-map (so the keys
    are converted once, not per row block), and each worker writes its rows of
    O and LSE straight into memory-mapped float64 outputs.  Returns (O, LSE) as
    float64 arrays: exactly what oracle.full_attention returns, row block by row
    block.
    """
    q = np.asarray(q)
    B, Hq, S, d = q.shape
    group = Hq // np.asarray(k).shape[1]
    workers = workers or min(16, os.cpu_count() or 1)
    tmp = tempfile.mkdtemp(prefix="ra_oracle_heads_")
    try:
        paths = [os.path.join(tmp, n + ".npy") for n in ("q", "k", "v", "o", "l")]
        for path, a in zip(paths[:3], (q, k, v)):
            np.save(path, np.asarray(a, np.float64))
        np.lib.format.open_memmap(paths[3], mode="w+", dtype=np.float64, shape=(B, Hq, S, d)).flush()
        np.lib.format.open_memmap(paths[4], mode="w+", dtype=np.float64, shape=(B, Hq, S)).flush()
        tasks = [(b, h, r0, min(S, r0 + rows_per_task), group, bool(causal), scale, chunk)
                 for b in range(B) for h in range(Hq) for r0 in range(0, S, rows_per_task)]
        if causal:  # longest tasks (latest rows) first, so the pool ends evenly
            tasks.sort(key=lambda t: -t[3])
        ctx = mp.get_context("spawn")
        saved = {name: os.environ.get(name) for name in _BLAS_THREAD_VARS}
        os.environ.update({name: "1" for name in _BLAS_THREAD_VARS})
        try:
            with ctx.Pool(workers, initializer=_init_heads, initargs=tuple(paths)) as pool:
                done = sum(pool.imap_unordered(_work_heads, tasks))
        finally:
            for name, val in saved.items():
                if val is None:
                    os.environ.pop(name, None)
                else:
                    os.environ[name] = val
        assert done == B * Hq * S
        return np.array(np.load(paths[3], mmap_mode="r")), np.array(np.load(paths[4], mmap_mode="r"))
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
