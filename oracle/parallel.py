"""The oracle's GEMMs run over blocks of output rows in worker processes.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): used by the
``cpu_baseline`` and ``--impl reference`` legs of ``bench.py`` to time the
oracle on every host core, and by the tests that pin it to the serial oracle.

Nothing here adds arithmetic.  An output element C[i, j] of the block-scaled
GEMM depends only on row i of A (with its scales) and row j of B ("Puro-2B:
Poor Lab's Qwen2-1.5B Trained on RTX 5090 within $5090", section 3.2: one
scale per 1x128 group of the reduction dimension, one per 128x128 weight
block), and ``gemm.block_scaled_gemm`` promotes each element over its slices
in the same ascending order whatever rows it is given.  So splitting the
output rows over processes, each running the unchanged oracle function on its
rows, gives the serial result bit for bit.  Quantisation stays in the calling
process (it is a small part of the work).

Processes are started with the ``spawn`` method: a pool forked from a process
that has already used a GPU can hang.
"""

import concurrent.futures as cf
import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np

from . import gemm, quant

_POOL = None
_WORKERS = 0


def workers():
    """Processes the pool uses: every CPU this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def pool():
    """The shared spawn pool (created on first use and kept)."""
    global _POOL, _WORKERS
    if _POOL is None:
        _WORKERS = workers()
        # one BLAS thread per worker process (the workers already fill every
        # core); the variables are read when a worker first loads its BLAS
        keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
        saved = {k: os.environ.get(k) for k in keys}
        os.environ.update({k: "1" for k in keys})
        try:
            _POOL = cf.ProcessPoolExecutor(max_workers=_WORKERS, mp_context=mp.get_context("spawn"))
            list(_POOL.map(_ready, range(_WORKERS)))  # start and import in every worker now
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
    return _POOL


def shutdown():
    global _POOL
    if _POOL is not None:
        _POOL.shutdown()
        _POOL = None


def _ready(_):
    return os.getpid()


def _attach(desc):
    """A read-only numpy view of an operand the parent placed in shared
    memory, and the segment (to close once the view is no longer used)."""
    name, shape, dtype = desc
    shm = shared_memory.SharedMemory(name=name)
    a = np.ndarray(shape, dtype=dtype, buffer=shm.buf)
    a.flags.writeable = False
    return a, shm


def _cols_job(fn_name, descs, rows, cols):
    views = [_attach(d) for d in descs]
    try:
        acc, out = getattr(gemm, fn_name)(*[v for v, _ in views], rows=rows, cols=cols)
        return np.array(acc), np.array(out)  # copies: nothing refers to the segments afterwards
    finally:
        for _, shm in views:
            shm.close()


def gemm_rows(fn_name, A, sa, B, sb, rows=None, cols=None):
    """gemm.<fn_name>(A, sa, B, sb, rows, cols) computed as one block of
    output rows or columns per worker, whichever operand is larger being the
    one split (each worker decodes only its block of it); returns (acc, out)
    exactly as the serial call does.  The operands reach the workers through
    shared memory (one copy in all), not pickled once per worker."""
    p = pool()
    ops = [np.ascontiguousarray(x) for x in (A, sa, B, sb)]
    rows = np.arange(ops[0].shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(ops[2].shape[0]) if cols is None else np.asarray(cols)
    by_rows = len(rows) > len(cols)
    split = rows if by_rows else cols
    blocks = [b for b in np.array_split(split, min(len(split), _WORKERS)) if len(b)]
    segs = []
    try:
        descs = []
        for x in ops:
            shm = shared_memory.SharedMemory(create=True, size=max(x.nbytes, 1))
            segs.append(shm)
            np.ndarray(x.shape, dtype=x.dtype, buffer=shm.buf)[...] = x
            descs.append((shm.name, x.shape, x.dtype.str))
        futs = [p.submit(_cols_job, fn_name, descs, b if by_rows else rows, cols if by_rows else b) for b in blocks]
        parts = [f.result() for f in futs]
    finally:
        for shm in segs:
            shm.close()
            shm.unlink()
    join = np.vstack if by_rows else np.hstack
    return join([a for a, _ in parts]), join([o for _, o in parts])


def _blocks(n, unit):
    """Index blocks of [0, n) in whole units (128-value groups), one per worker."""
    pool()
    groups = np.array_split(np.arange(n // unit), min(n // unit, _WORKERS))
    return [slice(int(g[0]) * unit, (int(g[-1]) + 1) * unit) for g in groups if len(g)]


def _act_rows_job(x, scale_mode):
    return quant.quantize_act_1x128(x, scale_mode)


def _act_tokens_job(x, scale_mode):
    return quant.quantize_act_tokens_1x128(x, scale_mode)


def _w_job(w, scale_mode):
    return quant.quantize_w_128x128(w, scale_mode)


def quantize_act_1x128(x, scale_mode="amax448"):
    """quant.quantize_act_1x128 over blocks of rows (each row's groups are its
    own): q [M, K] and s [K/128, M]."""
    x = np.asarray(x)
    parts = [f.result() for f in [pool().submit(_act_rows_job, np.ascontiguousarray(x[b]), scale_mode)
                                  for b in _blocks(x.shape[0], 128)]]
    return np.vstack([q for q, _ in parts]), np.hstack([s for _, s in parts])


def quantize_act_tokens_1x128(x, scale_mode="amax448"):
    """quant.quantize_act_tokens_1x128 over blocks of 128 columns (each
    column's token groups are its own): qT [K, M] and sT [M/128, K]."""
    x = np.asarray(x)
    parts = [f.result() for f in [pool().submit(_act_tokens_job, np.ascontiguousarray(x[:, b]), scale_mode)
                                  for b in _blocks(x.shape[1], 128)]]
    return np.vstack([q for q, _ in parts]), np.hstack([s for _, s in parts])


def quantize_w_128x128(w, scale_mode="amax448"):
    """quant.quantize_w_128x128 over blocks of 128 rows (whole 128x128
    blocks): Wq [N, K], WqT [K, N] and sW [N/128, K/128]."""
    w = np.asarray(w)
    parts = [f.result() for f in [pool().submit(_w_job, np.ascontiguousarray(w[b]), scale_mode)
                                  for b in _blocks(w.shape[0], 128)]]
    return (np.vstack([q for q, _, _ in parts]), np.hstack([qt for _, qt, _ in parts]),
            np.vstack([s for _, _, s in parts]))


def linear_fwd(X, W, scale_mode="amax448"):
    """gemm.linear_fwd with its quantisers and FPROP GEMM spread over the pool."""
    Wq, WqT, sW = quantize_w_128x128(W, scale_mode)
    Xq, sX = quantize_act_1x128(X, scale_mode)
    XqT, sXT = quantize_act_tokens_1x128(X, scale_mode)
    _, Y = gemm_rows("fprop", Xq, sX, Wq, sW)
    saved = dict(Wq=Wq, WqT=WqT, sW=sW, Xq=Xq, sX=sX, XqT=XqT, sXT=sXT)
    return Y, saved


def linear_bwd(dY, saved, scale_mode="amax448"):
    """gemm.linear_bwd (bf16 dW) with its quantisers, DGRAD and WGRAD spread
    over the pool (WGRAD by columns of dW: each keeps its whole reduction over
    tokens)."""
    dYq, sdY = quantize_act_1x128(dY, scale_mode)
    dYqT, sdYT = quantize_act_tokens_1x128(dY, scale_mode)
    _, dX = gemm_rows("dgrad", dYq, sdY, saved["WqT"], saved["sW"])
    _, dW = gemm_rows("wgrad", dYqT, sdYT, saved["XqT"], saved["sXT"])
    return dX, dW
