"""The attention oracle over many (sequence, kv head) pairs of a named workload, spread
over a pool of spawned CPU processes.

Each worker regenerates the workload's seeded inputs itself (the generator is
deterministic), runs the float64 oracle on its share of the pairs and returns only
those pairs' output slices, so nothing large crosses process boundaries.  The pool
is started with `spawn`: a worker forked from a process that has used the GPU can
hang.  This module imports no torch and nothing of the CUDA path.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def _job(args):
    name, pairs = args
    import gen
    from gen import inputs as gi
    from oracle import attention as oatt
    w = gen.get(name)
    x = gi.make_inputs(w, with_accept=False)
    dt = w.dtype
    ref = oatt.tree_attention(gi.as_float(x.q, dt), gi.as_float(x.k_pages, dt), gi.as_float(x.v_pages, dt),
                              x.page_table, x.prefix_lens, x.tree_parents, w.page_size, pairs)
    G = w.group
    return [(b, h, ref[b, :, h * G:(h + 1) * G, :].copy()) for b, h in pairs]


def oracle_attention_pairs(name: str, pairs, workers: int) -> np.ndarray:
    """float64 [B][N][Hq][D] with the listed pairs filled in and NaN elsewhere."""
    import gen
    w = gen.get(name)
    pairs = [(int(b), int(h)) for b, h in pairs]
    workers = max(1, min(workers, len(pairs), os.cpu_count() or 1))
    chunks = [pairs[i::workers] for i in range(workers)]
    out = np.full((w.batch, w.num_nodes, w.num_q_heads, w.head_dim), np.nan)
    # one BLAS thread per worker: the workers already use every core
    knobs = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in knobs}
    os.environ.update({k: "1" for k in knobs})
    try:
        with mp.get_context("spawn").Pool(workers) as pool:
            parts = pool.map(_job, [(name, c) for c in chunks if c])
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    for part in parts:
        for b, h, arr in part:
            out[b, :, h * w.group:(h + 1) * w.group, :] = arr
    return out
