"""Inputs for the Monte-Carlo check of the stochastic accept walk.

A fixed vocab-8 tree: a root with three children, each with two children
(N = 10).  The target and draft distributions of a depth-1 node depend only on
that node's token (as they do for a real model, where the next-token
distribution is a function of the context), so the emitted token sequence
must follow p_root(x) * p(y | x) exactly when the walk is lossless -- the
invariance statement of "Tech Radar: SGLang EAGLE-2" section 5 and of the n1n
page's "Mathematical Proof of Lossless Speedup".

Per trial: the children's tokens are drawn i.i.d. from q_root, the
grandchildren's from q(. | parent token), and every node gets a fresh uniform.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

MC_PARENTS = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3], dtype=np.int32)
MC_VOCAB = 8


@dataclass
class MCTables:
    root_logits: np.ndarray     # [V]
    root_q: np.ndarray          # [V]
    d1_logits: np.ndarray       # [V][V]  row x: target logits after token x
    d1_q: np.ndarray            # [V][V]
    d2_logits: np.ndarray       # [V][V]  leaves' rows (never tested, only sampled from)


def mc_tables(seed: int = 0) -> MCTables:
    rng = np.random.default_rng([77, seed])
    V = MC_VOCAB

    def probs(x):
        e = np.exp(x - x.max(axis=-1, keepdims=True))
        return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)

    root_logits = rng.normal(0, 1.5, V).astype(np.float32)
    root_q = probs(root_logits + rng.normal(0, 1.0, V))
    d1_logits = rng.normal(0, 1.5, (V, V)).astype(np.float32)
    d1_q = probs(d1_logits + rng.normal(0, 1.0, (V, V)))
    d2_logits = rng.normal(0, 1.5, (V, V)).astype(np.float32)
    return MCTables(root_logits, root_q, d1_logits, d1_q, d2_logits)


def _draw(rng, probs_rows, n):
    """One categorical draw per row of probs_rows[n][V] (float64 CDF)."""
    cdf = np.cumsum(probs_rows.astype(np.float64), axis=-1)
    u = rng.random(n)[:, None] * cdf[:, -1:]
    return np.minimum((cdf <= u).sum(axis=-1), probs_rows.shape[-1] - 1).astype(np.int32)


def mc_trials(tables: MCTables, trials: int, seed: int = 1):
    """Return (logits[T][N][V], q[T][N][V], tokens[T][N], uniforms[T][N], parents[T][N])."""
    rng = np.random.default_rng([78, seed])
    V, N = MC_VOCAB, len(MC_PARENTS)
    tokens = np.zeros((trials, N), dtype=np.int32)
    for c in (1, 2, 3):
        tokens[:, c] = _draw(rng, np.broadcast_to(tables.root_q, (trials, V)), trials)
    for c in range(4, N):
        parent = MC_PARENTS[c]
        tokens[:, c] = _draw(rng, tables.d1_q[tokens[:, parent]], trials)
    logits = np.empty((trials, N, V), dtype=np.float32)
    q = np.empty((trials, N, V), dtype=np.float32)
    logits[:, 0] = tables.root_logits
    q[:, 0] = tables.root_q
    for c in (1, 2, 3):
        logits[:, c] = tables.d1_logits[tokens[:, c]]
        q[:, c] = tables.d1_q[tokens[:, c]]
    for c in range(4, N):
        logits[:, c] = tables.d2_logits[tokens[:, c]]
        q[:, c] = np.float32(1.0 / V)       # leaves: never used for a test
    uniforms = rng.random((trials, N), dtype=np.float32)
    parents = np.broadcast_to(MC_PARENTS, (trials, N)).copy()
    return logits, q, tokens, uniforms, parents
