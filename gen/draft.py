"""Seeded stand-ins for the draft model's next-token log-probabilities (no method arithmetic:
random probability vectors and their logarithms)."""
from __future__ import annotations

import numpy as np


def draft_logprobs(seed: int, batch: int, frontier: int, vocab: int, concentration: float = 0.3,
                   ties: bool = False) -> np.ndarray:
    """[batch][frontier][vocab] float32 log-probabilities of Dirichlet(concentration) vectors;
    with ties=True the values are rounded to halves so many of them are equal."""
    rng = np.random.default_rng(seed)
    g = rng.gamma(concentration, size=(batch, frontier, vocab))
    p = g / g.sum(axis=-1, keepdims=True)
    lp = np.log(np.maximum(p, 1e-38)).astype(np.float32)
    if ties:
        lp = (np.round(lp * 2) / 2).astype(np.float32)
    return lp
