"""Seeded synthetic inputs for the tree-verify path.

Every array is drawn from `numpy.random.default_rng([cfg_id, b, stream])`, one
stream per quantity and sequence, so any sequence can be regenerated on its
own and the CPU oracle and the GPU path always see identical bytes.

Streams: tree=0, q=1, k=2, v=3, logits=4, noise=5, tokens=6, uniforms=7,
pages=8, prefix=9.

bf16 tensors are carried as uint16 bit patterns, rounded to nearest-even from
fp32 draws; `bf16_bits_to_f32` widens them exactly.  Unused page slots and
spare pool pages hold NaN, so a stray read shows up in the output instead of
passing silently.

This module computes nothing of the method itself.  The draft tokens and the
draft distribution q are inputs (they come from the drafter, not from the
verifier); to make them realistic they are derived from the target logits
with numpy's argmax / a softmax of noisy logits.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass
from typing import Optional

import numpy as np

from . import trees
from .configs import Workload

TREE, Q, K, V, LOGITS, NOISE, TOKENS, UNIFORMS, PAGES, PREFIX = range(10)
BF16_NAN = np.uint16(0x7FC0)


def rng_for(w: Workload, b: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([w.cfg_id, b, stream])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit pattern (inputs hold no NaN)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def as_float(x: np.ndarray, dtype: str) -> np.ndarray:
    """View a stored tensor (fp32, or bf16 bits) as exact fp32 values."""
    return bf16_bits_to_f32(x) if dtype == "bf16" else x


@dataclass
class TreeInputs:
    workload: Workload
    q: np.ndarray                  # [B][N][Hq][D]   f32 or bf16 bits
    k_pages: np.ndarray            # [P][ps][Hkv][D] f32 or bf16 bits
    v_pages: np.ndarray
    page_table: np.ndarray         # [B][max_pages] int32
    prefix_lens: np.ndarray        # [B] int32
    tree_parents: np.ndarray       # [B][N] int32
    target_logits: np.ndarray      # [B][N][V] f32
    draft_tokens: np.ndarray       # [B][N] int32
    draft_probs: Optional[np.ndarray]  # [B][N][V] f32 (stochastic only)
    uniforms: Optional[np.ndarray]     # [B][N] f32 (stochastic only)

    @property
    def temperature(self) -> float:
        return self.workload.temperature

    @property
    def num_pool_pages(self) -> int:
        return self.k_pages.shape[0]


def _pool(workers: Optional[int]) -> ThreadPoolExecutor:
    return ThreadPoolExecutor(max_workers=workers or min(32, os.cpu_count() or 1))


def _draw_kv(w: Workload, b: int, stream: int, ntok: int) -> np.ndarray:
    x = rng_for(w, b, stream).standard_normal(
        (ntok, w.num_kv_heads, w.head_dim), dtype=np.float32)
    return f32_to_bf16_bits(x) if w.dtype == "bf16" else x


def _softmax_rows(x: np.ndarray) -> np.ndarray:
    m = x.max(axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=-1, keepdims=True)


def _greedy_tokens(rng, parents, logits, vocab):
    """Parent's argmax with prob. 0.7, else uniform; siblings kept distinct."""
    n = len(parents)
    tok = np.zeros(n, dtype=np.int32)
    used: dict[int, set] = {}
    for c in range(1, n):
        p = int(parents[c])
        seen = used.setdefault(p, set())
        if rng.random() < 0.7:
            x = int(np.argmax(logits[p]))
        else:
            x = int(rng.integers(0, vocab))
        while x in seen:
            x = int(rng.integers(0, vocab))
        seen.add(x)
        tok[c] = x
    return tok


def _sampled_tokens(rng, parents, q):
    n = len(parents)
    tok = np.zeros(n, dtype=np.int32)
    for c in range(1, n):
        row = q[int(parents[c])].astype(np.float64)
        cdf = np.cumsum(row)
        x = int(np.searchsorted(cdf, rng.random() * cdf[-1], side="right"))
        tok[c] = min(x, len(row) - 1)
    return tok


def make_inputs(w: Workload, *, parents: Optional[np.ndarray] = None,
                prefix_lens: Optional[np.ndarray] = None,
                with_accept: bool = True, with_attention: bool = True,
                workers: Optional[int] = None, spare_pages: int = 2) -> TreeInputs:
    """Build the full input set of workload `w`.

    parents / prefix_lens override the recipe (shape [B][N] / [B]) for edge
    cases; with_accept=False skips the vocab-sized arrays and
    with_attention=False the KV pool (left as a single poisoned page).
    """
    B, N = w.batch, w.num_nodes
    ps, Hkv, D = w.page_size, w.num_kv_heads, w.head_dim
    if prefix_lens is None:
        if w.prefix_lo == w.prefix_hi:
            prefix_lens = np.full(B, w.prefix_lo, dtype=np.int32)
        else:
            prefix_lens = np.array(
                [rng_for(w, b, PREFIX).integers(w.prefix_lo, w.prefix_hi + 1) for b in range(B)],
                dtype=np.int32)
    prefix_lens = np.asarray(prefix_lens, dtype=np.int32)
    if parents is None:
        parents = np.stack([
            trees.build_tree(rng_for(w, b if w.vary_tree else 0, TREE), w.num_steps, w.topk, N)
            for b in range(B)])
    parents = np.asarray(parents, dtype=np.int32).reshape(B, N)

    ntok = prefix_lens + N
    npages = (ntok + ps - 1) // ps
    max_pages = int(npages.max())
    used = int(npages.sum())
    pool_pages = used + spare_pages
    if w.shuffle_pages:
        perm = np.random.default_rng([w.cfg_id, B, PAGES]).permutation(used).astype(np.int32)
    else:
        perm = np.arange(used, dtype=np.int32)
    page_table = np.full((B, max_pages), used, dtype=np.int32)   # unused -> a NaN spare page
    starts = np.concatenate([[0], np.cumsum(npages)[:-1]])
    for b in range(B):
        page_table[b, : npages[b]] = perm[starts[b]: starts[b] + npages[b]]

    store = np.uint16 if w.dtype == "bf16" else np.float32
    poison = BF16_NAN if w.dtype == "bf16" else np.float32(np.nan)
    if not with_attention:
        pool_pages = 1
        page_table[:] = 0
    k_pages = np.empty((pool_pages, ps, Hkv, D), dtype=store)
    v_pages = np.empty((pool_pages, ps, Hkv, D), dtype=store)

    def fill(args):
        b, stream, dst = args
        vals = _draw_kv(w, b, stream, int(ntok[b]))
        flat = np.full((npages[b] * ps, Hkv, D), poison, dtype=store)
        flat[: ntok[b]] = vals
        dst[page_table[b, : npages[b]]] = flat.reshape(npages[b], ps, Hkv, D)

    if with_attention:
        with _pool(workers) as ex:
            list(ex.map(fill, [(b, s, d) for b in range(B) for s, d in ((K, k_pages), (V, v_pages))]))
        k_pages[used:] = poison
        v_pages[used:] = poison
    else:
        k_pages[:] = poison
        v_pages[:] = poison

    def draw_q(b):
        x = rng_for(w, b, Q).standard_normal((N, w.num_q_heads, D), dtype=np.float32)
        return f32_to_bf16_bits(x) if w.dtype == "bf16" else x

    with _pool(workers) as ex:
        q = np.stack(list(ex.map(draw_q, range(B))))

    logits = tokens = probs = unif = None
    if with_accept:
        Vv = w.vocab
        logits = np.empty((B, N, Vv), dtype=np.float32)
        tokens = np.empty((B, N), dtype=np.int32)
        probs = None if w.greedy else np.empty((B, N, Vv), dtype=np.float32)
        unif = None if w.greedy else np.empty((B, N), dtype=np.float32)

        def draw_accept(b):
            lg = rng_for(w, b, LOGITS).standard_normal((N, Vv), dtype=np.float32)
            lg *= np.float32(w.logit_std)
            logits[b] = lg
            trng = rng_for(w, b, TOKENS)
            if w.greedy:
                tokens[b] = _greedy_tokens(trng, parents[b], lg, Vv)
            else:
                noise = rng_for(w, b, NOISE).standard_normal((N, Vv), dtype=np.float32)
                qb = _softmax_rows((lg.astype(np.float64) + noise) / w.temperature)
                probs[b] = qb.astype(np.float32)
                tokens[b] = _sampled_tokens(trng, parents[b], probs[b])
                unif[b] = rng_for(w, b, UNIFORMS).random(N, dtype=np.float32)

        with _pool(workers) as ex:
            list(ex.map(draw_accept, range(B)))

    return TreeInputs(w, q, k_pages, v_pages, page_table, prefix_lens, parents,
                      logits, tokens, probs, unif)
