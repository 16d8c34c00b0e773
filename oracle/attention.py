"""Tree attention over a paged KV cache, float64, by definition.

What is computed (the verification pass of "Tech Radar: SGLang EAGLE-2",
section 2, and of "EAGLE-2 & Lookahead Decoding", section 4 "Tree Attention
Masking and Target Verification"): the draft tree is flattened after the
cached prefix and verified in one pass ("Speculative Decoding in Production:
EAGLE-3 Dynamic Trees", section "From Linear Sequences to Dynamic Draft
Trees").  The query of node i, head hq, attends to

    T_i = {0 .. S-1}  U  {S + j : j in Ancestors(i) U {i}}

where S is the sequence's prefix length and the N tree tokens occupy logical
positions S .. S+N-1 in node order.  A tree padded to the batch's node count
(tree_mask.ABSENT entries) has N_b = tree_size nodes: its sequence is S + N_b
tokens long and the rows of the padding slots are zero.  With h = hq // (Hq/Hkv) its kv head,

    s_t = q . K[t, h] / sqrt(D),   w = softmax(s over T_i),   out = sum_t w_t V[t, h].

Readings where the pages are silent: scale 1/sqrt(D); GQA maps q head hq to kv
head hq // G; logical token t lives in physical page page_table[b][t // ps],
slot t % ps; page layout [P][ps][Hkv][D].
"""
from __future__ import annotations

import math
from typing import Iterable, Optional

import numpy as np

from .tree_mask import mask_matrix, tree_size


def gather_kv(pages, page_table_row, length: int, page_size: int, h: int) -> np.ndarray:
    """Logical tokens 0..length-1 of kv head h, float64 [length][D]."""
    t = np.arange(length)
    phys = np.asarray(page_table_row)[t // page_size]
    return np.asarray(pages[phys, t % page_size, h, :], dtype=np.float64)


def attend_one(q_vec, K, V, allowed) -> np.ndarray:
    """softmax(q.K[allowed]^T / sqrt(D)) @ V[allowed] for one query, float64."""
    q_vec = np.asarray(q_vec, dtype=np.float64)
    s = K[allowed] @ q_vec / math.sqrt(q_vec.shape[-1])
    w = np.exp(s - s.max())
    w /= w.sum()
    return w @ V[allowed]


def tree_attention_head(q_bh, K, V, prefix_len: int, parents) -> np.ndarray:
    """Output of one (sequence, kv head): q_bh [N][G][D] -> [N][G][D] float64.

    K, V are that sequence's logical tokens [S+N][D] for this kv head.
    """
    n = len(parents)
    m = mask_matrix(parents)
    out = np.empty(q_bh.shape, dtype=np.float64)
    for i in range(n):
        allowed = np.concatenate([np.arange(prefix_len), prefix_len + np.flatnonzero(m[i])])
        for g in range(q_bh.shape[1]):
            out[i, g] = attend_one(q_bh[i, g], K, V, allowed)
    return out


def tree_attention(q, k_pages, v_pages, page_table, prefix_lens, tree_parents,
                   page_size: int,
                   pairs: Optional[Iterable[tuple[int, int]]] = None) -> np.ndarray:
    """Tree attention for a batch.

    q [B][N][Hq][D], k_pages/v_pages [P][ps][Hkv][D] (float values of any
    precision, widened exactly to float64), page_table [B][max_pages],
    prefix_lens [B], tree_parents [B][N] (rows may be padded with ABSENT).
    Returns float64 [B][N][Hq][D].
    `pairs` restricts the work to the listed (b, kv head) pairs; other entries
    of the result are NaN.
    """
    B, N, Hq, D = q.shape
    Hkv = k_pages.shape[2]
    G = Hq // Hkv
    out = np.full((B, N, Hq, D), np.nan, dtype=np.float64)
    if pairs is None:
        pairs = [(b, h) for b in range(B) for h in range(Hkv)]
    for b, h in pairs:
        S = int(prefix_lens[b])
        nb = tree_size(tree_parents[b])
        K = gather_kv(k_pages, page_table[b], S + nb, page_size, h)
        V = gather_kv(v_pages, page_table[b], S + nb, page_size, h)
        q_bh = np.asarray(q[b, :nb, h * G:(h + 1) * G, :], dtype=np.float64)
        out[b, :nb, h * G:(h + 1) * G, :] = tree_attention_head(q_bh, K, V, S, tree_parents[b][:nb])
        out[b, nb:, h * G:(h + 1) * G, :] = 0.0
    return out
