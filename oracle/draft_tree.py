"""Draft-tree construction: beam expansion by cumulative confidence, then rerank.
TEST INFRASTRUCTURE ONLY.

"EAGLE-2 & Lookahead Decoding", section 4 ("Dynamic Tree Construction Mechanics"): a draft
path's confidence is the product of its conditional probabilities, so in log space a
node's score is its parent's score plus its own log-probability, and the drafter keeps
expanding only the most confident branches.  The SGLang page ("Speculative Decoding",
EAGLE decoding): each draft step branches every expanded node into its top
`speculative_eagle_topk` tokens, for `speculative_num_steps` steps, and a final rerank keeps
the top `speculative_num_draft_tokens` nodes as the draft tree.

Readings where the pages are silent (the CUDA entry points follow the same ones):
  * node 0 is the root (score 0).  Step s (0-based) expands a frontier of F nodes (the
    root at step 0, F = 1; the k best candidates of step s - 1 after that, F = k): each
    frontier node's children are its top-k tokens by log-probability, ties to the lower
    token id, and every one of the F*k candidates (frontier row f, rank r; candidate
    index f*k + r) becomes a node, in candidate order, from node base(s) = 1 at s = 0 and
    1 + k + (s - 1)*k*k after that.  The next frontier is the k candidates with the
    highest score, ties to the lower candidate index, best first;
  * scores are float32 sums (parent score + log-probability), the precision the kernel
    decides in, so both sides rank identically;
  * the rerank keeps the root and the N - 1 non-root nodes with the highest score, ties
    to the lower node index, numbered in increasing original index (a topological order,
    since a node's parent was added before it).  By default all scored candidates are
    eligible, so a tree may be larger than steps * k nodes; a caller may instead name the
    eligible nodes (a pool), e.g. only the nodes that entered some step's beam -- the
    reading under which a 5-step, top-4 expansion reranks 20 candidates.  A kept node
    whose parent was dropped (only possible with positive log-probabilities, or a pool
    that omits a kept node's parent) is attached to the root and flagged.  A pool with
    fewer than N - 1 eligible nodes gives a smaller tree: its row is padded after the last
    kept node with parent ABSENT (-2) and token -1, the layout of a batch that mixes tree
    sizes.
"""
from __future__ import annotations

import numpy as np

BAD_PARENT = 1
ABSENT = -2       # parent entry of a padding slot after a smaller tree


def step_base(step: int, topk: int) -> int:
    """First node index of a step's candidates."""
    return 1 if step == 0 else 1 + topk + (step - 1) * topk * topk


def num_nodes_after(steps: int, topk: int) -> int:
    return step_base(steps, topk)


def draft_step(logprobs: np.ndarray, frontier: np.ndarray, node_parent: np.ndarray, node_token: np.ndarray,
               node_score: np.ndarray, step: int, topk: int) -> np.ndarray:
    """One expansion step, in place on the node arrays [B][M].  logprobs [B][F][V] float32,
    one row per frontier node in the order of `frontier` [B][F] (ignored at step 0).
    Returns the next frontier [B][k] (node indices, best first)."""
    B, F, V = logprobs.shape
    k = topk
    base = step_base(step, k)
    nxt = np.zeros((B, k), dtype=np.int32)
    for b in range(B):
        if step == 0:
            node_parent[b, 0], node_token[b, 0], node_score[b, 0] = -1, -1, np.float32(0.0)
            front = [0]
        else:
            front = [int(x) for x in frontier[b]]
        assert len(front) == F
        cands = []                                           # (score, candidate index)
        for f, node in enumerate(front):
            row = logprobs[b, f].astype(np.float32)
            order = [int(v) for v in np.lexsort((np.arange(V), -row.astype(np.float64)))[:k]]   # value desc, id asc
            for r, tok in enumerate(order):
                c = f * k + r
                score = np.float32(np.float32(node_score[b, node]) + row[tok])
                node_parent[b, base + c], node_token[b, base + c], node_score[b, base + c] = node, tok, score
                cands.append((score, c))
        cands.sort(key=lambda t: (-float(t[0]), t[1]))
        nxt[b] = [base + c for _s, c in cands[:k]]
    return nxt


def rerank(node_parent: np.ndarray, node_token: np.ndarray, node_score: np.ndarray, num_nodes: int,
           pool: np.ndarray | None = None):
    """Returns (parents [B][N], tokens [B][N], status).  pool [B][P] (node ids) restricts the
    eligible non-root nodes; None makes every node 1 .. M-1 eligible."""
    B, M = node_parent.shape
    N = num_nodes
    parents = np.full((B, N), -1, dtype=np.int32)
    tokens = np.full((B, N), -1, dtype=np.int32)
    status = 0
    for b in range(B):
        eligible = range(1, M) if pool is None else sorted({int(i) for i in pool[b] if 0 < int(i) < M})
        ranked = sorted(eligible, key=lambda i: (-float(np.float32(node_score[b, i])), i))
        kept = sorted(ranked[:N - 1])
        parents[b, 1 + len(kept):] = ABSENT
        new = {0: 0}
        for j, i in enumerate(kept):
            new[i] = j + 1
        tokens[b, 0] = node_token[b, 0]
        for i in kept:
            par = int(node_parent[b, i])
            if par not in new:
                status |= BAD_PARENT
                par = 0
            parents[b, new[i]] = new[par]
            tokens[b, new[i]] = node_token[b, i]
    return parents, tokens, status
