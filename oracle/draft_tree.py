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
  * node 0 is the root (score 0); step s (0-based) adds nodes 1 + s*k .. 1 + s*k + k - 1;
    the frontier of step 0 is the root, of step s > 0 the k nodes step s - 1 added;
  * a frontier node's children are its top-k tokens by log-probability, ties to the
    lower token id; of the F*k candidates (frontier f, rank r) the k with the highest
    score are kept, ties to the lower candidate index f*k + r, in descending score order;
  * scores are float32 sums (parent score + log-probability), the precision the kernel
    decides in, so both sides rank identically;
  * the rerank keeps the root and the N - 1 non-root nodes with the highest score, ties
    to the lower node index, numbered in increasing original index (a topological order,
    since a node's parent was added before it).  A kept node whose parent was dropped
    (only possible with positive log-probabilities) is attached to the root and flagged.
"""
from __future__ import annotations

import numpy as np

BAD_PARENT = 1


def draft_step(logprobs: np.ndarray, node_parent: np.ndarray, node_token: np.ndarray, node_score: np.ndarray,
               step: int, topk: int) -> None:
    """One expansion step, in place on the node arrays [B][M].  logprobs [B][F][V] float32,
    one row per frontier node (F = 1 at step 0, else topk)."""
    B, F, V = logprobs.shape
    k = topk
    for b in range(B):
        if step == 0:
            node_parent[b, 0], node_token[b, 0], node_score[b, 0] = -1, -1, np.float32(0.0)
            frontier = [0]
        else:
            frontier = list(range(1 + (step - 1) * k, 1 + step * k))
        assert len(frontier) == F
        cands = []                                           # (score, candidate index, parent node, token)
        for f, node in enumerate(frontier):
            row = logprobs[b, f].astype(np.float32)
            order = sorted(range(V), key=lambda v: (-float(row[v]), v))[:k]
            for r, tok in enumerate(order):
                score = np.float32(np.float32(node_score[b, node]) + row[tok])
                cands.append((score, f * k + r, node, tok))
        cands.sort(key=lambda c: (-float(c[0]), c[1]))
        for r, (score, _ci, node, tok) in enumerate(cands[:k]):
            i = 1 + step * k + r
            node_parent[b, i], node_token[b, i], node_score[b, i] = node, tok, score


def rerank(node_parent: np.ndarray, node_token: np.ndarray, node_score: np.ndarray, num_nodes: int):
    """Returns (parents [B][N], tokens [B][N], status)."""
    B, M = node_parent.shape
    N = num_nodes
    parents = np.full((B, N), -1, dtype=np.int32)
    tokens = np.full((B, N), -1, dtype=np.int32)
    status = 0
    for b in range(B):
        ranked = sorted(range(1, M), key=lambda i: (-float(np.float32(node_score[b, i])), i))
        kept = sorted(ranked[:N - 1])
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
