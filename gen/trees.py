"""Seeded draft-tree shapes.

A tree is produced the way the SGLang docs ("Speculative Decoding", section
"References") describe EAGLE-2 drafting: expand the tree step by step with
`topk` children per expanded node, keep a beam of the `topk` most probable
nodes by cumulative log-probability, and finally rerank the candidates to the
`num_draft_tokens - 1` best, which together with the root form the verified
tree.  The draft model's log-probabilities are synthetic: the sorted top-k of
a log-softmax over 64 i.i.d. N(0, 2^2) values.  Only the tree shape (a parent
array) leaves this module; it is input data for both the kernels and the
oracle.

Node order: root first, then by (depth, creation order), so parent[i] < i.
"""
from __future__ import annotations

import numpy as np


def _child_logprobs(rng: np.random.Generator, topk: int) -> np.ndarray:
    x = rng.normal(0.0, 2.0, 64)
    lp = x - (np.log(np.sum(np.exp(x - x.max()))) + x.max())
    return np.sort(lp)[::-1][:topk]


def build_tree(rng: np.random.Generator, num_steps: int, topk: int,
               num_nodes: int) -> np.ndarray:
    """Return parents[num_nodes] (int32, parents[0] = -1) of a reranked draft tree."""
    if num_nodes < 1:
        raise ValueError("num_nodes must be >= 1")
    # candidate record: (cum_logprob, depth, creation_id, parent_creation_id)
    cands: list[tuple[float, int, int, int]] = []
    beam_nodes: list[int] = []          # creation ids that were in some beam
    beam: list[int] = []
    for lp in _child_logprobs(rng, topk):
        cid = len(cands)
        cands.append((float(lp), 1, cid, -1))
        beam.append(cid)
    beam_nodes.extend(beam)
    for step in range(2, num_steps + 1):
        expanded = []
        for pid in beam:
            for lp in _child_logprobs(rng, topk):
                cid = len(cands)
                cands.append((cands[pid][0] + float(lp), step, cid, pid))
                expanded.append(cid)
        expanded.sort(key=lambda c: (-cands[c][0], cands[c][2]))
        beam = expanded[:topk]
        beam_nodes.extend(beam)
    if num_steps * topk >= num_nodes - 1:
        pool = beam_nodes
    else:
        pool = list(range(len(cands)))
    if len(pool) < num_nodes - 1:
        raise ValueError("tree recipe yields fewer candidates than num_nodes - 1")
    ranked = sorted(pool, key=lambda c: (-cands[c][0], cands[c][1], cands[c][2]))
    kept = sorted(ranked[: num_nodes - 1], key=lambda c: (cands[c][1], cands[c][2]))
    index = {cid: i + 1 for i, cid in enumerate(kept)}
    parents = np.full(num_nodes, -1, dtype=np.int32)
    for cid in kept:
        pc = cands[cid][3]
        parents[index[cid]] = 0 if pc < 0 else index[pc]
    return parents


def chain(num_nodes: int) -> np.ndarray:
    p = np.arange(-1, num_nodes - 1, dtype=np.int32)
    return p


def star(num_nodes: int) -> np.ndarray:
    p = np.zeros(num_nodes, dtype=np.int32)
    p[0] = -1
    return p


def random_recursive(rng: np.random.Generator, num_nodes: int) -> np.ndarray:
    """parents[i] uniform in [0, i): any topologically ordered tree shape."""
    p = np.empty(num_nodes, dtype=np.int32)
    p[0] = -1
    for i in range(1, num_nodes):
        p[i] = rng.integers(0, i)
    return p


def depths(parents: np.ndarray) -> np.ndarray:
    d = np.zeros(len(parents), dtype=np.int32)
    for i in range(1, len(parents)):
        d[i] = d[parents[i]] + 1
    return d


def random_root_path(parents: np.ndarray, rng: np.random.Generator, stop_prob: float = 0.25) -> list:
    """A root-to-node walk through the tree (root excluded), in the form of an accept path:
    at each node continue to a uniformly chosen child with probability 1 - stop_prob."""
    kids = {}
    for c in range(1, len(parents)):
        kids.setdefault(int(parents[c]), []).append(c)
    path, cur = [], 0
    while kids.get(cur) and rng.random() >= stop_prob:
        cur = int(rng.choice(kids[cur]))
        path.append(cur)
    return path


PAD = -2    # parent entry of a padding slot past the end of a smaller tree


def padded(parent_rows, num_nodes: int) -> np.ndarray:
    """Stack trees of different sizes into one [B][num_nodes] parent array, each row
    padded with PAD after its own nodes."""
    out = np.full((len(parent_rows), num_nodes), PAD, dtype=np.int32)
    for b, row in enumerate(parent_rows):
        row = np.asarray(row, dtype=np.int32)
        out[b, : len(row)] = row
    return out
