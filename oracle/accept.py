"""Accept walk over a verified draft tree, float64, step by step as the pages state it.

Greedy (temperature 0): "EAGLE-2 & Lookahead Decoding", section 4, accepts the
longest path whose tokens the target agrees with.  From the root, the walk
moves to the first child (ascending node index) whose token equals the
argmax of the current node's target row (ties: lowest token id); when no
child matches it stops, and the bonus token is that argmax.

Stochastic (temperature T > 0): the rejection rule of "Speculative Decoding in
Production: EAGLE-3 Dynamic Trees", section "Mathematical Proof of Lossless
Speedup", steps 1-3 (also "Tech Radar: SGLang EAGLE-2", section 5):
  1. alpha = min(1, p(x) / q(x)) for a draft token x;
  2. draw r ~ U(0, 1); accept iff r <= alpha (written here as u*q(x) <= p(x),
     with p(x) > 0 required);
  3. on rejection, resample from the normalised residual max(0, p - q).
Over a tree, a rejected child hands the residual to its next sibling ("If
branch B1 is rejected but branch B2 matches ... accepts B2 -> C2", section
"From Linear Sequences to Dynamic Draft Trees" of the same page): the next
sibling is tested against the residual instead of p.  When no child is
accepted, the bonus token is drawn from the current distribution (the
residual, or p at a leaf) by inverse CDF with the sequence's own uniform.

Readings where the pages are silent: p_i = softmax(logits_i / T); q_i is used
as given; uniforms[0] is the final-sample coin and uniforms[c] the accept coin
of node c; a residual whose total is 0 is left unchanged; a CDF that never
exceeds the threshold (rounding) yields the largest token with r > 0.

Margins: for every stochastic decision the oracle records how far it was from
flipping (relative to the size of the quantities involved), so a comparison
with a float32 implementation can tell a genuine disagreement from a
rounding tie.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .tree_mask import children, tree_size, validate_parents


@dataclass
class WalkResult:
    path: list                       # accepted node indices, root excluded
    bonus: int
    min_margin: float = float("inf")
    decisions: list = field(default_factory=list)

    @property
    def length(self) -> int:
        return len(self.path)


def softmax(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(x - x.max())
    return e / e.sum()


def greedy_walk(logits, tokens, parents) -> WalkResult:
    """logits [N][V], tokens [N], parents [N] -> accepted path and bonus token."""
    validate_parents(parents)
    cur, path = 0, []
    while True:
        best = int(np.argmax(np.asarray(logits[cur], dtype=np.float64)))  # first max = lowest id
        nxt = next((c for c in children(parents, cur) if int(tokens[c]) == best), None)
        if nxt is None:
            return WalkResult(path, best)
        path.append(nxt)
        cur = nxt


def stochastic_walk(logits, tokens, q, parents, uniforms, temperature: float) -> WalkResult:
    """Rejection-sampling walk; q [N][V] is the draft distribution each node's children came from."""
    validate_parents(parents)
    T = float(temperature)
    cur, path = 0, []
    res = WalkResult(path, -1)
    r = softmax(np.asarray(logits[0], dtype=np.float64) / T)
    scale = r.copy()                       # magnitude of the terms behind r (for margins)
    while True:
        accepted = None
        q_cur = np.asarray(q[cur], dtype=np.float64)
        for c in children(parents, cur):
            x = int(tokens[c])
            lhs = float(uniforms[c]) * q_cur[x]
            ok = r[x] > 0 and lhs <= r[x]
            margin = abs(lhs - r[x]) / max(lhs, r[x], scale[x], 1e-300)
            res.decisions.append(("test", c, x, bool(ok), margin))
            res.min_margin = min(res.min_margin, margin)
            if ok:
                accepted = c
                break
            resid = np.maximum(0.0, r - q_cur)
            z = resid.sum()
            if z > 0:
                r = resid / z
                scale = (scale + q_cur) / z
        if accepted is None:
            break
        path.append(accepted)
        cur = accepted
        r = softmax(np.asarray(logits[cur], dtype=np.float64) / T)
        scale = r.copy()
    cdf = np.cumsum(r)
    total = cdf[-1]
    thr = float(uniforms[0]) * total
    above = np.flatnonzero(cdf > thr)
    if len(above):
        v = int(above[0])
        lo = cdf[v - 1] if v > 0 else 0.0
        margin = min(cdf[v] - thr, thr - lo) / total
    else:
        v = int(np.flatnonzero(r > 0)[-1])
        margin = 0.0
    res.decisions.append(("sample", cur, v, True, margin))
    res.min_margin = min(res.min_margin, margin)
    res.bonus = v
    return res


def tree_accept(target_logits, draft_tokens, draft_probs, tree_parents, uniforms,
                temperature: float):
    """Batch form of the walk.

    Returns (accept_path [B][N] int32, -1 padded; accept_len [B]; bonus_token [B];
    list of WalkResult).  A parent row padded with ABSENT is walked as its first
    tree_size entries; the padding slots' rows are not read.
    """
    B, N = np.asarray(draft_tokens).shape
    path = np.full((B, N), -1, dtype=np.int32)
    length = np.zeros(B, dtype=np.int32)
    bonus = np.zeros(B, dtype=np.int32)
    results = []
    for b in range(B):
        nb = tree_size(tree_parents[b])
        if temperature == 0:
            w = greedy_walk(target_logits[b][:nb], draft_tokens[b][:nb], tree_parents[b][:nb])
        else:
            w = stochastic_walk(target_logits[b][:nb], draft_tokens[b][:nb], draft_probs[b][:nb],
                                tree_parents[b][:nb], uniforms[b][:nb], temperature)
        path[b, : w.length] = w.path
        length[b] = w.length
        bonus[b] = w.bonus
        results.append(w)
    return path, length, bonus, results
