"""Tree ancestry: the mask that decides which draft nodes a node may attend to.

"Tech Radar: SGLang EAGLE-2", section 2 ("Dynamic Tree-Attention Verification"):
candidate i attends to candidate j iff j is an ancestor of i or j = i.
Section 5, item 1: for trees of at most 64 nodes that relation is packed into
one 64-bit word per node, and "is j an ancestor of i" is a single AND of the
word with (1 << j).

The tree arrives as a parent array in topological order: parents[0] = -1
(the root, i.e. the last verified token) and 0 <= parents[i] < i.

Trees larger than 64 nodes ("EAGLE-2 & Lookahead Decoding", section 6: the tree size
follows the load, so a lightly loaded server verifies bigger trees; the radar page's
single word stops at 64).  Reading: the same relation for up to 128 nodes is two 64-bit
words per node, word w holding bits 64w .. 64w+63 of the set; "is j an ancestor of i"
tests bit j % 64 of word j // 64.

A batch may hold trees of different sizes ("EAGLE-2 & Lookahead Decoding",
section 6, "Batched Dynamic Tree Slicing": the tree is cut to fewer tokens under
load).  Reading: each row of the batch's parent array is padded to the batch's
node count with ABSENT; a tree is the entries before its first ABSENT.
"""
from __future__ import annotations

import numpy as np


ABSENT = -2     # parent entry of a padding slot past the end of a smaller tree


def tree_size(parents) -> int:
    """Number of nodes of a padded parent row: the entries before the first ABSENT.

    The root must be present, and no present entry may follow an ABSENT one.
    """
    p = [int(x) for x in parents]
    n = next((i for i, x in enumerate(p) if x == ABSENT), len(p))
    if n == 0:
        raise ValueError("the root (node 0) must be present")
    if any(x != ABSENT for x in p[n:]):
        raise ValueError("a present node follows an absent one")
    return n


def validate_parents(parents) -> None:
    p = [int(x) for x in parents]
    if len(p) == 0 or p[0] != -1:
        raise ValueError("parents[0] must be -1")
    for i in range(1, len(p)):
        if not (0 <= p[i] < i):
            raise ValueError(f"parents[{i}] = {p[i]} is not in [0, {i})")


def ancestors(parents, i: int) -> list[int]:
    """Strict ancestors of node i, found by following parent pointers to the root."""
    out = []
    j = int(parents[i])
    while j >= 0:
        out.append(j)
        j = int(parents[j])
    return out


def mask_matrix(parents) -> np.ndarray:
    """Dense M[i][j] = 1 iff j in Ancestors(i) or j == i (section 2 of the radar page)."""
    validate_parents(parents)
    n = len(parents)
    m = np.zeros((n, n), dtype=bool)
    for i in range(n):
        m[i, i] = True
        for j in ancestors(parents, i):
            m[i, j] = True
    return m


def ancestor_bitmasks(parents) -> list[int]:
    """mask_i with bit j set iff M[i][j] (section 5 item 1 of the radar page); N <= 64."""
    m = mask_matrix(parents)
    n = len(parents)
    if n > 64:
        raise ValueError("a 64-bit ancestry mask holds at most 64 nodes")
    return [sum(1 << j for j in range(n) if m[i, j]) for i in range(n)]


def ancestor_words(parents, n_words: int = 2) -> list[list[int]]:
    """words[i][w] = bits 64w .. 64w+63 of mask_i (bit j set iff M[i][j]); N <= 64 * n_words."""
    m = mask_matrix(parents)
    n = len(parents)
    if n > 64 * n_words:
        raise ValueError(f"{n_words} 64-bit words hold at most {64 * n_words} nodes")
    return [[sum(1 << (j - 64 * w) for j in range(64 * w, min(n, 64 * w + 64)) if m[i, j])
             for w in range(n_words)] for i in range(n)]


def children(parents, i: int) -> list[int]:
    """Children of node i in ascending node index (the order the walk tries them)."""
    return [c for c in range(1, len(parents)) if int(parents[c]) == i]
