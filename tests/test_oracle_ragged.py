"""Pins for trees of different sizes in one batch (parent rows padded with -2).

"EAGLE-2 & Lookahead Decoding", section 6 ("Batched Dynamic Tree Slicing") cuts the
tree to fewer tokens under load, so one batch can hold trees of several sizes.  The
pins tie the padded batch to the unpadded single-tree definitions: every present
row equals the result for its tree alone, the rows of padding slots are zero, and
nothing past a tree's own tokens is read (those pages and rows hold NaN).
"""
import numpy as np
import pytest
from scipy import special

from gen import trees
from oracle import accept as oacc
from oracle import attention as oatt
from oracle.tree_mask import ABSENT, tree_size


def test_tree_size_counts_the_nodes_before_the_padding():
    assert tree_size([-1, 0, 0, 1]) == 4
    assert tree_size([-1, 0, ABSENT, ABSENT]) == 2
    assert tree_size([-1, ABSENT, ABSENT]) == 1
    assert trees.PAD == ABSENT


@pytest.mark.parametrize("bad", [[ABSENT, ABSENT], [-1, ABSENT, 0], [-1, 0, ABSENT, 1, ABSENT]])
def test_tree_size_rejects_a_missing_root_or_a_node_after_the_padding(bad):
    with pytest.raises(ValueError):
        tree_size(bad)


def _ragged_attention_case(seed, sizes, prefix, N=8, Hq=4, Hkv=2, D=16, ps=16):
    rng = np.random.default_rng(seed)
    B = len(sizes)
    rows = [trees.random_recursive(rng, n) for n in sizes]
    parents = trees.padded(rows, N)
    pages_per_seq = -(-(max(prefix) + N) // ps)
    P = B * pages_per_seq + 1                       # the last page is all NaN
    k = rng.normal(size=(P, ps, Hkv, D))
    v = rng.normal(size=(P, ps, Hkv, D))
    k[-1] = np.nan
    v[-1] = np.nan
    table = np.full((B, pages_per_seq), P - 1, dtype=np.int32)
    for b in range(B):
        used = -(-(prefix[b] + sizes[b]) // ps)     # pages holding the sequence's own tokens
        table[b, :used] = b * pages_per_seq + np.arange(used)
    q = rng.normal(size=(B, N, Hq, D))
    q[parents < 0] = np.nan                        # padding slots' queries: never read either
    q[:, 0] = rng.normal(size=(B, Hq, D))
    return q, k, v, table, np.asarray(prefix, dtype=np.int32), parents, rows, ps


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_padded_attention_equals_each_tree_alone(seed):
    sizes, prefix = [8, 3, 1, 5], [5, 20, 0, 16]
    q, k, v, table, S, parents, rows, ps = _ragged_attention_case(seed, sizes, prefix)
    out = oatt.tree_attention(q, k, v, table, S, parents, ps)
    assert np.isfinite(out).all()
    for b, n in enumerate(sizes):
        alone = oatt.tree_attention(q[b:b + 1, :n], k, v, table[b:b + 1], S[b:b + 1], rows[b][None, :], ps)
        np.testing.assert_array_equal(out[b, :n], alone[0])
        assert (out[b, n:] == 0).all()


def _ragged_accept_case(seed, sizes, N=8, V=40, stochastic=True):
    rng = np.random.default_rng(seed)
    rows = [trees.random_recursive(rng, n) for n in sizes]
    parents = trees.padded(rows, N)
    B = len(sizes)
    logits = rng.normal(0, 3, (B, N, V)).astype(np.float32)
    q = special.softmax(logits.astype(np.float64) + rng.normal(0, 1, (B, N, V)), axis=-1).astype(np.float32)
    tokens = rng.integers(0, V, (B, N)).astype(np.int32)
    am = logits.argmax(-1)
    for b in range(B):
        for c in range(1, sizes[b]):
            if not stochastic and rng.random() < 0.7:
                tokens[b, c] = am[b, parents[b, c]]
    u = rng.random((B, N)).astype(np.float32)
    for b, n in enumerate(sizes):                   # padding slots' rows: never read
        logits[b, n:] = np.nan
        q[b, n:] = np.nan
    return logits, tokens, q, parents, u, rows


@pytest.mark.parametrize("temperature", [0.0, 0.7])
@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_padded_accept_equals_each_tree_alone(seed, temperature):
    sizes = [8, 4, 1, 6]
    logits, tokens, q, parents, u, rows = _ragged_accept_case(seed, sizes, stochastic=temperature > 0)
    probs = q if temperature > 0 else None
    unif = u if temperature > 0 else None
    path, length, bonus, _ = oacc.tree_accept(logits, tokens, probs, parents, unif, temperature)
    for b, n in enumerate(sizes):
        alone = oacc.tree_accept(logits[b:b + 1, :n], tokens[b:b + 1, :n], None if probs is None else probs[b:b + 1, :n],
                                 rows[b][None, :], None if unif is None else unif[b:b + 1, :n], temperature)
        assert length[b] == alone[1][0] and bonus[b] == alone[2][0]
        assert (path[b, : length[b]] == alone[0][0, : length[b]]).all()
        assert (path[b, length[b]:] == -1).all()
        assert all(0 <= int(x) < n for x in path[b, : length[b]])
