"""Pins for the float64 tree-attention oracle.

Each check ties the oracle to something other than its own formula:
torch's scaled_dot_product_attention on a contiguous sequence (a library
routine, run in float64 on the CPU), closed forms, invariances, and an
ancestor set computed by a different algorithm (matrix-power closure).
"""
import inspect
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from gen import trees
from oracle import attention as oatt
from oracle import tree_mask

PS = 16


def make_case(rng, B, N, Hq, Hkv, D, prefix, parents=None, shuffle=True):
    """Random paged inputs; tree K/V at logical positions S..S+N-1."""
    prefix = np.asarray(prefix, dtype=np.int64)
    if parents is None:
        parents = np.stack([trees.random_recursive(rng, N) for _ in range(B)])
    ntok = prefix + N
    npages = (ntok + PS - 1) // PS
    total = int(npages.sum())
    perm = rng.permutation(total + 1) if shuffle else np.arange(total + 1)
    table = np.zeros((B, int(npages.max())), dtype=np.int64)
    seqs_k, seqs_v = [], []
    kp = np.full((total + 1, PS, Hkv, D), np.nan)
    vp = np.full((total + 1, PS, Hkv, D), np.nan)
    start = 0
    for b in range(B):
        table[b, : npages[b]] = perm[start:start + npages[b]]
        table[b, npages[b]:] = perm[-1]
        start += npages[b]
        k = rng.standard_normal((ntok[b], Hkv, D))
        v = rng.standard_normal((ntok[b], Hkv, D))
        seqs_k.append(k)
        seqs_v.append(v)
        for t in range(ntok[b]):
            kp[table[b, t // PS], t % PS] = k[t]
            vp[table[b, t // PS], t % PS] = v[t]
    q = rng.standard_normal((B, N, Hq, D))
    return dict(q=q, k_pages=kp, v_pages=vp, page_table=table, prefix_lens=prefix,
                tree_parents=parents, seqs_k=seqs_k, seqs_v=seqs_v)


def run_oracle(c):
    return oatt.tree_attention(c["q"], c["k_pages"], c["v_pages"], c["page_table"],
                               c["prefix_lens"], c["tree_parents"], PS)


def sdpa(q, k, v):
    """torch SDPA, float64: q [Hq][Lq][D], k/v [Hkv][Lk][D] with GQA by head repetition."""
    G = q.shape[0] // k.shape[0]
    kt = torch.from_numpy(np.repeat(k, G, axis=0))
    vt = torch.from_numpy(np.repeat(v, G, axis=0))
    return F.scaled_dot_product_attention(torch.from_numpy(q), kt, vt).numpy()


def closure_by_matrix_powers(parents):
    """Ancestor-or-self relation via powers of the child->parent adjacency matrix."""
    n = len(parents)
    A = np.zeros((n, n), dtype=np.int64)
    for i in range(1, n):
        A[i, parents[i]] = 1
    R = np.eye(n, dtype=np.int64)
    P = np.eye(n, dtype=np.int64)
    for _ in range(n):
        P = P @ A
        R = R + P
    return R > 0


# ---------------------------------------------------------------- the mask

@pytest.mark.parametrize("seed", range(20))
def test_dense_mask_equals_matrix_power_closure(seed):
    rng = np.random.default_rng(seed)
    p = trees.random_recursive(rng, int(rng.integers(1, 65)))
    assert np.array_equal(tree_mask.mask_matrix(p), closure_by_matrix_powers(p))


def test_mask_special_shapes():
    n = 9
    assert np.array_equal(tree_mask.mask_matrix(trees.chain(n)), np.tril(np.ones((n, n), bool)))
    star = np.eye(n, dtype=bool)
    star[:, 0] = True
    assert np.array_equal(tree_mask.mask_matrix(trees.star(n)), star)


@pytest.mark.parametrize("seed", range(10))
def test_bitmask_is_dense_mask(seed):
    rng = np.random.default_rng(100 + seed)
    p = trees.random_recursive(rng, 64)
    m = closure_by_matrix_powers(p)
    words = tree_mask.ancestor_bitmasks(p)
    for i in range(64):
        for j in range(64):
            assert bool(words[i] & (1 << j)) == m[i, j]


@pytest.mark.parametrize("bad", [[0, 0], [-1, 1], [-1, 0, 3], [-1, -1], [-1, 0, -2]])
def test_invalid_parents_rejected(bad):
    with pytest.raises(ValueError):
        tree_mask.mask_matrix(bad)


def test_bitmask_limit():
    with pytest.raises(ValueError):
        tree_mask.ancestor_bitmasks(trees.chain(65))
    with pytest.raises(ValueError):
        tree_mask.ancestor_words(trees.chain(129), 2)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("n", [65, 100, 128])
def test_two_word_masks_are_the_dense_mask(seed, n):
    """Trees past 64 nodes: bit j % 64 of word j // 64 equals the matrix-power closure."""
    rng = np.random.default_rng(200 + seed)
    p = trees.random_recursive(rng, n)
    m = closure_by_matrix_powers(p)
    words = tree_mask.ancestor_words(p, 2)
    for i in range(n):
        for j in range(n):
            assert bool((words[i][j // 64] >> (j % 64)) & 1) == m[i, j]
        assert words[i][1] == 0 or n > 64


def test_two_word_masks_closed_forms():
    """A chain of 128: node i holds bits 0..i.  A star of 128: the root and itself.
    A tree of at most 64 nodes: word 0 is the single-word mask, word 1 is empty."""
    for i, (w0, w1) in enumerate(tree_mask.ancestor_words(trees.chain(128), 2)):
        full = (1 << (i + 1)) - 1
        assert (w0, w1) == (full & (2**64 - 1), full >> 64)
    for i, (w0, w1) in enumerate(tree_mask.ancestor_words(trees.star(128), 2)):
        bits = {0, i}
        assert w0 == sum(1 << j for j in bits if j < 64) and w1 == sum(1 << (j - 64) for j in bits if j >= 64)
    p = trees.random_recursive(np.random.default_rng(5), 64)
    assert [w[0] for w in tree_mask.ancestor_words(p, 2)] == tree_mask.ancestor_bitmasks(p)
    assert all(w[1] == 0 for w in tree_mask.ancestor_words(p, 2))


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("S", [0, 5, 37])
def test_chain_equals_causal_attention(S):
    """A chain-shaped tree is ordinary causal attention over prefix + chain."""
    rng = np.random.default_rng(S)
    N, Hq, Hkv, D = 7, 4, 2, 16
    c = make_case(rng, 1, N, Hq, Hkv, D, [S], parents=trees.chain(N)[None])
    out = run_oracle(c)
    L = S + N
    qfull = rng.standard_normal((Hq, L, D))
    qfull[:, S:, :] = c["q"][0].transpose(1, 0, 2)
    k = c["seqs_k"][0].transpose(1, 0, 2)
    v = c["seqs_v"][0].transpose(1, 0, 2)
    G = Hq // Hkv
    ref = F.scaled_dot_product_attention(
        torch.from_numpy(qfull), torch.from_numpy(np.repeat(k, G, 0)),
        torch.from_numpy(np.repeat(v, G, 0)), is_causal=True).numpy()
    np.testing.assert_allclose(out[0], ref[:, S:, :].transpose(1, 0, 2), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(8))
def test_node_equals_attention_along_its_root_path(seed):
    """Every node's output is plain attention over prefix + its root->node path, laid out
    contiguously; seeds 6 and 7 draw trees past 64 nodes (up to 128)."""
    rng = np.random.default_rng(1000 + seed)
    B, N, Hq, Hkv, D = 2, int(rng.integers(2, 20) if seed < 6 else rng.integers(65, 129)), 8, 2, 32
    prefix = rng.integers(0, 70, B)
    c = make_case(rng, B, N, Hq, Hkv, D, prefix)
    out = run_oracle(c)
    for b in range(B):
        S = int(prefix[b])
        p = c["tree_parents"][b]
        for i in range(N):
            path = [i]
            while p[path[-1]] >= 0:
                path.append(int(p[path[-1]]))
            path = path[::-1]
            idx = list(range(S)) + [S + j for j in path]
            k = c["seqs_k"][b][idx].transpose(1, 0, 2)
            v = c["seqs_v"][b][idx].transpose(1, 0, 2)
            ref = sdpa(c["q"][b, i][:, None, :], k, v)[:, 0, :]
            np.testing.assert_allclose(out[b, i], ref, rtol=1e-12, atol=1e-12)


def test_single_node_is_decode_attention():
    rng = np.random.default_rng(7)
    S, Hq, Hkv, D = 45, 6, 3, 64
    c = make_case(rng, 1, 1, Hq, Hkv, D, [S], parents=np.array([[-1]]))
    out = run_oracle(c)
    ref = sdpa(c["q"][0, 0][:, None, :], c["seqs_k"][0].transpose(1, 0, 2),
               c["seqs_v"][0].transpose(1, 0, 2))[:, 0]
    np.testing.assert_allclose(out[0, 0], ref, rtol=1e-12, atol=1e-12)


def test_zero_query_gives_mean_of_attended_values():
    rng = np.random.default_rng(8)
    N, S, Hq, Hkv, D = 12, 19, 4, 4, 8
    c = make_case(rng, 1, N, Hq, Hkv, D, [S])
    c["q"][:] = 0.0
    out = run_oracle(c)
    m = closure_by_matrix_powers(c["tree_parents"][0])
    for i in range(N):
        idx = list(range(S)) + [S + j for j in np.flatnonzero(m[i])]
        for hq in range(Hq):
            np.testing.assert_allclose(out[0, i, hq], c["seqs_v"][0][idx, hq].mean(0), rtol=1e-12,
                                       atol=1e-13)


def test_page_table_permutation_invariance():
    rng = np.random.default_rng(9)
    c = make_case(rng, 2, 9, 4, 2, 16, [33, 50])
    out = run_oracle(c)
    P = c["k_pages"].shape[0]
    perm = rng.permutation(P)               # new physical position of each page
    inv = np.argsort(perm)
    c2 = dict(c)
    c2["k_pages"] = c["k_pages"][inv]
    c2["v_pages"] = c["v_pages"][inv]
    c2["page_table"] = perm[c["page_table"]]
    np.testing.assert_allclose(run_oracle(c2), out, rtol=1e-12, atol=1e-12)


def test_topological_relabelling_permutes_outputs():
    """Listing the nodes in another topological order permutes the outputs the same way."""
    rng = np.random.default_rng(10)
    N, S = 14, 21
    c = make_case(rng, 1, N, 4, 1, 16, [S])
    out = run_oracle(c)
    p = c["tree_parents"][0]
    d = trees.depths(p)
    order = sorted(range(N), key=lambda i: (d[i], -i))    # BFS order, reversed within a level
    new_of = {old: new for new, old in enumerate(order)}
    p2 = np.array([-1] + [new_of[int(p[old])] for old in order[1:]])
    c2 = make_case(np.random.default_rng(0), 1, N, 4, 1, 16, [S], parents=p2[None], shuffle=False)
    k = c["seqs_k"][0].copy()
    v = c["seqs_v"][0].copy()
    k[S:] = c["seqs_k"][0][S:][order]
    v[S:] = c["seqs_v"][0][S:][order]
    for t in range(S + N):
        c2["k_pages"][c2["page_table"][0, t // PS], t % PS] = k[t]
        c2["v_pages"][c2["page_table"][0, t // PS], t % PS] = v[t]
    c2["q"] = c["q"][:, order]
    np.testing.assert_allclose(run_oracle(c2)[0], out[0][order], rtol=1e-12, atol=1e-12)


# ------------------------------------------------- planted mistakes are caught

def _planted(func, old, new):
    src = inspect.getsource(func)
    assert old in src
    ns = dict(vars(inspect.getmodule(func)))
    exec(compile(src.replace(old, new), "<planted>", "exec"), ns)
    return ns[func.__name__]


@pytest.mark.parametrize("func,old,new", [
    (oatt.attend_one, "math.sqrt(q_vec.shape[-1])", "q_vec.shape[-1]"),          # wrong scale
    (tree_mask.mask_matrix, "m[i, i] = True", "pass"),                           # self dropped
    (oatt.tree_attention, "h * G:(h + 1) * G", "h:h + G"),                       # wrong GQA map
])
def test_planted_mistakes_fail_the_path_pin(monkeypatch, func, old, new):
    mod = inspect.getmodule(func)
    planted = _planted(func, old, new)
    monkeypatch.setattr(mod, func.__name__, planted)
    if mod is tree_mask:
        monkeypatch.setattr(oatt, func.__name__, planted)
    with pytest.raises(AssertionError):
        test_node_equals_attention_along_its_root_path(0)
