"""Pins of oracle.kv_commit (keeping the accepted path's K/V; CPU only)."""
import inspect

import numpy as np
import pytest

from gen import trees
from oracle import kv_commit as okc

PS = 16


def tagged_pool(pages, hkv=2, d=4):
    """Pool whose every value names its (page, slot, head, dim): 1000 page + slot + head/10 + dim/100."""
    p = np.arange(pages)[:, None, None, None] * 1000.0 + np.arange(PS)[None, :, None, None]
    return p + np.arange(hkv)[None, None, :, None] / 10 + np.arange(d)[None, None, None, :] / 100 + np.zeros(
        (pages, PS, hkv, d))


def test_hand_worked_example_across_a_page_boundary():
    # S = 14 prefix tokens, tree of N = 6 nodes at logical positions 14..19; pages [7, 3]:
    # positions 0..15 live in page 7, 16..31 in page 3.  Accepted path [2, 5]:
    #   node 2 (position 16 = page 3 slot 0) -> position 15 (page 7 slot 15)
    #   node 5 (position 19 = page 3 slot 3) -> position 16 (page 3 slot 0)
    # the root (position 14, page 7 slot 14) stays; new length 14 + 1 + 2 = 17.
    k = tagged_pool(8)
    v = -tagged_pool(8)
    pt = np.array([[7, 3]], dtype=np.int32)
    k2, v2, lens, st = okc.kv_commit(k, v, pt, np.array([14]), np.array([[2, 5, -1, -1, -1, -1]]),
                                      np.array([2]), num_nodes=6)
    assert st == 0 and lens.tolist() == [17]
    assert np.allclose(k2[7, 15], 3000 + np.arange(2)[:, None] / 10 + np.arange(4)[None, :] / 100)
    assert np.allclose(k2[3, 0], 3003 + np.arange(2)[:, None] / 10 + np.arange(4)[None, :] / 100)
    assert np.allclose(v2[7, 15], -k2[7, 15]) and np.allclose(v2[3, 0], -k2[3, 0])
    changed = np.argwhere((k2 != k).any(axis=(2, 3)))
    assert sorted(map(tuple, changed.tolist())) == [(3, 0), (7, 15)]     # nothing else moved
    assert k2[7, 14, 0, 0] == 7014 and k2[3, 3, 0, 0] == 3003            # root and old source stay


def test_planted_off_by_one_destination_fails_the_example():
    src = inspect.getsource(okc.kv_commit).replace("S + 1 + k", "S + k")
    ns = {"np": np, "BAD_PAGE": 2, "BAD_LENGTH": 4, "BAD_PATH": 64}
    exec(src, ns)
    k = tagged_pool(8)
    k2, _v, _l, _s = ns["kv_commit"](k, -k, np.array([[7, 3]], dtype=np.int32), np.array([14]),
                                     np.array([[2, 5, -1, -1, -1, -1]]), np.array([2]), num_nodes=6)
    assert not np.allclose(k2[7, 15, 0, 0], 3000)


def test_in_order_path_and_empty_path_change_nothing():
    k = tagged_pool(4)
    pt = np.array([[2, 0, 3, 1]], dtype=np.int32)
    for n in (0, 1, 5):
        path = np.full((1, 8), -1)
        path[0, :n] = np.arange(1, n + 1)
        k2, v2, lens, st = okc.kv_commit(k, -k, pt, np.array([20]), path, np.array([n]), num_nodes=8)
        assert st == 0 and lens.tolist() == [21 + n]
        assert np.array_equal(k2, k) and np.array_equal(v2, -k)


@pytest.mark.parametrize("seed", range(6))
def test_sequence_becomes_prefix_root_and_path(seed):
    # independent statement: gather each sequence densely, build the expected sequence by
    # list slicing, and compare with the committed pool read back through the page table
    rng = np.random.default_rng(seed)
    B, N, pages_per_seq = 3, 12, 4
    P = B * pages_per_seq + 2
    k = rng.standard_normal((P, PS, 2, 4))
    v = rng.standard_normal((P, PS, 2, 4))
    pt = rng.permutation(P)[:B * pages_per_seq].reshape(B, pages_per_seq).astype(np.int32)
    S = rng.integers(0, pages_per_seq * PS - N + 1, size=B)
    paths = np.full((B, N), -1)
    lens = np.zeros(B, dtype=np.int64)
    for b in range(B):
        par = trees.random_recursive(rng, N)
        pth = trees.random_root_path(par, rng, stop_prob=0.1)
        paths[b, :len(pth)] = pth
        lens[b] = len(pth)
    k2, v2, new_lens, st = okc.kv_commit(k, v, pt, S, paths, lens, num_nodes=N)
    assert st == 0
    for b in range(B):
        dense_k = [k[pt[b, t // PS], t % PS] for t in range(pages_per_seq * PS)]
        want = dense_k[:S[b] + 1] + [dense_k[S[b] + int(x)] for x in paths[b, :lens[b]]]
        got = [k2[pt[b, t // PS], t % PS] for t in range(int(new_lens[b]))]
        assert new_lens[b] == S[b] + 1 + lens[b]
        assert all(np.array_equal(g, w) for g, w in zip(got, want))
        tail = [k2[pt[b, t // PS], t % PS] for t in range(int(new_lens[b]), pages_per_seq * PS)]
        assert all(np.array_equal(g, w) for g, w in zip(tail, dense_k[int(new_lens[b]):]))   # untouched


@pytest.mark.parametrize("S,path,n,bit", [
    (-1, [1], 1, okc.BAD_LENGTH),            # negative prefix
    (62, [2], 1, okc.BAD_LENGTH),            # the source at 62 + 2 lies past the page table (64 slots)
    (64, [], 0, okc.BAD_LENGTH),             # even the root lies past it
    (0, [2, 2], 2, okc.BAD_PATH),            # not strictly increasing
    (0, [0], 1, okc.BAD_PATH),               # the root is not a path entry
    (0, [9], 1, okc.BAD_PATH),               # node index >= N
    (0, [1], 8, okc.BAD_PATH),               # more accepted nodes than N - 1
])
def test_invalid_sequences_are_left_unchanged(S, path, n, bit):
    k = tagged_pool(4)
    pth = np.full((1, 8), -1)
    pth[0, :len(path)] = path
    k2, _v, lens, st = okc.kv_commit(k, -k, np.array([[0, 1, 2, 3]], dtype=np.int32), np.array([S]), pth,
                                      np.array([n]), num_nodes=8)
    assert st & bit and lens.tolist() == [-1] and np.array_equal(k2, k)


def test_bad_page_is_reported_and_nothing_moves():
    k = tagged_pool(4)
    k2, _v, lens, st = okc.kv_commit(k, -k, np.array([[0, 9, 2, 3]], dtype=np.int32), np.array([14]),
                                      np.array([[2, -1, -1, -1, -1, -1, -1, -1]]), np.array([1]), num_nodes=8)
    assert st & okc.BAD_PAGE and lens.tolist() == [-1] and np.array_equal(k2, k)


def test_bound_is_the_deepest_position_touched_not_the_tree_size():
    # A tree of N = 8 nodes at S = 60 would run past 64 slots, but a commit only touches
    # positions S .. S + max(path): path [1, 3] touches 60..63 and fits; path [1, 4] reaches
    # position 64 and does not.  An empty path touches only the root.
    k = tagged_pool(4)
    pt = np.array([[0, 1, 2, 3]], dtype=np.int32)
    for path, n, ok in [([1, 3], 2, True), ([1, 4], 2, False), ([], 0, True), ([3], 1, True)]:
        pth = np.full((1, 8), -1)
        pth[0, :len(path)] = path
        k2, _v, lens, st = okc.kv_commit(k, -k, pt, np.array([60]), pth, np.array([n]), num_nodes=8)
        if ok:
            assert st == 0 and lens.tolist() == [61 + n]
            for j, x in enumerate(path):          # node x (position 60 + x) now sits at 61 + j
                src, dst = 60 + x, 61 + j
                assert np.array_equal(k2[pt[0, dst // PS], dst % PS], k[pt[0, src // PS], src % PS])
        else:
            assert st & okc.BAD_LENGTH and lens.tolist() == [-1] and np.array_equal(k2, k)


def test_padded_tree_commits_like_the_same_tree_unpadded():
    # the same 5-node tree, once alone (N = 5) and once padded to N = 12 with absent slots:
    # the committed pools and lengths agree, also where S + 12 exceeds the page table
    rng = np.random.default_rng(3)
    k = rng.standard_normal((4, PS, 2, 4))
    pt = np.array([[2, 0, 3, 1]], dtype=np.int32)
    path = np.array([[1, 4] + [-1] * 10])
    for S in (10, 57, 59):
        a = okc.kv_commit(k, -k, pt, np.array([S]), path[:, :5], np.array([2]), num_nodes=5)
        b = okc.kv_commit(k, -k, pt, np.array([S]), path, np.array([2]), num_nodes=12)
        assert a[3] == b[3] == 0 and a[2].tolist() == b[2].tolist() == [S + 3]
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
