"""Input generator checks: tree recipes, page layout, dtype conversion, seeding."""
import json
import os

import numpy as np
import pytest

import gen
from gen import inputs as gi
from gen import trees


def test_mtp_two_node_tree():
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "mtp_two_node_tree.json")))
    p = trees.build_tree(np.random.default_rng(0), g["num_steps"], g["topk"], g["num_nodes"])
    assert p.tolist() == g["expected_parents"]


@pytest.mark.parametrize("name", list(gen.WORKLOADS))
def test_recipe_trees_are_valid_and_shallow(name):
    w = gen.get(name)
    for b in range(3):
        p = trees.build_tree(gi.rng_for(w, b, gi.TREE), w.num_steps, w.topk, w.num_nodes)
        assert p[0] == -1 and all(0 <= p[i] < i for i in range(1, len(p)))
        d = trees.depths(p)
        assert d.max() <= w.num_steps
        assert all(d[i] >= d[i - 1] for i in range(1, len(p)))   # (depth, creation) order
        kids = np.bincount(p[1:], minlength=len(p))
        assert kids.max() <= w.topk


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-3, 3.0e38], dtype=np.float32)
    bits = gi.f32_to_bf16_bits(x)
    back = gi.bf16_bits_to_f32(bits)
    assert back[0] == 1.0
    assert back[1] == 1.0                       # tie -> even
    assert back[2] == np.float32(1.0 + 4 * 2 ** -8)   # tie -> even (up)
    assert back[3] == -2.5
    assert abs(back[4] - 1e-3) <= 2 ** -9 * 1e-3
    import torch
    t = torch.from_numpy(np.random.default_rng(0).standard_normal(10000).astype(np.float32))
    ref = t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gi.f32_to_bf16_bits(t.numpy()), ref)


def test_small_workload_layout():
    w = gen.get("c1_tiny_f32_greedy")
    x = gi.make_inputs(w)
    B, N = w.batch, w.num_nodes
    assert x.q.shape == (B, N, w.num_q_heads, w.head_dim)
    ps = w.page_size
    for b in range(B):
        L = int(x.prefix_lens[b]) + N
        used = x.page_table[b, : (L + ps - 1) // ps]
        assert len(set(used.tolist())) == len(used)
        # every logical token is finite, the rest of the last page is poisoned
        flat = x.k_pages[used].reshape(-1, w.num_kv_heads, w.head_dim)
        assert np.isfinite(flat[:L]).all() and np.isnan(flat[L:]).all()
    assert np.isnan(x.k_pages[-1]).all()
    assert x.target_logits.shape == (B, N, w.vocab)
    assert x.draft_probs is None and x.uniforms is None


def test_seeding_is_per_sequence():
    w = gen.get("c3_llama2_7b_bf16_stoch").with_batch(2)
    a = gi.make_inputs(w)
    w1 = w.with_batch(1)
    b = gi.make_inputs(w1)
    assert np.array_equal(a.q[0], b.q[0])
    assert np.array_equal(a.target_logits[0], b.target_logits[0])
    assert np.array_equal(a.draft_tokens[0], b.draft_tokens[0])
    np.testing.assert_allclose(a.draft_probs.sum(-1), 1.0, atol=1e-5)


def test_greedy_siblings_distinct():
    w = gen.get("c2_llama3_8b_bf16_greedy")
    x = gi.make_inputs(w)
    p = x.tree_parents[0]
    for node in range(w.num_nodes):
        toks = [x.draft_tokens[0, c] for c in range(1, w.num_nodes) if p[c] == node]
        assert len(toks) == len(set(toks))
