"""GPU parity for batches of trees of different sizes (parent rows padded with -2)."""
import numpy as np
import pytest
import torch
from scipy import special

import gen
from gen import inputs as gi
from gen import trees

from gpu_util import (assert_attention_close, attn_device_inputs, compare_accept, dev_tensor, oracle_attention)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import __graft_entry__
    __graft_entry__.build()
    import eagle_speculative_tree_gb300 as mod
    return mod


SIZES = [64, 17, 1, 40]
PREFIX = [100, 37, 0, 300]


@pytest.mark.parametrize("kernel,splits", [(1, 1), (1, 0), (2, 1), (2, 0), (3, 1), (3, 0), (4, 1), (4, 0), (5, 0)])
def test_attention_over_trees_of_different_sizes(ts, cuda_device, kernel, splits):
    """Present rows match the oracle, padding rows are zero, and no page past a tree's
    own S + N_b tokens is read (those page ids are made invalid)."""
    rng = np.random.default_rng(7)
    w = gen.get("c4_llama3_70b_bf16_greedy").with_batch(len(SIZES))
    parents = trees.padded([trees.random_recursive(rng, n) for n in SIZES], w.num_nodes)
    x = gi.make_inputs(w, parents=parents, prefix_lens=np.asarray(PREFIX, dtype=np.int32), with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    table = d["page_table"].clone()
    for b, (n, s) in enumerate(zip(SIZES, PREFIX)):
        table[b, -(-(s + n) // w.page_size):] = 1 << 30
    prob = ts.attn_problem(d["q"], d["k_pages"], table, kernel=kernel, num_splits=splits)
    assert ts.attn_plan(prob).kernel == kernel
    ws = torch.empty(ts.attn_workspace_bytes(prob), dtype=torch.uint8, device=cuda_device)
    out = ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], table, d["prefix_lens"], d["tree_parents"],
                              kernel=kernel, num_splits=splits, workspace=ws)
    torch.cuda.synchronize()
    assert ts.read_status(ws) == 0
    ref = oracle_attention(x)
    assert_attention_close(out, ref, w.dtype)
    for b, n in enumerate(SIZES):
        assert torch.all(out[b, n:] == 0)


@pytest.mark.parametrize("kernel", [1, 2, 3, 4, 5])
def test_attention_over_trees_of_up_to_128_nodes_of_different_sizes(ts, cuda_device, kernel):
    """A batch of 128-node rows holding trees of 128, 65, 64 and 3 nodes."""
    from dataclasses import replace
    rng = np.random.default_rng(17)
    sizes, prefix = [128, 65, 64, 3], [90, 1000, 0, 33]
    w = replace(gen.get("c4_llama3_70b_bf16_greedy").with_batch(len(sizes)), num_nodes=128)
    parents = trees.padded([trees.random_recursive(rng, n) for n in sizes], w.num_nodes)
    x = gi.make_inputs(w, parents=parents, prefix_lens=np.asarray(prefix, dtype=np.int32), with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    out = ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["prefix_lens"],
                              d["tree_parents"], kernel=kernel)
    torch.cuda.synchronize()
    assert_attention_close(out, oracle_attention(x), w.dtype)
    for b, n in enumerate(sizes):
        assert torch.all(out[b, n:] == 0)


def test_attention_flags_a_node_after_the_padding(ts, cuda_device):
    w = gen.get("c2_llama3_8b_bf16_greedy").with_batch(1)
    x = gi.make_inputs(w, parents=np.asarray([[-1, 0, trees.PAD, 1, trees.PAD, trees.PAD, trees.PAD, trees.PAD]],
                                             dtype=np.int32), with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    ws = torch.empty(ts.attn_workspace_bytes(ts.attn_problem(d["q"], d["k_pages"], d["page_table"])),
                     dtype=torch.uint8, device=cuda_device)
    ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["prefix_lens"], d["tree_parents"],
                        workspace=ws)
    torch.cuda.synchronize()
    assert ts.read_status(ws) & 1


def _ragged_accept(seed, sizes, N, V, temperature):
    rng = np.random.default_rng(seed)
    rows = [trees.random_recursive(rng, n) for n in sizes]
    parents = trees.padded(rows, N)
    B = len(sizes)
    logits = rng.normal(0, 3, (B, N, V)).astype(np.float32)
    q = special.softmax(logits.astype(np.float64) + rng.normal(0, 1, (B, N, V)), axis=-1).astype(np.float32)
    tokens = np.zeros((B, N), dtype=np.int32)
    am = logits.argmax(-1)
    for b, n in enumerate(sizes):
        for c in range(1, n):
            par = parents[b, c]
            if temperature == 0:
                tokens[b, c] = am[b, par] if rng.random() < 0.7 else rng.integers(0, V)
            else:
                row = q[b, par].astype(np.float64)
                tokens[b, c] = min(int(np.searchsorted(np.cumsum(row), rng.random() * row.sum())), V - 1)
        logits[b, n:] = np.nan                       # padding slots' rows: never read
        q[b, n:] = np.nan
    u = rng.random((B, N)).astype(np.float32)
    return logits, tokens, q, parents, u


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("temperature", [0.0, 0.7])
@pytest.mark.parametrize("V", [1000, 128256])
def test_accept_over_trees_of_different_sizes(ts, cuda_device, mode, temperature, V):
    sizes, N = [16, 5, 1, 9, 2, 16], 16
    logits, tokens, q, parents, u = _ragged_accept(11, sizes, N, V, temperature)
    stoch = temperature > 0
    res = ts.tree_accept(dev_tensor(logits, cuda_device), dev_tensor(tokens, cuda_device),
                         dev_tensor(q, cuda_device) if stoch else None, dev_tensor(parents, cuda_device),
                         dev_tensor(u, cuda_device) if stoch else None, temperature, mode=mode)
    torch.cuda.synchronize()
    path, length, _bonus = (t.cpu().numpy() for t in res)
    for b, n in enumerate(sizes):
        assert length[b] < n and all(0 < int(c) < n for c in path[b, : length[b]])
    n_seq, _ties, flipped = compare_accept(res, logits, tokens, q if stoch else None, parents,
                                           u if stoch else None, temperature)
    assert flipped <= max(1, n_seq // 16)
