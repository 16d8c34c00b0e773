"""GPU parity of tree_attn_verify against the float64 oracle (through the C-ABI)."""
import numpy as np
import pytest
import torch

import gen
from gen import inputs as gi
from gen import trees

from gpu_util import (assert_attention_close, attn_device_inputs, dev_tensor, oracle_attention)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import __graft_entry__
    __graft_entry__.build()
    import eagle_speculative_tree_gb300 as mod
    return mod


def run(ts, x, device, **kw):
    d = attn_device_inputs(x, device)
    out = ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["prefix_lens"],
                              d["tree_parents"], **kw)
    torch.cuda.synchronize()
    return out


SMALL = [
    ("c1_tiny_f32_greedy", None),
    ("c2_llama3_8b_bf16_greedy", None),
    ("c3_llama2_7b_bf16_stoch", 2),
    ("c4_llama3_70b_bf16_greedy", 1),
    ("c5_ragged_b64_bf16_stoch", 3),
]


def row_blocks(w):
    return -(-w.num_nodes * w.group // 128)


@pytest.mark.parametrize("kernel", [0, 1, 2, 3, 4, 5])
@pytest.mark.parametrize("name,batch", SMALL)
def test_configs_match_oracle(ts, cuda_device, name, batch, kernel):
    w = gen.get(name)
    if batch is not None:
        w = w.with_batch(batch)
    if kernel >= 2 and w.dtype != "bf16":
        pytest.skip("the tensor-core kernels take bf16")
    if kernel >= 3 and row_blocks(w) % 2:
        pytest.skip("the two-tile and CTA-pair kernels need an even number of 128-row blocks")
    x = gi.make_inputs(w, with_accept=False)
    out = run(ts, x, cuda_device, kernel=kernel)
    assert_attention_close(out, oracle_attention(x), w.dtype)


def test_auto_plan_picks_tensor_cores_for_bf16_head128(ts, cuda_device):
    for name, want in [("c2_llama3_8b_bf16_greedy", 2), ("c3_llama2_7b_bf16_stoch", 2),
                       ("c4_llama3_70b_bf16_greedy", 5), ("c5_ragged_b64_bf16_stoch", 2),
                       ("c1_tiny_f32_greedy", 1)]:
        w = gen.get(name)
        prob = ts.AttnProblem(w.batch, w.num_nodes, w.num_q_heads, w.num_kv_heads, w.head_dim, 16, 64, 100,
                              ts.DTYPE_BF16 if w.dtype == "bf16" else ts.DTYPE_F32)
        assert ts.attn_plan(prob).kernel == want, name


@pytest.mark.parametrize("kernel", [1, 2, 3, 4])
@pytest.mark.parametrize("splits", [1, 3, 40])
def test_split_counts(ts, cuda_device, kernel, splits):
    w = gen.get("c2_llama3_8b_bf16_greedy") if kernel < 3 else gen.get("c4_llama3_70b_bf16_greedy").with_batch(1)
    x = gi.make_inputs(w, with_accept=False)
    out = run(ts, x, cuda_device, kernel=kernel, num_splits=splits)
    assert_attention_close(out, oracle_attention(x), w.dtype)


def _custom(name, parents, prefix, batch=None):
    w = gen.get(name)
    parents = np.asarray(parents, dtype=np.int32)
    w = w.with_batch(batch or parents.shape[0])
    from dataclasses import replace
    w = replace(w, num_nodes=parents.shape[1])
    return w, gi.make_inputs(w, parents=parents, prefix_lens=np.asarray(prefix, dtype=np.int32),
                             with_accept=False)


@pytest.mark.parametrize("dtype_cfg,kernel", [("c1_tiny_f32_greedy", 1), ("c2_llama3_8b_bf16_greedy", 1),
                                              ("c2_llama3_8b_bf16_greedy", 2), ("c4_llama3_70b_bf16_greedy", 2),
                                              ("c4_llama3_70b_bf16_greedy", 3), ("c4_llama3_70b_bf16_greedy", 4),
                                              ("c4_llama3_70b_bf16_greedy", 5)])
@pytest.mark.parametrize("case", ["single_node", "prefix0", "ragged_tail", "chain64", "star64",
                                  "random64", "random32", "chain128", "star128", "random128", "random100"])
def test_edge_cases(ts, cuda_device, dtype_cfg, kernel, case):
    rng = np.random.default_rng(hash(case) % 2**32)
    if case == "single_node":
        parents, prefix = [[-1], [-1]], [37, 0]
    elif case == "prefix0":
        parents, prefix = [trees.random_recursive(rng, 9)], [0]
    elif case == "ragged_tail":
        parents, prefix = [trees.random_recursive(rng, 11), trees.chain(11)], [17, 301]
    elif case == "chain64":
        parents, prefix = [trees.chain(64)], [129]
    elif case == "star64":
        parents, prefix = [trees.star(64)], [40]
    elif case == "random32":
        parents, prefix = [trees.random_recursive(rng, 32), trees.random_recursive(rng, 32)], [700, 3]
    elif case == "chain128":                       # trees past 64 nodes: two ancestor words per node
        parents, prefix = [trees.chain(128)], [300]
    elif case == "star128":
        parents, prefix = [trees.star(128)], [77]
    elif case == "random128":
        parents, prefix = [trees.random_recursive(rng, 128), trees.random_recursive(rng, 128)], [0, 517]
    elif case == "random100":
        parents, prefix = [trees.random_recursive(rng, 100)], [129]
    else:
        parents, prefix = [trees.random_recursive(rng, 64), trees.random_recursive(rng, 64)], [5, 999]
    w, x = _custom(dtype_cfg, parents, prefix)
    if kernel >= 3 and row_blocks(w) % 2:
        pytest.skip("the two-tile and CTA-pair kernels need an even number of 128-row blocks")
    out = run(ts, x, cuda_device, kernel=kernel)
    assert_attention_close(out, oracle_attention(x), w.dtype)


def test_bad_parents_and_lengths_are_flagged(ts, cuda_device):
    w = gen.get("c2_llama3_8b_bf16_greedy").with_batch(2)
    x = gi.make_inputs(w, with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    bad_parents = d["tree_parents"].clone()
    bad_parents[0, 3] = 5                          # not an earlier node
    ws = torch.empty(ts.attn_workspace_bytes(ts.attn_problem(d["q"], d["k_pages"], d["page_table"])),
                     dtype=torch.uint8, device=cuda_device)
    ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["prefix_lens"], bad_parents,
                        workspace=ws)
    assert ts.read_status(ws) & 1
    bad_len = d["prefix_lens"].clone()
    bad_len[1] = 10 ** 6
    out = ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], d["page_table"], bad_len,
                              d["tree_parents"], workspace=ws)
    assert ts.read_status(ws) & 4
    assert torch.all(out[1] == 0)
    out = ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["prefix_lens"],
                              d["tree_parents"], workspace=ws)
    assert ts.read_status(ws) == 0
    assert_attention_close(out, oracle_attention(x), w.dtype)


def test_bad_page_id_is_flagged_not_read(ts, cuda_device):
    w = gen.get("c1_tiny_f32_greedy")
    x = gi.make_inputs(w, with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    d["page_table"][0, 1] = 1 << 30
    ws = torch.empty(ts.attn_workspace_bytes(ts.attn_problem(d["q"], d["k_pages"], d["page_table"])),
                     dtype=torch.uint8, device=cuda_device)
    ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["prefix_lens"],
                        d["tree_parents"], workspace=ws)
    assert ts.read_status(ws) & 2


def full_size_pairs(w, n, seed):
    """n (sequence, kv head) pairs: the first and the last sequence and head, the rest drawn
    at random.  Every pair covers all of its kv head's row blocks (all N * G rows)."""
    rng = np.random.default_rng(seed)
    pairs = {(0, 0), (w.batch - 1, w.num_kv_heads - 1), (0, w.num_kv_heads - 1), (w.batch - 1, 0)}
    while len(pairs) < n:
        pairs.add((int(rng.integers(0, w.batch)), int(rng.integers(0, w.num_kv_heads))))
    return sorted(pairs)


def test_full_size_bench_workload_sampled(ts, cuda_device):
    """The bench's workload at full size, in the bench's launch configuration (the automatic
    plan); the oracle checks 16 (sequence, kv head) pairs, each over all four row blocks."""
    from oracle_pool import oracle_attention_pairs
    name = "c4_llama3_70b_bf16_greedy"
    w = gen.get(name)
    x = gi.make_inputs(w, with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    assert ts.attn_plan(ts.attn_problem(d["q"], d["k_pages"], d["page_table"])).kernel == ts.KERNEL_TC_STREAM
    out = run(ts, x, cuda_device)
    pairs = full_size_pairs(w, 16, 0)
    ref = oracle_attention_pairs(name, pairs, workers=8)
    mask = ~np.isnan(ref)
    assert mask.sum() == len(pairs) * w.num_nodes * w.group * w.head_dim
    assert_attention_close(out, ref, w.dtype, mask=mask)
    assert torch.isfinite(out.float()).all()


def test_batch8_automatic_plan_in_full(ts, cuda_device):
    """The Llama-3-70B shape at batch 8 through the automatic plan (the CTA-pair kernel),
    every (sequence, kv head) pair against the oracle."""
    from oracle_pool import oracle_attention_pairs
    name = "c4_llama3_70b_bf16_greedy@b8"
    w = gen.get(name)
    x = gi.make_inputs(w, with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    plan = ts.attn_plan(ts.attn_problem(d["q"], d["k_pages"], d["page_table"]))
    assert plan.kernel == ts.KERNEL_TC_2SM
    out = run(ts, x, cuda_device)
    pairs = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    ref = oracle_attention_pairs(name, pairs, workers=16)
    assert_attention_close(out, ref, w.dtype)


@pytest.mark.parametrize("kernel", [0, 1, 2])
def test_llama2_mha_at_its_full_batch(ts, cuda_device, kernel):
    """The Llama-2-7B shape (32 q / 32 kv heads, 16 nodes) at its batch of 8, in full."""
    w = gen.get("c3_llama2_7b_bf16_stoch")
    assert w.batch == 8
    x = gi.make_inputs(w, with_accept=False)
    out = run(ts, x, cuda_device, kernel=kernel)
    assert_attention_close(out, oracle_attention(x), w.dtype)


def test_full_size_ragged_sampled(ts, cuda_device):
    w = gen.get("c5_ragged_b64_bf16_stoch")
    x = gi.make_inputs(w, with_accept=False)
    out = run(ts, x, cuda_device)
    order = np.argsort(x.prefix_lens)
    pairs = [(int(order[0]), 0), (int(order[-1]), 7), (int(order[len(order) // 2]), 3)]
    ref = oracle_attention(x, pairs)
    mask = ~np.isnan(ref)
    assert_attention_close(out, ref, w.dtype, mask=mask)
    assert torch.isfinite(out.float()).all()


def test_two_tile_kernel_refuses_an_odd_number_of_row_blocks(ts, cuda_device):
    w = gen.get("c2_llama3_8b_bf16_greedy")           # 8 nodes x 4 query heads: one 128-row block
    x = gi.make_inputs(w, with_accept=False)
    with pytest.raises((ValueError, ts.TreespecError)):
        run(ts, x, cuda_device, kernel=ts.KERNEL_TC_PAIR)


@pytest.mark.parametrize("kernel", [1, 2, 3, 4, 5])
def test_full_size_every_kernel_on_sampled_pairs(ts, cuda_device, kernel):
    """Every attention kernel on the full bench workload, checked on sampled pairs."""
    w = gen.get("c4_llama3_70b_bf16_greedy")
    x = gi.make_inputs(w, with_accept=False)
    out = run(ts, x, cuda_device, kernel=kernel)
    pairs = [(0, 0), (w.batch - 1, w.num_kv_heads - 1), (w.batch // 2, 3)]
    ref = oracle_attention(x, pairs)
    mask = ~np.isnan(ref)
    assert_attention_close(out, ref, w.dtype, mask=mask)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("kernel", [2, 3, 4, 5])
@pytest.mark.parametrize("splits", [1, 0])
def test_tensor_core_kernels_flag_bad_lengths_and_pages(ts, cuda_device, kernel, splits):
    """An invalid sequence gets zero rows (written by the kernel itself with one split, by
    the merge otherwise) and the other sequences stay exact; a bad page id is flagged."""
    w = gen.get("c4_llama3_70b_bf16_greedy").with_batch(2)
    x = gi.make_inputs(w, with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    prob = ts.attn_problem(d["q"], d["k_pages"], d["page_table"], kernel=kernel, num_splits=splits)
    assert ts.attn_plan(prob).kernel == kernel
    ws = torch.empty(ts.attn_workspace_bytes(prob), dtype=torch.uint8, device=cuda_device)
    bad_len = d["prefix_lens"].clone()
    bad_len[1] = 10 ** 6
    out = ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], d["page_table"], bad_len, d["tree_parents"],
                              kernel=kernel, num_splits=splits, workspace=ws)
    torch.cuda.synchronize()
    assert ts.read_status(ws) & 4
    assert torch.all(out[1] == 0)
    ref = oracle_attention(x, [(0, 0), (0, 5)])
    mask = ~np.isnan(ref)
    mask[1] = False
    assert_attention_close(out, ref, w.dtype, mask=mask)
    bad_pages = d["page_table"].clone()
    bad_pages[0, 3] = 1 << 30
    ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], bad_pages, d["prefix_lens"], d["tree_parents"],
                        kernel=kernel, num_splits=splits, workspace=ws)
    torch.cuda.synchronize()
    assert ts.read_status(ws) & 2


@pytest.mark.parametrize("batch,prefix", [(1, [8192]), (2, [8192, 0]), (3, [300, 5000, 17]), (5, [64, 1, 4096, 2048, 63])])
def test_persistent_kernel_cuts_units_into_pieces(ts, cuda_device, batch, prefix):
    """Few sequences on 152 SMs: every (sequence, kv head, row-block pair) unit is cut into
    several pieces whose partials the last piece merges; ragged lengths move the cuts."""
    w = gen.get("c4_llama3_70b_bf16_greedy")
    rng = np.random.default_rng(batch)
    parents = np.stack([trees.random_recursive(rng, w.num_nodes) for _ in range(batch)])
    w2, x = _custom("c4_llama3_70b_bf16_greedy", parents, prefix)
    out = run(ts, x, cuda_device, kernel=ts.KERNEL_TC_STREAM)
    assert_attention_close(out, oracle_attention(x), w2.dtype)
    out2 = run(ts, x, cuda_device, kernel=ts.KERNEL_TC_STREAM)          # counters reset for the next call
    assert torch.equal(out, out2)


def test_persistent_kernel_with_every_sequence_invalid(ts, cuda_device):
    w = gen.get("c4_llama3_70b_bf16_greedy").with_batch(3)
    x = gi.make_inputs(w, with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    prob = ts.attn_problem(d["q"], d["k_pages"], d["page_table"], kernel=ts.KERNEL_TC_STREAM)
    ws = torch.empty(ts.attn_workspace_bytes(prob), dtype=torch.uint8, device=cuda_device)
    out = torch.full_like(d["q"], 7.0)
    bad = torch.full_like(d["prefix_lens"], 10 ** 6)
    ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], d["page_table"], bad, d["tree_parents"], out,
                        kernel=ts.KERNEL_TC_STREAM, workspace=ws)
    torch.cuda.synchronize()
    assert ts.read_status(ws) & 4
    assert torch.all(out == 0)
