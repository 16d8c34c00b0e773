"""GPU parity of tree_kv_commit against the oracle (through the C-ABI): pools bit-exact."""
import numpy as np
import pytest
import torch

import gen
from gen import inputs as gi
from gen import trees
from oracle import kv_commit as okc

from gpu_util import dev_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import __graft_entry__
    __graft_entry__.build()
    import eagle_speculative_tree_gb300 as mod
    return mod


def random_paths(parents: np.ndarray, seed: int, stop_prob: float = 0.2):
    rng = np.random.default_rng(seed)
    B, N = parents.shape
    path = np.full((B, N), -1, dtype=np.int32)
    lens = np.zeros(B, dtype=np.int32)
    for b in range(B):
        p = trees.random_root_path(parents[b], rng, stop_prob)
        path[b, :len(p)] = p
        lens[b] = len(p)
    return path, lens


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.cpu()
    return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)).numpy()


def run_both(ts, x, device, path, lens, prefix_lens=None, page_table=None):
    bf = x.workload.dtype == "bf16"
    pl = x.prefix_lens if prefix_lens is None else prefix_lens
    pt = x.page_table if page_table is None else page_table
    k = dev_tensor(x.k_pages, device, bf)
    v = dev_tensor(x.v_pages, device, bf)
    ws = torch.empty(ts.commit_workspace_bytes(), dtype=torch.uint8, device=device)
    new = ts.tree_kv_commit(k, v, dev_tensor(pt, device), dev_tensor(pl, device), dev_tensor(path, device),
                            dev_tensor(lens, device), workspace=ws)
    st = ts.read_status(ws)
    k2, v2, want_lens, want_st = okc.kv_commit(x.k_pages, x.v_pages, pt, pl, path, lens, x.workload.num_nodes)
    view = np.int16 if bf else np.int32
    assert np.array_equal(bits(k), k2.view(view)), "K pool differs from the oracle"
    assert np.array_equal(bits(v), v2.view(view)), "V pool differs from the oracle"
    assert new.cpu().numpy().tolist() == want_lens.tolist()
    return st, want_st


@pytest.mark.parametrize("name,batch", [("c1_tiny_f32_greedy", None), ("c2_llama3_8b_bf16_greedy", None),
                                        ("c3_llama2_7b_bf16_stoch", 2), ("c4_llama3_70b_bf16_greedy", 2),
                                        ("c5_ragged_b64_bf16_stoch", 4)])
@pytest.mark.parametrize("seed", [0, 1])
def test_commit_matches_oracle(ts, cuda_device, name, batch, seed):
    w = gen.get(name if batch is None else f"{name}@b{batch}")
    x = gi.make_inputs(w, with_accept=False)
    path, lens = random_paths(x.tree_parents, seed)
    st, want = run_both(ts, x, cuda_device, path, lens)
    assert st == 0 and want == 0


@pytest.mark.parametrize("shape", ["chain64", "star64", "random64", "chain128", "random128"])
def test_commit_edge_trees(ts, cuda_device, shape):
    from dataclasses import replace
    n = int(shape[-3:]) if shape.endswith("128") else 64
    make = {"chain": lambda r: trees.chain(n), "star": lambda r: trees.star(n),
            "random": lambda r: trees.random_recursive(r, n)}[shape.rstrip("0123456789")]
    rng = np.random.default_rng(5)
    parents = np.stack([make(rng) for _ in range(3)]).astype(np.int32)
    w = replace(gen.get("c2_llama3_8b_bf16_greedy").with_batch(3), num_nodes=n)
    x = gi.make_inputs(w, parents=parents, prefix_lens=np.array([0, 15, 200], dtype=np.int32), with_accept=False)
    path, lens = random_paths(x.tree_parents, 3, stop_prob=0.0)     # walk to a leaf
    if shape.startswith("chain"):
        assert lens.tolist() == [n - 1] * 3                         # the whole chain: nothing moves
    st, want = run_both(ts, x, cuda_device, path, lens)
    assert st == 0 and want == 0


def test_commit_empty_paths(ts, cuda_device):
    x = gi.make_inputs(gen.get("c1_tiny_f32_greedy"), with_accept=False)
    B, N = x.tree_parents.shape
    st, _ = run_both(ts, x, cuda_device, np.full((B, N), -1, np.int32), np.zeros(B, np.int32))
    assert st == 0


def test_commit_rejects_bad_inputs_without_moving(ts, cuda_device):
    x = gi.make_inputs(gen.get("c2_llama3_8b_bf16_greedy@b4"), with_accept=False)
    B, N = x.tree_parents.shape
    path, lens = random_paths(x.tree_parents, 7, stop_prob=0.0)
    pl = x.prefix_lens.copy()
    pt = x.page_table.copy()
    path[0, :2] = [3, 3]                          # not increasing
    lens[1] = N                                   # too many nodes
    pl[2] = -5                                    # bad prefix length
    pt[3, (pl[3] + 1) // 16] = x.num_pool_pages + 7   # a destination page outside the pool
    st, want = run_both(ts, x, cuda_device, path, lens, prefix_lens=pl, page_table=pt)
    assert st == want and st & okc.BAD_PATH and st & okc.BAD_LENGTH and st & okc.BAD_PAGE


def test_commit_of_a_padded_tree_near_the_end_of_its_pages(ts, cuda_device):
    """A 5-node tree padded to the batch's 64 nodes, its prefix placed so that S + 64 runs
    past its page table while S + 5 fits: the accepted path commits (bound S + 1 +
    max(path)), bit-exact against the oracle, beside a full 64-node tree."""
    from dataclasses import replace
    rng = np.random.default_rng(11)
    w = replace(gen.get("c2_llama3_8b_bf16_greedy").with_batch(2), num_nodes=64)
    parents = trees.padded([trees.random_recursive(rng, 64), trees.chain(5)], 64)
    prefix = np.array([100, 170], dtype=np.int32)
    x = gi.make_inputs(w, parents=parents, prefix_lens=prefix, with_accept=False)
    table = np.ascontiguousarray(x.page_table[:, :11])       # 176 slots: 100 + 64 and 170 + 5 fit, 170 + 64 not
    path = np.full((2, 64), -1, dtype=np.int32)
    lens = np.zeros(2, dtype=np.int32)
    p0 = trees.random_root_path(parents[0], rng, 0.0)
    path[0, :len(p0)], lens[0] = p0, len(p0)
    path[1, :4], lens[1] = [1, 2, 3, 4], 4                    # touches positions 170 .. 174
    st, want = run_both(ts, x, cuda_device, path, lens, page_table=table)
    assert st == 0 and want == 0
    prefix2 = prefix.copy()
    prefix2[1] = 172                                          # now node 4 would sit at 176: past the table
    st, want = run_both(ts, x, cuda_device, path, lens, prefix_lens=prefix2, page_table=table)
    assert st == want and st & okc.BAD_LENGTH
