"""GPU parity of tree_draft_step / tree_rerank against the oracle (through the C-ABI): exact."""
import numpy as np
import pytest
import torch

from gen import draft as gd
from oracle import draft_tree as odt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import __graft_entry__
    __graft_entry__.build()
    import eagle_speculative_tree_gb300 as mod
    return mod


def build_both(ts, device, B, V, k, steps, N, seed, ties=False):
    M = odt.num_nodes_after(steps, k)
    lps = [gd.draft_logprobs(seed * 100 + s, B, 1 if s == 0 else k, V, ties=ties) for s in range(steps)]
    # GPU
    par = torch.zeros((B, M), dtype=torch.int32, device=device)
    tok = torch.zeros((B, M), dtype=torch.int32, device=device)
    sc = torch.zeros((B, M), dtype=torch.float32, device=device)
    status = 0
    front = None
    fronts = []
    for s, lp in enumerate(lps):
        front, ws = ts.tree_draft_step(torch.from_numpy(lp).to(device), s, k, front, par, tok, sc)
        status |= ts.read_status(ws)
        fronts.append(front.cpu().numpy())
    wsr = torch.empty(256, dtype=torch.uint8, device=device)
    gp, gt = ts.tree_rerank(par, tok, sc, N, workspace=wsr)
    status |= ts.read_status(wsr)
    # oracle
    opar = np.zeros((B, M), np.int32)
    otok = np.zeros((B, M), np.int32)
    osc = np.zeros((B, M), np.float32)
    ofront = np.zeros((B, 1), np.int32)
    for s, lp in enumerate(lps):
        ofront = odt.draft_step(lp, ofront, opar, otok, osc, s, k)
        assert np.array_equal(fronts[s], ofront), f"frontier of step {s} differs"
    op, ot, ost = odt.rerank(opar, otok, osc, N)
    assert np.array_equal(par.cpu().numpy(), opar), "node parents differ"
    assert np.array_equal(tok.cpu().numpy(), otok), "node tokens differ"
    assert np.array_equal(sc.cpu().numpy().view(np.int32), osc.view(np.int32)), "node scores differ"
    assert np.array_equal(gp.cpu().numpy(), op) and np.array_equal(gt.cpu().numpy(), ot)
    return status, ost


@pytest.mark.parametrize("B,V,k,steps,N", [
    (1, 256, 2, 3, 8),          # tiny
    (4, 32000, 4, 3, 16),       # Llama-2 vocabulary
    (2, 128256, 8, 6, 64),      # Llama-3 vocabulary, the 64-node tree
    (3, 1001, 16, 2, 24),       # scalar loads (V % 4 != 0), the largest branching
    (2, 5003, 1, 7, 8),         # topk 1: the greedy chain
    (2, 32000, 8, 6, 128),      # a 128-node tree: two ancestor words per node downstream
    (32, 128256, 8, 2, 64),     # 256 frontier rows of the Llama-3 vocabulary, one part each
    (8, 128256, 8, 2, 64),      # 64 such rows, two parts each
])
@pytest.mark.parametrize("ties", [False, True])
def test_draft_tree_matches_oracle(ts, cuda_device, B, V, k, steps, N, ties):
    st, ost = build_both(ts, cuda_device, B, V, k, steps, N, seed=V + k, ties=ties)
    assert st == 0 and ost == 0


def test_rerank_flags_bad_parents(ts, cuda_device):
    par = torch.tensor([[-1, 0, 5, 1]], dtype=torch.int32, device=cuda_device)   # node 2's parent is after it
    tok = torch.tensor([[-1, 7, 8, 9]], dtype=torch.int32, device=cuda_device)
    sc = torch.tensor([[0, -1.0, -2.0, -3.0]], dtype=torch.float32, device=cuda_device)
    ws = torch.empty(256, dtype=torch.uint8, device=cuda_device)
    p, t = ts.tree_rerank(par, tok, sc, 4, workspace=ws)
    assert ts.read_status(ws) & 1
    assert p.cpu().numpy().tolist() == [[-1, 0, 0, 1]] and t.cpu().numpy().tolist() == [[-1, 7, 8, 9]]


def test_rows_without_enough_values_are_flagged(ts, cuda_device):
    lp = torch.full((1, 1, 64), float("nan"), device=cuda_device)
    lp[0, 0, 5] = -1.0                                 # one usable value, topk 2
    par = torch.zeros((1, 5), dtype=torch.int32, device=cuda_device)
    tok = torch.zeros_like(par)
    sc = torch.zeros((1, 5), dtype=torch.float32, device=cuda_device)
    _front, ws = ts.tree_draft_step(lp, 0, 2, None, par, tok, sc)
    assert ts.read_status(ws) & 8


@pytest.mark.parametrize("name", ["c1_tiny_f32_greedy", "c2_llama3_8b_bf16_greedy", "c3_llama2_7b_bf16_stoch",
                                  "c4_llama3_70b_bf16_greedy", "c5_ragged_b64_bf16_stoch"])
def test_entry_points_rebuild_the_generator_trees(ts, cuda_device, name):
    """tree_draft_step x steps + the rerank, fed the generator's own child log-probabilities
    (placed at random token ids of a 1000-token row, the rest far below), rebuild the
    parent arrays gen.trees.build_tree makes for every workload: the rerank takes the
    beam nodes (the union of the steps' frontiers) where the recipe's steps * topk >=
    N - 1 -- c2's 20 candidates -- and every candidate otherwise."""
    import gen
    from gen import inputs as gi, trees
    w = gen.get(name)
    k, steps, N, V = w.topk, w.num_steps, w.num_nodes, 1000
    M = odt.num_nodes_after(steps, k)
    for b in range(min(w.batch, 4) if w.vary_tree else 1):
        want = trees.build_tree(gi.rng_for(w, b, gi.TREE), steps, k, N)
        rng = gi.rng_for(w, b, gi.TREE)
        place = np.random.default_rng(1234 + b)
        par = torch.zeros((1, M), dtype=torch.int32, device=cuda_device)
        tok = torch.zeros_like(par)
        sc = torch.zeros((1, M), dtype=torch.float32, device=cuda_device)
        front, fronts = None, []
        for s in range(steps):
            F = 1 if s == 0 else k
            rows = np.full((1, F, V), -1e30, np.float32)
            for f in range(F):                       # draws in frontier order, as the generator expands
                rows[0, f, place.choice(V, size=k, replace=False)] = trees._child_logprobs(rng, k).astype(np.float32)
            front, ws = ts.tree_draft_step(torch.from_numpy(rows).to(cuda_device), s, k, front, par, tok, sc)
            assert ts.read_status(ws) == 0
            fronts.append(front)
        pool = torch.cat(fronts, dim=1) if steps * k >= N - 1 else None
        gp, _gt = ts.tree_rerank(par, tok, sc, N, pool=pool)
        assert gp.cpu().numpy()[0].tolist() == want.tolist(), (name, b)


@pytest.mark.parametrize("pool_size", [1, 5, 20, 200])
def test_rerank_pool_matches_oracle(ts, cuda_device, pool_size):
    """Random pools, with duplicates and ids out of range, some smaller than N - 1 (the tree
    is then padded): GPU and oracle agree exactly."""
    B, V, k, steps, N = 3, 5003, 4, 4, 16
    M = odt.num_nodes_after(steps, k)
    lps = [gd.draft_logprobs(900 + s, B, 1 if s == 0 else k, V) for s in range(steps)]
    par = torch.zeros((B, M), dtype=torch.int32, device=cuda_device)
    tok = torch.zeros_like(par)
    sc = torch.zeros((B, M), dtype=torch.float32, device=cuda_device)
    front = None
    for s, lp in enumerate(lps):
        front, _ws = ts.tree_draft_step(torch.from_numpy(lp).to(cuda_device), s, k, front, par, tok, sc)
    rng = np.random.default_rng(pool_size)
    pool = rng.integers(-3, M + 3, size=(B, pool_size)).astype(np.int32)
    wsr = torch.empty(256, dtype=torch.uint8, device=cuda_device)
    gp, gt = ts.tree_rerank(par, tok, sc, N, pool=torch.from_numpy(pool).to(cuda_device), workspace=wsr)
    st = ts.read_status(wsr)
    op, ot, ost = odt.rerank(par.cpu().numpy(), tok.cpu().numpy(), sc.cpu().numpy(), N, pool=pool)
    assert np.array_equal(gp.cpu().numpy(), op) and np.array_equal(gt.cpu().numpy(), ot)
    assert st == ost
