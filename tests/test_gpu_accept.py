"""GPU parity of tree_accept against the oracle: bit-exact paths, lengths and bonus tokens."""
import numpy as np
import pytest
import torch
from scipy import special, stats

import gen
from gen import inputs as gi
from gen import mc, trees

from gpu_util import accept_device_inputs, compare_accept, dev_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import __graft_entry__
    __graft_entry__.build()
    import eagle_speculative_tree_gb300 as mod
    return mod


def run(ts, x, device, mode=0):
    d = accept_device_inputs(x, device)
    res = ts.tree_accept(d["target_logits"], d["draft_tokens"], d["draft_probs"], d["tree_parents"],
                         d["uniforms"], x.temperature, mode=mode)
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("name", ["c1_tiny_f32_greedy", "c2_llama3_8b_bf16_greedy",
                                  "c3_llama2_7b_bf16_stoch", "c4_llama3_70b_bf16_greedy",
                                  "c4_llama3_70b_bf16_t0.7", "c5_ragged_b64_bf16_stoch"])
def test_configs_full_size(ts, cuda_device, name, mode):
    w = gen.get(name)
    x = gi.make_inputs(w, with_attention=False)
    res = run(ts, x, cuda_device, mode)
    n, ties, flipped = compare_accept(res, x.target_logits, x.draft_tokens, x.draft_probs, x.tree_parents,
                                      x.uniforms, x.temperature)
    print(f"{name}: {n} sequences, {ties} with a decision within the rounding margin, {flipped} took the "
          f"other side")
    # compare_accept fails any difference outside the float32 bound; on these seeds only
    # c5 sequence 54 (bonus draw margin 6.9e-9 of the mass) may take the adjacent token
    assert flipped <= (1 if name == "c5_ragged_b64_bf16_stoch" else 0)


def _small(B, N, V, parents, temperature, seed, tied=False, dup=False):
    rng = np.random.default_rng(seed)
    logits = rng.normal(0, 3, (B, N, V)).astype(np.float32)
    if tied:
        logits = np.round(logits).astype(np.float32)          # many exact ties
    parents = np.broadcast_to(np.asarray(parents, dtype=np.int32), (B, N)).copy()
    if temperature == 0:
        tokens = rng.integers(0, V, (B, N)).astype(np.int32)
        am = logits.argmax(-1)
        hit = rng.random((B, N)) < 0.7
        tokens = np.where(hit, am[np.arange(B)[:, None], parents.clip(0)], tokens).astype(np.int32)
        tokens[:, 0] = 0
        return logits, tokens, None, parents, None
    q = special.softmax(logits.astype(np.float64) + rng.normal(0, 1, (B, N, V)), axis=-1).astype(np.float32)
    tokens = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        for c in range(1, N):
            row = q[b, parents[b, c]].astype(np.float64)
            tokens[b, c] = min(int(np.searchsorted(np.cumsum(row), rng.random() * row.sum())), V - 1)
        if dup and N > 2:
            tokens[b, 2] = tokens[b, 1]
    u = rng.random((B, N)).astype(np.float32)
    return logits, tokens, q, parents, u


def _run_small(ts, device, logits, tokens, q, parents, u, T, mode=0):
    res = ts.tree_accept(dev_tensor(logits, device), dev_tensor(tokens, device),
                         None if q is None else dev_tensor(q, device), dev_tensor(parents, device),
                         None if u is None else dev_tensor(u, device), T, mode=mode)
    torch.cuda.synchronize()
    return compare_accept(res, logits, tokens, q, parents, u, T)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("T", [0.0, 1.0, 0.05, 20.0])
@pytest.mark.parametrize("shape", ["root_only", "chain64", "star64", "random64", "mtp", "chain128", "star128",
                                   "random128"])
@pytest.mark.parametrize("V", [7, 256, 5003, 40000])
def test_edge_shapes(ts, cuda_device, T, shape, V, mode):
    rng = np.random.default_rng(V)
    parents = {"root_only": [-1], "chain64": trees.chain(64), "star64": trees.star(64),
               "random64": trees.random_recursive(rng, 64), "mtp": [-1, 0], "chain128": trees.chain(128),
               "star128": trees.star(128), "random128": trees.random_recursive(rng, 128)}[shape]
    N = len(parents)
    data = _small(16 if V < 40000 else 4, N, V, parents, T, seed=V + N)
    n, ties, flipped = _run_small(ts, cuda_device, *data, T, mode)
    print(f"{shape} V={V} T={T}: {n} sequences, {ties} within the rounding margin, {flipped} took the other side")
    assert flipped == 0


@pytest.mark.parametrize("mode", [1, 2])
def test_greedy_ties_take_lowest_id(ts, cuda_device, mode):
    data = _small(64, 16, 64, trees.random_recursive(np.random.default_rng(1), 16), 0.0, seed=3, tied=True)
    _run_small(ts, cuda_device, *data, 0.0, mode)


@pytest.mark.parametrize("mode", [1, 2])
def test_duplicate_sibling_tokens(ts, cuda_device, mode):
    parents = [-1, 0, 0, 0, 1, 2, 3]
    data = _small(256, 7, 300, parents, 1.0, seed=4, dup=True)
    _run_small(ts, cuda_device, *data, 1.0, mode)


@pytest.mark.parametrize("mode", [1, 2])
def test_zero_draft_probability(ts, cuda_device, mode):
    logits, tokens, q, parents, u = _small(64, 5, 64, [-1, 0, 0, 1, 1], 1.0, seed=5)
    q[:, :, ::2] = 0.0
    q /= q.sum(-1, keepdims=True)
    _run_small(ts, cuda_device, logits, tokens, q, parents, u, 1.0, mode)


@pytest.mark.parametrize("mode", [1, 2])
def test_bad_tokens_are_flagged(ts, cuda_device, mode):
    logits, tokens, q, parents, u = _small(4, 5, 64, [-1, 0, 0, 1, 1], 0.0, seed=6)
    tokens[0, 1] = 64
    tokens[1, 2] = -3
    ws = torch.empty(ts.accept_workspace_bytes(4, 5, 64), dtype=torch.uint8, device=cuda_device)
    ts.tree_accept(dev_tensor(logits, cuda_device), dev_tensor(tokens, cuda_device), None,
                   dev_tensor(parents, cuda_device), None, 0.0, mode=mode, workspace=ws)
    assert ts.read_status(ws) & 8


@pytest.mark.parametrize("mode", [1, 2])
def test_bad_parents_are_flagged(ts, cuda_device, mode):
    logits, tokens, q, parents, u = _small(4, 5, 64, [-1, 0, 0, 1, 1], 0.0, seed=7)
    parents[2, 3] = 4
    ws = torch.empty(ts.accept_workspace_bytes(4, 5, 64), dtype=torch.uint8, device=cuda_device)
    ts.tree_accept(dev_tensor(logits, cuda_device), dev_tensor(tokens, cuda_device), None,
                   dev_tensor(parents, cuda_device), None, 0.0, mode=mode, workspace=ws)
    assert ts.read_status(ws) & 1


@pytest.mark.parametrize("mode", [1, 2])
def test_monte_carlo_invariance_on_gpu(ts, cuda_device, mode):
    """2^20 trials of the vocab-8 tree: emitted tokens follow p_root then p(. | first)."""
    tables = mc.mc_tables(11)
    trials = 1 << 20
    logits, q, tokens, uniforms, parents = mc.mc_trials(tables, trials, 12)
    path, length, bonus = ts.tree_accept(dev_tensor(logits, cuda_device), dev_tensor(tokens, cuda_device),
                                         dev_tensor(q, cuda_device), dev_tensor(parents, cuda_device),
                                         dev_tensor(uniforms, cuda_device), 1.0, mode=mode)
    path, length, bonus = path.cpu().numpy(), length.cpu().numpy(), bonus.cpu().numpy()
    rows = np.arange(trials)
    first = np.where(length >= 1, tokens[rows, path[:, 0].clip(0)], bonus)
    second = np.where(length >= 2, tokens[rows, path[:, 1].clip(0)], np.where(length == 1, bonus, -1))
    V = mc.MC_VOCAB
    p_root = special.softmax(tables.root_logits.astype(np.float64))
    c1 = np.bincount(first, minlength=V)
    assert stats.chisquare(c1, c1.sum() * p_root).pvalue > 1e-3
    stat, dof = 0.0, 0
    for x in range(V):
        sel = (first == x) & (second >= 0)
        cnt = np.bincount(second[sel], minlength=V)
        exp = sel.sum() * special.softmax(tables.d1_logits[x].astype(np.float64))
        stat += float(((cnt - exp) ** 2 / exp).sum())
        dof += V - 1
    assert stats.chi2.sf(stat, dof) > 1e-3


@pytest.mark.parametrize("name", ["c2_llama3_8b_bf16_greedy", "c3_llama2_7b_bf16_stoch@b2",
                                  "c4_llama3_70b_bf16_t0.7@b2"])
@pytest.mark.parametrize("mode", [1, 2])
def test_rows_in_pinned_host_memory_match_device_rows(ts, cuda_device, name, mode):
    x = gi.make_inputs(gen.get(name), with_attention=False)
    d = accept_device_inputs(x, cuda_device)
    want = ts.tree_accept(d["target_logits"], d["draft_tokens"], d["draft_probs"], d["tree_parents"],
                          d["uniforms"], x.temperature, mode=mode)
    host_lg = torch.from_numpy(np.ascontiguousarray(x.target_logits)).pin_memory()
    host_q = None if x.draft_probs is None else torch.from_numpy(np.ascontiguousarray(x.draft_probs)).pin_memory()
    got = ts.tree_accept(host_lg, d["draft_tokens"], host_q, d["tree_parents"], d["uniforms"], x.temperature,
                         mode=mode)
    torch.cuda.synchronize()
    for a, b in zip(got, want):
        assert torch.equal(a, b)
