"""Pins of oracle.draft_tree (beam expansion and rerank; CPU only)."""
import inspect

import numpy as np
import pytest

from oracle import draft_tree as odt


def log_rows(rng, shape, ties=False):
    p = rng.dirichlet(np.ones(shape[-1]) * 0.5, size=shape[:-1])
    lp = np.log(np.maximum(p, 1e-30)).astype(np.float32)
    if ties:                                            # repeated values exercise the tie rules
        lp = np.round(lp * 2) / 2
    return lp


def run_steps(lp_steps, k):
    B = lp_steps[0].shape[0]
    M = odt.num_nodes_after(len(lp_steps), k)
    par = np.zeros((B, M), np.int32)
    tok = np.zeros((B, M), np.int32)
    sc = np.zeros((B, M), np.float32)
    front = np.zeros((B, 1), np.int32)
    fronts = []
    for s, lp in enumerate(lp_steps):
        front = odt.draft_step(lp, front, par, tok, sc, s, k)
        fronts.append(front)
    return par, tok, sc, fronts


@pytest.mark.parametrize("seed,ties", [(0, False), (1, True), (2, True), (3, False)])
def test_step_equals_top_k_over_all_frontier_token_pairs(seed, ties):
    # brute force: no per-node preselection -- rank every (frontier f, token v) pair by
    # (score desc, f, v) and take k; equal to the two-stage rule because a pair in the
    # global top k has at most k-1 better pairs, so it is within its own node's top k
    rng = np.random.default_rng(seed)
    k, V = 3, 7
    lp0 = log_rows(rng, (2, 1, V), ties)
    lp1 = log_rows(rng, (2, k, V), ties)
    par, tok, sc, fronts = run_steps([lp0, lp1], k)
    for b in range(2):
        frontier = fronts[0][b].tolist()                     # step 1 expanded these, in this order
        assert sorted(frontier) == [1, 2, 3]                 # step 0: the root's k children, all kept
        pairs = [(np.float32(sc[b, n] + lp1[b, f, v]), f, v) for f, n in enumerate(frontier) for v in range(V)]
        best = sorted(pairs, key=lambda t: (-float(t[0]), t[1], t[2]))[:k]
        got = [(int(par[b, n]), int(tok[b, n]), sc[b, n]) for n in fronts[1][b]]
        assert got == [(frontier[f], v, s) for s, f, v in best]


def test_topk_one_is_the_greedy_chain():
    rng = np.random.default_rng(7)
    steps = [log_rows(rng, (3, 1, 11)) for _ in range(5)]
    par, tok, sc, _f = run_steps(steps, 1)
    for b in range(3):
        assert par[b].tolist() == [-1, 0, 1, 2, 3, 4]
        assert tok[b, 1:].tolist() == [int(np.argmax(s[b, 0])) for s in steps]
        assert np.isclose(sc[b, -1], sum(float(np.max(s[b, 0])) for s in steps), rtol=1e-5)


def test_rerank_hand_example():
    # root, a(-0.1, root), b(-0.5, root), c(-0.3, a), d(-2.0, b), e(-0.3, c): keep 4 of 5
    # by score: a(-0.1), c(-0.3, index 3), e(-0.3, index 5), b(-0.5); drop d.  Numbered by
    # original index: a->1, b->2, c->3, e->4; parents a:0, b:0, c:1 (a), e:3 (c).
    par = np.array([[-1, 0, 0, 1, 2, 3]], np.int32)
    tok = np.array([[-1, 10, 20, 30, 40, 50]], np.int32)
    sc = np.array([[0, -0.1, -0.5, -0.3, -2.0, -0.3]], np.float32)
    parents, tokens, st = odt.rerank(par, tok, sc, num_nodes=5)
    assert st == 0
    assert parents.tolist() == [[-1, 0, 0, 1, 3]]
    assert tokens.tolist() == [[-1, 10, 20, 30, 50]]


@pytest.mark.parametrize("seed", range(5))
def test_built_trees_are_ancestor_closed_and_scores_are_path_sums(seed):
    rng = np.random.default_rng(seed)
    k, steps, N, V = 4, 5, 40, 9
    lps = [log_rows(rng, (2, 1 if s == 0 else k, V)) for s in range(steps)]
    par, tok, sc, fronts = run_steps(lps, k)
    assert par.shape[1] == 1 + 4 + 4 * 16                  # every scored candidate is a node
    parents, tokens, st = odt.rerank(par, tok, sc, N)
    assert st == 0
    for b in range(2):
        assert parents[b, 0] == -1 and all(0 <= parents[b, i] < i for i in range(1, N))
        # every node's score is the float32 running sum of the log-probs along its path;
        # a node of step s > 0 came from the row of its parent in step s - 1's frontier
        for i in range(1, par.shape[1]):
            chain, n = [], i
            while n > 0:
                chain.append(n)
                n = int(par[b, n])
            s = np.float32(0)
            for depth, n in enumerate(reversed(chain)):
                row = 0 if depth == 0 else fronts[depth - 1][b].tolist().index(int(par[b, n]))
                s = np.float32(s + lps[depth][b, row, tok[b, n]])
            assert s == sc[b, i]


def test_rerank_keeping_everything_is_the_identity():
    rng = np.random.default_rng(11)
    par, tok, sc, _f = run_steps([log_rows(rng, (1, 1, 6)), log_rows(rng, (1, 2, 6))], 2)
    assert par.shape[1] == 7
    parents, tokens, st = odt.rerank(par, tok, sc, num_nodes=7)
    assert st == 0 and parents[0].tolist() == par[0].tolist() and tokens[0].tolist() == tok[0].tolist()


def test_positive_logprobs_can_orphan_and_are_flagged():
    par = np.array([[-1, 0, 1]], np.int32)
    tok = np.array([[-1, 5, 6]], np.int32)
    sc = np.array([[0, -1.0, 2.0]], np.float32)       # the child outscores its parent
    parents, _t, st = odt.rerank(par, tok, sc, num_nodes=2)
    assert st & odt.BAD_PARENT and parents.tolist() == [[-1, 0]]


def test_planted_reversed_ranking_fails_the_brute_force():
    src = inspect.getsource(odt.draft_step).replace("cands.sort(key=lambda t: (-float(t[0]), t[1]))",
                                                    "cands.sort(key=lambda t: (float(t[0]), t[1]))")
    ns = {"np": np, "step_base": odt.step_base}
    exec(src, ns)
    rng = np.random.default_rng(0)
    lp0 = log_rows(rng, (1, 1, 7))
    lp1 = log_rows(rng, (1, 3, 7))
    M = odt.num_nodes_after(2, 3)
    par = np.zeros((1, M), np.int32)
    tok = np.zeros((1, M), np.int32)
    sc = np.zeros((1, M), np.float32)
    f0 = odt.draft_step(lp0, np.zeros((1, 1), np.int32), par, tok, sc, 0, 3)
    f1 = ns["draft_step"](lp1, f0, par, tok, sc, 1, 3)
    frontier = f0[0].tolist()
    pairs = [(np.float32(sc[0, n] + lp1[0, f, v]), f, v) for f, n in enumerate(frontier) for v in range(7)]
    best = sorted(pairs, key=lambda t: (-float(t[0]), t[1], t[2]))[:3]
    assert [(int(par[0, n]), int(tok[0, n])) for n in f1[0]] != [(frontier[f], v) for _s, f, v in best]


def replay_generator_tree(rng, steps, k, n):
    """The draft steps and rerank of this oracle fed the generator's own draws: each
    expanded node's children get the next sorted top-k log-probabilities from `rng`, drawn
    in frontier order (best first), as gen.trees.build_tree draws them.  The rerank takes
    the beam nodes when steps * k >= n - 1 (the generator's candidate set then) and every
    candidate otherwise.  Returns the reranked parent array."""
    from gen import trees
    M = odt.num_nodes_after(steps, k)
    par = np.zeros((1, M), np.int32)
    tok = np.zeros((1, M), np.int32)
    sc = np.zeros((1, M), np.float32)
    front = np.zeros((1, 1), np.int32)
    beam = []
    for s in range(steps):
        F = 1 if s == 0 else k
        rows = np.stack([trees._child_logprobs(rng, k) for _ in range(F)]).astype(np.float32)[None]
        front = odt.draft_step(rows, front, par, tok, sc, s, k)
        beam.extend(front[0].tolist())
    pool = np.asarray([beam]) if steps * k >= n - 1 else None
    parents, _tokens, status = odt.rerank(par, tok, sc, n, pool=pool)
    assert status == 0
    return parents[0]


@pytest.mark.parametrize("name", ["c1_tiny_f32_greedy", "c2_llama3_8b_bf16_greedy", "c3_llama2_7b_bf16_stoch",
                                  "c4_llama3_70b_bf16_greedy", "c5_ragged_b64_bf16_stoch"])
def test_steps_and_rerank_rebuild_the_generator_trees(name):
    """The generator (gen/trees.py) and this oracle state the same drafting reading in code
    of their own (float64 sums there, float32 here): on every workload's seeded tree
    recipe they must produce the same parent arrays, including the 20-candidate beam
    rerank of the 5-step, top-4 recipe."""
    import gen
    from gen import inputs as gi, trees
    w = gen.get(name)
    for b in range(min(w.batch, 8) if w.vary_tree else 1):
        want = trees.build_tree(gi.rng_for(w, b, gi.TREE), w.num_steps, w.topk, w.num_nodes)
        got = replay_generator_tree(gi.rng_for(w, b, gi.TREE), w.num_steps, w.topk, w.num_nodes)
        assert np.array_equal(got, want), (name, b)


def test_pool_restricts_the_rerank():
    # a chain of beam picks: with the pool {1, 4} only those two can be kept; with no pool
    # the best two of all nodes
    par = np.array([[-1, 0, 0, 1, 1]], np.int32)
    tok = np.array([[-1, 10, 11, 12, 13]], np.int32)
    sc = np.array([[0, -1.0, -0.5, -3.0, -2.0]], np.float32)
    p_all, t_all, st = odt.rerank(par, tok, sc, 3)
    assert st == 0 and t_all[0].tolist() == [-1, 10, 11]
    p_pool, t_pool, st = odt.rerank(par, tok, sc, 3, pool=np.array([[1, 4]]))
    assert st == 0 and t_pool[0].tolist() == [-1, 10, 13] and p_pool[0].tolist() == [-1, 0, 1]


def test_small_pool_pads_the_tree():
    par = np.array([[-1, 0, 0, 1]], np.int32)
    tok = np.array([[-1, 10, 11, 12]], np.int32)
    sc = np.array([[0, -1.0, -0.5, -3.0]], np.float32)
    p, t, st = odt.rerank(par, tok, sc, 4, pool=np.array([[2]]))
    assert st == 0 and p[0].tolist() == [-1, 0, odt.ABSENT, odt.ABSENT] and t[0].tolist() == [-1, 11, -1, -1]
