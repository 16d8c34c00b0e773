"""Pins for the accept-walk oracle.

Greedy: brute force over every root path on all small trees, and the pages'
worked examples (golden fixtures).  Stochastic: the invariance theorem -- the
emitted tokens follow the target distribution -- checked by Monte-Carlo with a
chi-square bound, plus special cases with closed forms.  Planted mistakes in
the walk must fail the Monte-Carlo pin.
"""
import inspect
import itertools
import json
import os

import numpy as np
import pytest
from scipy import special, stats

from gen import trees
from gen import mc
from oracle import accept as oacc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def all_parent_arrays(n):
    """Every topologically ordered tree on n nodes: parents[i] in [0, i)."""
    for choice in itertools.product(*[range(i) for i in range(1, n)]):
        yield np.array((-1,) + choice, dtype=np.int32)


def brute_force_greedy(logits, tokens, parents):
    """Longest root path whose every token equals the argmax of its parent's row."""
    n = len(parents)
    best_path = []
    for node in range(1, n):
        path = [node]
        while parents[path[-1]] != 0:
            path.append(int(parents[path[-1]]))
        path = path[::-1]
        ok = all(tokens[c] == np.argmax(logits[parents[c]]) for c in path)
        if ok and len(path) > len(best_path):
            best_path = path
    last = best_path[-1] if best_path else 0
    return best_path, int(np.argmax(logits[last]))


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7])
def test_greedy_equals_brute_force_on_all_small_trees(n):
    rng = np.random.default_rng(n)
    V = 4 if n <= 5 else 8
    for parents in all_parent_arrays(n):
        for _ in range(3 if n < 7 else 1):
            logits = rng.integers(0, 3, (n, V)).astype(np.float32)   # small ints: many ties
            tokens = np.zeros(n, dtype=np.int32)
            for p in set(parents[1:].tolist()):
                kids = [c for c in range(1, n) if parents[c] == p]
                if len(kids) > V:
                    continue
                tokens[kids] = rng.permutation(V)[: len(kids)]       # distinct siblings
            if any(len([c for c in range(1, n) if parents[c] == p]) > V for p in range(n)):
                continue
            w = oacc.greedy_walk(logits, tokens, parents)
            ref_path, ref_bonus = brute_force_greedy(logits, tokens, parents)
            assert w.path == ref_path and w.bonus == ref_bonus


def longest_matching_path_by_dfs(logits, tokens, parents):
    """Independent statement for large trees: depth-first search from the root over the
    children whose token is the argmax of their parent's row; the deepest node reached
    (ties: the one whose root path comes first in node order) ends the path."""
    n = len(parents)
    kids = {i: [c for c in range(1, n) if parents[c] == i] for i in range(n)}
    best = []

    def dfs(node, path):
        nonlocal best
        if len(path) > len(best):
            best = list(path)
        a = int(np.argmax(logits[node]))
        for c in kids[node]:
            if tokens[c] == a:
                dfs(c, path + [c])

    dfs(0, [])
    last = best[-1] if best else 0
    return best, int(np.argmax(logits[last]))


@pytest.mark.parametrize("n", [65, 100, 128])
def test_greedy_on_trees_past_64_nodes_equals_dfs(n):
    """Distinct sibling tokens make the matching path unique; the walk must find it."""
    rng = np.random.default_rng(n)
    V = 512
    for trial in range(20):
        parents = trees.chain(n) if trial == 0 else trees.random_recursive(rng, n)
        logits = rng.normal(0, 3, (n, V)).astype(np.float32)
        tokens = np.zeros(n, dtype=np.int32)
        for p in range(n):
            kids = [c for c in range(1, n) if parents[c] == p]
            if not kids:
                continue
            toks = rng.permutation(V)[: len(kids)]           # distinct siblings
            a = int(np.argmax(logits[p]))
            if rng.random() < 0.8 and a not in toks:         # the argmax sits on one child most of the time
                toks[rng.integers(0, len(kids))] = a
            tokens[kids] = toks
        w = oacc.greedy_walk(logits, tokens, parents)
        ref_path, ref_bonus = longest_matching_path_by_dfs(logits, tokens, parents)
        assert w.path == ref_path and w.bonus == ref_bonus


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("name", ["branch_fallthrough_greedy.json", "linear_cascade_greedy.json"])
def test_pages_worked_examples(name):
    g = _golden(name)
    n, V = len(g["parents"]), g["vocab"]
    logits = np.zeros((n, V), dtype=np.float32)
    logits[np.arange(n), g["target_argmax_per_node"]] = 5.0
    path, length, bonus, _ = oacc.tree_accept(logits[None], np.array([g["tokens"]]), None,
                                              np.array([g["parents"]]), None, 0.0)
    e = g["expected"]
    assert length[0] == e["accept_len"]
    assert list(path[0, : length[0]]) == e["accept_path"]
    assert all(path[0, length[0]:] == -1)
    assert bonus[0] == e["bonus_token"]


def test_greedy_tie_takes_lowest_token_id():
    logits = np.array([[1, 3, 3, 0], [0, 0, 0, 0]], dtype=np.float32)
    w = oacc.greedy_walk(logits, np.array([0, 2]), np.array([-1, 0]))
    assert w.path == [] and w.bonus == 1
    w = oacc.greedy_walk(logits, np.array([0, 1]), np.array([-1, 0]))
    assert w.path == [1] and w.bonus == 0


# ------------------------------------------------------------- stochastic walk

def run_mc(walk, trials, seed, temperature=1.0):
    t = mc.mc_tables(seed)
    logits, q, tokens, uniforms, parents = mc.mc_trials(t, trials, seed)
    first = np.empty(trials, dtype=np.int64)
    second = np.full(trials, -1, dtype=np.int64)
    for i in range(trials):
        w = walk(logits[i], tokens[i], q[i], parents[i], uniforms[i], temperature)
        emitted = [int(tokens[i][c]) for c in w.path] + [w.bonus]
        first[i] = emitted[0]
        if w.length >= 1:
            second[i] = emitted[1]
    return t, first, second


def chi2_pvalues(t, first, second, temperature=1.0):
    V = mc.MC_VOCAB
    p_root = special.softmax(t.root_logits.astype(np.float64) / temperature)
    c1 = np.bincount(first, minlength=V)
    p1 = stats.chisquare(c1, c1.sum() * p_root).pvalue
    stat, dof = 0.0, 0
    for x in range(V):
        sel = (first == x) & (second >= 0)
        if sel.sum() < 200:
            continue
        cnt = np.bincount(second[sel], minlength=V)
        exp = sel.sum() * special.softmax(t.d1_logits[x].astype(np.float64) / temperature)
        stat += float(((cnt - exp) ** 2 / exp).sum())
        dof += V - 1
    p2 = stats.chi2.sf(stat, dof)
    return p1, p2


@pytest.mark.parametrize("temperature", [1.0, 0.7])
def test_monte_carlo_emitted_tokens_follow_target(temperature):
    """Invariance: first token ~ p_root, next token ~ p(. | first) (chi-square, alpha = 1e-3)."""
    t, first, second = run_mc(oacc.stochastic_walk, 60000, 3, temperature)
    p1, p2 = chi2_pvalues(t, first, second, temperature)
    assert p1 > 1e-3 and p2 > 1e-3, (p1, p2)


def _planted_walk(old, new):
    src = inspect.getsource(oacc.stochastic_walk)
    assert old in src
    ns = dict(vars(oacc))
    exec(compile(src.replace(old, new), "<planted>", "exec"), ns)
    return ns["stochastic_walk"]


@pytest.mark.parametrize("old,new", [
    ("r = resid / z", "r = resid"),                                    # residual not normalised
    ("resid = np.maximum(0.0, r - q_cur)", "resid = r"),                # siblings re-test against p
    ("ok = r[x] > 0 and lhs <= r[x]", "ok = r[x] > 0 and lhs * r[x] <= q_cur[x]"),   # ratio inverted
    ("cdf = np.cumsum(r)", "cdf = np.cumsum(q_cur if accepted is None and path == [] else r)"),
])
def test_planted_mistakes_fail_monte_carlo(old, new):
    t, first, second = run_mc(_planted_walk(old, new), 30000, 4)
    p1, p2 = chi2_pvalues(t, first, second)
    assert min(p1, p2) < 1e-3, (p1, p2)


def test_q_equal_p_accepts_first_child():
    rng = np.random.default_rng(5)
    for _ in range(200):
        V, n = 8, 4
        logits = rng.normal(0, 2, (n, V)).astype(np.float32)
        q = special.softmax(logits.astype(np.float64), axis=-1)
        parents = np.array([-1, 0, 0, 1])
        tokens = rng.integers(0, V, n)
        u = rng.random(n) * 0.999999
        w = oacc.stochastic_walk(logits, tokens, q, parents, u, 1.0)
        assert w.length >= 1 and w.path[0] == 1


def test_single_child_is_the_textbook_accept_test():
    """One candidate x: accepted exactly when u <= min(1, p(x)/q(x))."""
    rng = np.random.default_rng(6)
    for _ in range(100):
        V = 8
        logits = rng.normal(0, 2, (2, V))
        q = rng.dirichlet(np.ones(V), 2)
        x = int(rng.integers(0, V))
        p = special.softmax(logits[0])
        alpha = min(1.0, p[x] / q[0, x])
        for u in np.linspace(0.0005, 0.9995, 41):
            if abs(u - alpha) < 1e-9:
                continue
            w = oacc.stochastic_walk(logits, np.array([0, x]), q, np.array([-1, 0]),
                                     np.array([0.5, u]), 1.0)
            assert (w.length == 1) == (u <= alpha)


def test_leaf_sample_is_inverse_cdf_of_target():
    """With no children the bonus is the inverse-CDF draw of p with the final coin."""
    rng = np.random.default_rng(7)
    logits = rng.normal(0, 1, (1, 16))
    p = special.softmax(logits[0] / 0.8)
    for u0 in rng.random(200):
        w = oacc.stochastic_walk(logits, np.array([0]), np.ones((1, 16)) / 16, np.array([-1]),
                                 np.array([u0]), 0.8)
        assert w.bonus == int(np.searchsorted(np.cumsum(p), u0, side="right"))


def test_tiny_temperature_with_one_hot_draft_equals_greedy():
    rng = np.random.default_rng(8)
    for _ in range(200):
        n, V = 7, 6
        parents = np.array([-1, 0, 0, 1, 1, 3, 2])
        logits = np.zeros((n, V), dtype=np.float32)
        for i in range(n):
            logits[i] = rng.permutation(V).astype(np.float32)       # distinct integer logits
        q = np.zeros((n, V))
        q[np.arange(n), np.argmax(logits, axis=1)] = 1.0
        tokens = np.zeros(n, dtype=np.int32)
        for p in range(n):
            kids = [c for c in range(1, n) if parents[c] == p]
            tokens[kids] = rng.permutation(V)[: len(kids)]
        g = oacc.greedy_walk(logits, tokens, parents)
        s = oacc.stochastic_walk(logits, tokens, q, parents, rng.random(n) * 0.99, 1e-3)
        assert (s.path, s.bonus) == (g.path, g.bonus)


def test_margins_flag_near_ties():
    logits = np.log(np.array([[0.5, 0.5], [0.5, 0.5]]))
    q = np.array([[0.5, 0.5], [0.5, 0.5]])
    w = oacc.stochastic_walk(logits, np.array([0, 1]), q, np.array([-1, 0]),
                             np.array([0.3, 1.0]), 1.0)
    assert w.min_margin < 1e-12           # u*q(x) == p(x): a tie
    w = oacc.stochastic_walk(logits, np.array([0, 1]), q, np.array([-1, 0]),
                             np.array([0.3, 0.5]), 1.0)
    assert w.min_margin > 0.1
