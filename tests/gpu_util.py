"""Shared helpers of the GPU parity tests: move generated inputs to the device, call the
library through its binding, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from gen import inputs as gi
from oracle import accept as oacc
from oracle import attention as oatt
from oracle.tree_mask import tree_size

# Attention tolerances: float32 |err| <= 1e-4; bfloat16 |err| <= 1e-2 + 1e-2 |ref|.
F32_ATOL = 1e-4
BF16_ATOL, BF16_RTOL = 1e-2, 1e-2
# Stochastic decisions whose float64 margin is below this are rounding ties (both
# outcomes are correct); derived in the design notes from float32 error bounds.
TIE_MARGIN = 2e-5
# A sequence may take a tie neighbour only where its decision margin is below the error of
# the kernels' float32 arithmetic: a probability 2^(x c - M) / S carries a few ulp from the
# exp2 and the scaling plus about 30 roundings of the cluster-wide sum S, and any prefix of
# the bonus draw's weights about 33 roundings of the total -- 2e-6 of the mass at 2^-24 each.
# A flip with a larger margin is a bug.
FLOAT32_BOUND = 2e-6


def dev_tensor(a: np.ndarray, device, bf16: bool = False) -> torch.Tensor:
    if bf16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def attn_device_inputs(x: gi.TreeInputs, device):
    bf = x.workload.dtype == "bf16"
    return dict(q=dev_tensor(x.q, device, bf), k_pages=dev_tensor(x.k_pages, device, bf),
                v_pages=dev_tensor(x.v_pages, device, bf), page_table=dev_tensor(x.page_table, device),
                prefix_lens=dev_tensor(x.prefix_lens, device), tree_parents=dev_tensor(x.tree_parents, device))


def oracle_attention(x: gi.TreeInputs, pairs=None) -> np.ndarray:
    dt = x.workload.dtype
    return oatt.tree_attention(gi.as_float(x.q, dt), gi.as_float(x.k_pages, dt), gi.as_float(x.v_pages, dt),
                               x.page_table, x.prefix_lens, x.tree_parents, x.workload.page_size, pairs)


def assert_attention_close(out: torch.Tensor, ref: np.ndarray, dtype: str, mask=None) -> float:
    got = out.float().cpu().numpy().astype(np.float64)
    if mask is not None:
        got, ref = got[mask], ref[mask]
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), "non-finite attention output"
    if dtype == "f32":
        bad = err > F32_ATOL
    else:
        bad = err > BF16_ATOL + BF16_RTOL * np.abs(ref)
    assert not bad.any(), f"{bad.sum()} elements out of tolerance, max err {err.max():.3e}"
    return float(err.max())


def accept_device_inputs(x: gi.TreeInputs, device):
    d = dict(target_logits=dev_tensor(x.target_logits, device), draft_tokens=dev_tensor(x.draft_tokens, device),
             tree_parents=dev_tensor(x.tree_parents, device), draft_probs=None, uniforms=None)
    if x.draft_probs is not None:
        d["draft_probs"] = dev_tensor(x.draft_probs, device)
        d["uniforms"] = dev_tensor(x.uniforms, device)
    return d


def oracle_accept(logits, tokens, probs, parents, uniforms, temperature):
    return oacc.tree_accept(logits, tokens, probs, parents, uniforms, temperature)


def _walk_one(logits, tokens, probs, parents, uniforms, temperature):
    if temperature == 0:
        w = oacc.greedy_walk(logits, tokens, parents)
    else:
        w = oacc.stochastic_walk(logits, tokens, probs, parents, uniforms, temperature)
    return tuple(w.path), w.bonus


def tie_alternatives(logits, tokens, probs, parents, uniforms, temperature, result):
    """Outcomes the oracle reaches when a near-tie coin is nudged across its boundary.

    A child test's margin is relative to the terms it compares, so its coin is scaled by
    1 -/+ 8 TIE_MARGIN.  A bonus draw's margin is the distance of u from a CDF boundary in
    units of the total mass, and the token on the far side of that boundary may hold far
    less than TIE_MARGIN of the mass (a nudge of 1e-6 can pass over two tokens), so its
    coin moves by -/+ TIE_MARGIN 2^-k for k = 0 .. 36: every token whose CDF interval meets
    the tie window and is not much narrower than its distance from u is reached."""
    alts = {(tuple(result.path), result.bonus)}
    for kind, node, _x, _ok, margin in result.decisions:
        if margin >= TIE_MARGIN:
            continue
        u0 = np.array(uniforms, dtype=np.float64)
        if kind == "test":
            moved = [(node, u0[node] * f) for f in (1 - 8 * TIE_MARGIN, 1 + 8 * TIE_MARGIN)]
        else:
            steps = TIE_MARGIN * 0.5 ** np.arange(37)
            moved = [(0, u0[0] + s * d) for d in steps for s in (-1.0, 1.0)]
        for coin, u in moved:
            u2 = u0.copy()
            u2[coin] = min(max(u, 0.0), np.nextafter(1.0, 0.0))
            alts.add(_walk_one(logits, tokens, probs, parents, u2, temperature))
    return alts


def compare_accept(gpu, logits, tokens, probs, parents, uniforms, temperature):
    """Bit-exact comparison; a sequence whose decision margin is below FLOAT32_BOUND may take a
    neighbouring outcome (it is then printed); any other difference fails.

    Returns (number of sequences, number with a tie, number that took the other side)."""
    path, length, bonus = (t.cpu().numpy() for t in gpu)
    opath, olen, obonus, results = oracle_accept(logits, tokens, probs, parents, uniforms, temperature)
    ties = flipped = 0
    for b in range(len(olen)):
        got = (tuple(path[b, : length[b]].tolist()), int(bonus[b]))
        assert (path[b, length[b]:] == -1).all(), f"sequence {b}: path not -1 padded"
        want = (tuple(opath[b, : olen[b]].tolist()), int(obonus[b]))
        if got == want:
            if results[b].min_margin < TIE_MARGIN:
                ties += 1
            continue
        assert results[b].min_margin < FLOAT32_BOUND, \
            f"sequence {b}: gpu {got} != oracle {want} (margin {results[b].min_margin:.3g})"
        ties += 1
        nb = tree_size(parents[b])
        alts = tie_alternatives(logits[b][:nb], tokens[b][:nb], None if probs is None else probs[b][:nb],
                                parents[b][:nb], None if uniforms is None else uniforms[b][:nb], temperature,
                                results[b])
        assert got in alts, f"sequence {b}: gpu {got} is not the oracle's {want} nor a tie neighbour"
        print(f"sequence {b}: margin {results[b].min_margin:.3g} below the float32 bound, took {got} "
              f"for the oracle's {want}")
        flipped += 1
    return len(olen), ties, flipped
