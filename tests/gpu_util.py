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
    """Outcomes the oracle reaches when a near-tie coin is nudged across its boundary."""
    alts = {(tuple(result.path), result.bonus)}
    for kind, node, _x, _ok, margin in result.decisions:
        if margin >= TIE_MARGIN:
            continue
        coin = node if kind == "test" else 0
        for f in (1 - 8 * TIE_MARGIN, 1 + 8 * TIE_MARGIN):
            u2 = np.array(uniforms, dtype=np.float64).copy()
            u2[coin] = min(max(u2[coin] * f, 0.0), 1.0)
            alts.add(_walk_one(logits, tokens, probs, parents, u2, temperature))
    return alts


def compare_accept(gpu, logits, tokens, probs, parents, uniforms, temperature):
    """Bit-exact comparison; sequences with a rounding tie may take a neighbouring outcome.

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
        assert results[b].min_margin < TIE_MARGIN, f"sequence {b}: gpu {got} != oracle {want}"
        ties += 1
        nb = tree_size(parents[b])
        alts = tie_alternatives(logits[b][:nb], tokens[b][:nb], None if probs is None else probs[b][:nb],
                                parents[b][:nb], None if uniforms is None else uniforms[b][:nb], temperature,
                                results[b])
        assert got in alts, f"sequence {b}: gpu {got} is not the oracle's {want} nor a tie neighbour"
        flipped += 1
    return len(olen), ties, flipped
