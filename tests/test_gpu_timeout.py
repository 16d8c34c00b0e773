"""The tensor-core kernels' bounded waits: a wait that runs out sets the TIMEOUT status
bit and the call still returns; the next call on the same workspace is exact again.

The wait bound is shortened from the host (treespec_set_wait_limit_ns) so that the
kernels give up at their first hand-off that is not already complete.  Nothing here
faults or hangs the GPU: every abandoned CTA waits, under the normal bound, for the
copies and tensor-core work it already started before it frees its tensor memory."""
import time

import numpy as np
import pytest
import torch

import gen
from gen import inputs as gi

from gpu_util import assert_attention_close, attn_device_inputs, oracle_attention

pytestmark = pytest.mark.gpu

TIMEOUT_BIT = 1 << 4


@pytest.fixture(scope="module")
def ts():
    import __graft_entry__
    __graft_entry__.build()
    import eagle_speculative_tree_gb300 as mod
    yield mod
    mod.set_wait_limit_ns(0)


@pytest.mark.parametrize("kernel,splits", [(2, 1), (3, 1), (2, 0), (4, 1), (4, 0), (5, 0)])
def test_a_wait_that_runs_out_is_reported_and_the_next_call_is_exact(ts, cuda_device, kernel, splits):
    w = gen.get("c4_llama3_70b_bf16_greedy").with_batch(2)
    x = gi.make_inputs(w, with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    prob = ts.attn_problem(d["q"], d["k_pages"], d["page_table"], kernel=kernel, num_splits=splits)
    assert ts.attn_plan(prob).kernel == kernel
    ws = torch.empty(ts.attn_workspace_bytes(prob), dtype=torch.uint8, device=cuda_device)
    args = (d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["prefix_lens"], d["tree_parents"])
    ts.set_wait_limit_ns(1)
    try:
        t0 = time.monotonic()
        ts.tree_attn_verify(*args, kernel=kernel, num_splits=splits, workspace=ws)
        status = ts.read_status(ws)
        elapsed = time.monotonic() - t0
    finally:
        ts.set_wait_limit_ns(0)
    assert status & TIMEOUT_BIT, f"status {status:#x}: no wait ran out"
    assert elapsed < 10.0
    out = ts.tree_attn_verify(*args, kernel=kernel, num_splits=splits, workspace=ws)
    assert ts.read_status(ws) == 0
    ref = oracle_attention(x, [(0, 0), (1, 7)])
    assert_attention_close(out, ref, w.dtype, mask=~np.isnan(ref))
