"""tree_attn_verify_noalloc against tree_attn_verify, through the C-ABI.

The no-allocation entry point serves callers that cannot allocate device memory
where they verify a tree (their application owns all device memory, or an
allocation's implicit synchronisation is too costly); it keeps its scratch in a
fixed device array inside the library.  Its results must match the workspace
entry point's on consecutive calls (the array keeps the previous call's contents,
so the second call checks that nothing stale leaks through).
"""
import ctypes

import numpy as np
import pytest
import torch

import gen
from gen import inputs as gi

from gpu_util import BF16_ATOL, BF16_RTOL, F32_ATOL, attn_device_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ts():
    import __graft_entry__
    __graft_entry__.build()
    import eagle_speculative_tree_gb300 as mod
    lib = mod.raw_library()
    lib.tree_attn_verify_noalloc.argtypes = [ctypes.c_void_p] * 7 + [ctypes.POINTER(mod.AttnShape), ctypes.c_void_p]
    lib.tree_attn_verify_noalloc.restype = ctypes.c_int
    lib.treespec_noalloc_read_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p]
    lib.treespec_noalloc_read_status.restype = ctypes.c_int
    return mod


def _noalloc_status(ts):
    st = ctypes.c_uint32(0)
    assert ts.raw_library().treespec_noalloc_read_status(ctypes.byref(st),
                                                          torch.cuda.current_stream().cuda_stream) == 0
    return st.value


def _noalloc(ts, d, out, prob):
    return ts.raw_library().tree_attn_verify_noalloc(
        d["q"].data_ptr(), d["k_pages"].data_ptr(), d["v_pages"].data_ptr(), d["page_table"].data_ptr(),
        d["prefix_lens"].data_ptr(), d["tree_parents"].data_ptr(), out.data_ptr(), ctypes.byref(prob.c_shape()),
        torch.cuda.current_stream().cuda_stream)


def _close(got, ref, dtype):
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    tol = F32_ATOL if dtype == "f32" else BF16_ATOL + BF16_RTOL * np.abs(r)
    assert np.isfinite(g).all()
    assert (np.abs(g - r) <= tol).all(), float(np.abs(g - r).max())


@pytest.mark.parametrize("name", ["c1_tiny_f32_greedy", "c2_llama3_8b_bf16_greedy",
                                  "c4_llama3_70b_bf16_greedy@b1", "c5_ragged_b64_bf16_stoch@b2"])
def test_noalloc_matches_workspace_entry_point_twice(ts, cuda_device, name):
    w = gen.get(name)
    x = gi.make_inputs(w, with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    ref = ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["prefix_lens"],
                              d["tree_parents"])
    prob = ts.attn_problem(d["q"], d["k_pages"], d["page_table"])
    for _ in range(2):
        out = torch.full_like(d["q"], float("nan"))
        assert _noalloc(ts, d, out, prob) == 0
        torch.cuda.synchronize()
        _close(out, ref, w.dtype)


def test_noalloc_runs_the_one_range_kernel_where_the_persistent_one_does_not_fit(ts, cuda_device):
    """At the full Llama-3-70B batch the automatic plan is the persistent two-tile kernel,
    whose partial slots exceed the fixed array: the no-allocation entry runs the two-tile
    kernel one range per CTA instead, and agrees with the workspace entry point."""
    w = gen.get("c4_llama3_70b_bf16_greedy")
    x = gi.make_inputs(w, with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    prob = ts.attn_problem(d["q"], d["k_pages"], d["page_table"])
    assert ts.attn_plan(prob).kernel == ts.KERNEL_TC_STREAM
    assert ts.attn_workspace_bytes(prob) > 32 << 20
    ref = ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["prefix_lens"],
                              d["tree_parents"])
    out = torch.full_like(d["q"], float("nan"))
    assert _noalloc(ts, d, out, prob) == 0
    torch.cuda.synchronize()
    _close(out, ref, w.dtype)


def test_noalloc_rejects_shapes_beyond_its_scratch(ts, cuda_device):
    w = gen.get("c4_llama3_70b_bf16_greedy@b1")
    x = gi.make_inputs(w, with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    prob = ts.attn_problem(d["q"], d["k_pages"], d["page_table"], num_splits=65)
    assert ts.attn_workspace_bytes(prob) > 32 << 20
    out = torch.zeros_like(d["q"])
    assert _noalloc(ts, d, out, prob) == -4
    bad = ts.attn_problem(d["q"], d["k_pages"], d["page_table"])
    bad.num_nodes = 129
    assert _noalloc(ts, d, out, bad) == -2


def test_noalloc_padded_trees_back_to_back(ts, cuda_device):
    """Trees of different sizes (rows padded with -2), two calls in a row with different
    padding: the second call reuses the array's node counts and ancestor words the first
    one left, and must still match the workspace entry point."""
    from gen import trees
    w = gen.get("c4_llama3_70b_bf16_greedy").with_batch(4)
    rng = np.random.default_rng(21)
    for sizes in ([64, 17, 1, 40], [9, 64, 33, 2]):
        parents = trees.padded([trees.random_recursive(rng, n) for n in sizes], w.num_nodes)
        x = gi.make_inputs(w, parents=parents, prefix_lens=np.asarray([100, 37, 0, 300], dtype=np.int32),
                           with_accept=False)
        d = attn_device_inputs(x, cuda_device)
        ref = ts.tree_attn_verify(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["prefix_lens"],
                                  d["tree_parents"])
        out = torch.full_like(d["q"], float("nan"))
        assert _noalloc(ts, d, out, ts.attn_problem(d["q"], d["k_pages"], d["page_table"])) == 0
        assert _noalloc_status(ts) == 0
        _close(out, ref, w.dtype)
        for b, n in enumerate(sizes):
            assert torch.all(out[b, n:] == 0)


def test_noalloc_status_word_flags_a_bad_page_then_clears(ts, cuda_device):
    w = gen.get("c2_llama3_8b_bf16_greedy")
    x = gi.make_inputs(w, with_accept=False)
    d = attn_device_inputs(x, cuda_device)
    prob = ts.attn_problem(d["q"], d["k_pages"], d["page_table"])
    good = d["page_table"].clone()
    d["page_table"][0, 2] = 1 << 30
    out = torch.zeros_like(d["q"])
    assert _noalloc(ts, d, out, prob) == 0
    assert _noalloc_status(ts) & 2                     # TREESPEC_STATUS_BAD_PAGE
    d["page_table"] = good
    assert _noalloc(ts, d, out, prob) == 0
    assert _noalloc_status(ts) == 0
