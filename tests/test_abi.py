"""The C-ABI library loads, exports every declared symbol, and rejects bad arguments on
the host before any launch.  Runs without a GPU (fake device pointers are never
dereferenced because every call below fails validation first)."""
import ctypes
import re

import pytest

import __graft_entry__

__graft_entry__.build()
import eagle_speculative_tree_gb300 as ts  # noqa: E402

FAKE = 0x10000          # 16-byte aligned, never dereferenced


def test_every_declared_symbol_is_exported():
    names = ts.exported_symbols()
    assert {"tree_attn_verify", "tree_accept", "treespec_attn_workspace_bytes",
            "treespec_accept_workspace_bytes", "treespec_read_status"} <= set(names)
    lib = ctypes.CDLL(ts.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_header_declarations_are_extern_c():
    text = open(ts.HEADER_PATH).read()
    assert re.search(r'extern "C"', text)


def test_version_and_error_strings():
    assert ts.version() >= 100
    lib = ts.raw_library()
    for code in range(-8, 1):
        assert lib.treespec_error_string(code)


def shape(**kw):
    base = dict(batch=1, num_nodes=8, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                max_pages_per_seq=129, num_pool_pages=200, dtype=ts.DTYPE_BF16)
    base.update(kw)
    return ts.AttnProblem(**base)


@pytest.mark.parametrize("kw", [
    dict(num_nodes=129), dict(num_nodes=0), dict(num_q_heads=30), dict(head_dim=96),
    dict(page_size=32), dict(batch=0), dict(dtype=7), dict(max_pages_per_seq=0),
    dict(num_splits=-1), dict(kernel=9),
    dict(kernel=3),                       # two-tile kernel: 8 nodes x 4 query heads is one 128-row block
    dict(kernel=4),                       # CTA-pair kernel: the same
])
def test_attention_rejects_bad_shapes(kw):
    prob = shape(**kw)
    assert ts.raw_library().treespec_attn_workspace_bytes(ctypes.byref(prob.c_shape())) == 0
    rc = ts.raw_library().tree_attn_verify(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                           ctypes.byref(prob.c_shape()), FAKE * 256, 1 << 30, None)
    assert rc in (ts.TreespecError(-2).code, -3, -2)
    assert rc < 0


def test_attention_rejects_null_and_misaligned():
    prob = shape()
    lib = ts.raw_library()
    assert lib.tree_attn_verify(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(prob.c_shape()),
                                FAKE * 256, 1 << 30, None) == -1
    assert lib.tree_attn_verify(FAKE + 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(prob.c_shape()),
                                FAKE * 256, 1 << 30, None) == -6
    assert lib.tree_attn_verify(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(prob.c_shape()),
                                FAKE + 16, 1 << 30, None) == -4


def test_plan_and_workspace_query():
    prob = shape()
    plan = ts.attn_plan(prob)
    assert plan.num_splits >= 1 and plan.split_tokens % 128 == 0
    assert plan.num_splits * plan.split_tokens >= prob.max_pages_per_seq * 16
    assert ts.attn_workspace_bytes(prob) > 0
    single = ts.attn_plan(shape(num_splits=1))
    assert single.num_splits == 1 and single.merge == 0


def test_plan_pairs_query_tiles_when_the_row_blocks_pair_up():
    """Without a device the planner assumes 152 SMs."""
    wide = dict(num_nodes=64, num_q_heads=64, num_kv_heads=8)      # 512 rows: four 128-row blocks
    b8 = ts.attn_plan(shape(batch=8, **wide))                      # 128 two-tile CTAs: under one wave
    assert b8.kernel == ts.KERNEL_TC_2SM and b8.rows_per_block == 128 and b8.row_blocks == 4
    # two waves of two-tile CTAs or more: the persistent form, one CTA per SM
    b32 = ts.attn_plan(shape(batch=32, **wide))
    assert b32.kernel == ts.KERNEL_TC_STREAM and b32.num_splits == 1 and b32.merge == 0
    assert ts.attn_plan(shape(batch=19, **wide)).kernel == ts.KERNEL_TC_STREAM  # 304 two-tile units
    assert ts.attn_plan(shape(batch=18, **wide)).kernel == ts.KERNEL_TC_PAIR    # 288: under two waves
    assert ts.attn_plan(shape(batch=10, **wide)).kernel == ts.KERNEL_TC_PAIR    # 160: a wave and more
    assert ts.attn_plan(shape(batch=257, **wide)).kernel == ts.KERNEL_TC_PAIR   # past its batch limit
    with pytest.raises(ValueError):                                                # refused, not truncated
        ts.attn_workspace_bytes(shape(batch=257, kernel=ts.KERNEL_TC_STREAM, **wide))
    assert ts.attn_plan(shape(batch=9, **wide)).kernel == ts.KERNEL_TC_2SM      # 144: under one wave
    assert ts.attn_plan(shape(batch=1, **wide)).kernel == ts.KERNEL_TC_2SM
    assert ts.attn_plan(shape(batch=8, kernel=ts.KERNEL_TC, **wide)).kernel == ts.KERNEL_TC
    assert ts.attn_plan(shape(batch=32, kernel=ts.KERNEL_TC_PAIR, **wide)).kernel == ts.KERNEL_TC_PAIR
    assert ts.attn_plan(shape(batch=8, num_nodes=40, num_q_heads=64, num_kv_heads=8)).kernel == ts.KERNEL_TC
    assert ts.attn_plan(shape()).kernel == ts.KERNEL_TC                                             # 32 rows
    assert ts.attn_plan(shape(batch=8, dtype=ts.DTYPE_F32, **wide)).kernel == ts.KERNEL_SIMT


def test_accept_rejects_bad_arguments():
    lib = ts.raw_library()

    def call(logits=FAKE, probs=FAKE, unif=FAKE, temp=1.0, B=2, N=8, V=100, ws=FAKE * 256, wsb=1 << 30):
        return lib.tree_accept(logits, FAKE, probs, FAKE, unif, ctypes.c_float(temp), FAKE, FAKE, FAKE,
                               B, N, V, ws, wsb, None)

    assert call(N=129) == -2
    assert call(B=0) == -2
    assert call(V=0) == -2
    assert call(logits=None) == -1
    assert call(temp=-1.0) == -5
    assert call(temp=float("nan")) == -5
    assert call(probs=None) == -5
    assert call(unif=None) == -5
    assert call(logits=FAKE + 8) == -6
    assert call(ws=FAKE + 64) == -4
    assert call(wsb=16) == -4
    assert lib.treespec_accept_workspace_bytes(2, 129, 100) == 0


def test_valid_call_without_device_reports_no_device():
    """Every host check passes; with no GPU present the call stops at the device check."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    prob = shape()
    lib = ts.raw_library()
    rc = lib.tree_attn_verify(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.byref(prob.c_shape()),
                              FAKE * 256, 1 << 30, None)
    assert rc == -7


def test_padding_sentinel_matches_the_header():
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "treespec.h")).read()
    m = re.search(r"#define\s+TREESPEC_ABSENT\s+\((-?\d+)\)", hdr)
    assert m and int(m.group(1)) == ts.ABSENT == -2
    from gen import trees
    from oracle.tree_mask import ABSENT
    assert trees.PAD == ABSENT == ts.ABSENT
