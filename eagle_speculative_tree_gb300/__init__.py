"""Python binding of libtreespec (tree-attention verify + accept walk on GB300).

Argument marshalling only: every step runs in the CUDA library.  torch tensors
carry device memory and streams; nothing here computes any part of the method.
Importing the package fails if the compiled library is missing -- build it with
`python -m eagle_speculative_tree_gb300.build` (or `__graft_entry__.build()`).
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtreespec.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "treespec.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libtreespec.so is not built ({LIB_PATH}); run eagle_speculative_tree_gb300/build.py")

_lib = ctypes.CDLL(LIB_PATH)

DTYPE_F32, DTYPE_BF16 = 0, 1
KERNEL_AUTO, KERNEL_SIMT, KERNEL_TC, KERNEL_TC_PAIR, KERNEL_TC_2SM, KERNEL_TC_STREAM = 0, 1, 2, 3, 4, 5
ACCEPT_AUTO, ACCEPT_ALL_ROWS, ACCEPT_PATH_ONLY = 0, 1, 2
ABSENT = -2                     # parent entry of a padding slot after a smaller tree
STATUS_BITS = {1: "BAD_PARENT", 2: "BAD_PAGE", 4: "BAD_LENGTH", 8: "BAD_TOKEN", 16: "TIMEOUT", 32: "INTERNAL",
               64: "BAD_PATH"}


class AttnShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_nodes", "num_q_heads", "num_kv_heads", "head_dim", "page_size",
        "max_pages_per_seq", "num_pool_pages", "dtype", "kernel", "num_splits")]


class AttnPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "kernel", "num_splits", "split_tokens", "rows_per_block", "row_blocks", "merge")]


_vp, _i32p, _f32p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
_lib.treespec_attn_workspace_bytes.argtypes = [ctypes.POINTER(AttnShape)]
_lib.treespec_attn_workspace_bytes.restype = ctypes.c_size_t
_lib.treespec_attn_plan_for.argtypes = [ctypes.POINTER(AttnShape), ctypes.POINTER(AttnPlan)]
_lib.treespec_attn_plan_for.restype = ctypes.c_int
_lib.tree_attn_verify.argtypes = [_vp] * 7 + [ctypes.POINTER(AttnShape), _vp, ctypes.c_size_t, _vp]
_lib.tree_attn_verify.restype = ctypes.c_int
_lib.treespec_accept_workspace_bytes.argtypes = [ctypes.c_int32] * 3
_lib.treespec_accept_workspace_bytes.restype = ctypes.c_size_t
_lib.tree_accept.argtypes = [_vp] * 5 + [ctypes.c_float] + [_vp] * 3 + [ctypes.c_int32] * 3 + \
    [_vp, ctypes.c_size_t, _vp]
_lib.tree_accept.restype = ctypes.c_int
_lib.tree_accept_with_mode.argtypes = [_vp] * 5 + [ctypes.c_float] + [_vp] * 3 + [ctypes.c_int32] * 4 + \
    [_vp, ctypes.c_size_t, _vp]
_lib.tree_accept_with_mode.restype = ctypes.c_int
_lib.treespec_commit_workspace_bytes.argtypes = []
_lib.treespec_commit_workspace_bytes.restype = ctypes.c_size_t
_lib.tree_kv_commit.argtypes = [_vp] * 7 + [ctypes.POINTER(AttnShape), _vp, ctypes.c_size_t, _vp]
_lib.tree_kv_commit.restype = ctypes.c_int
_lib.treespec_draft_workspace_bytes.argtypes = [ctypes.c_int32] * 3
_lib.treespec_draft_workspace_bytes.restype = ctypes.c_size_t
_lib.tree_draft_step.argtypes = [_vp] + [ctypes.c_int32] * 5 + [_vp] * 4 + [ctypes.c_int32, _vp, _vp, ctypes.c_size_t, _vp]
_lib.tree_draft_step.restype = ctypes.c_int
_lib.tree_rerank.argtypes = [_vp] * 3 + [ctypes.c_int32] * 3 + [_vp] * 3 + [ctypes.c_size_t, _vp]
_lib.tree_rerank.restype = ctypes.c_int
_lib.tree_rerank_pool.argtypes = [_vp] * 4 + [ctypes.c_int32] * 4 + [_vp] * 3 + [ctypes.c_size_t, _vp]
_lib.tree_rerank_pool.restype = ctypes.c_int
_lib.treespec_read_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint32), _vp]
_lib.treespec_read_status.restype = ctypes.c_int
_lib.treespec_error_string.argtypes = [ctypes.c_int]
_lib.treespec_error_string.restype = ctypes.c_char_p
_lib.treespec_version.restype = ctypes.c_int
_lib.treespec_launch_count.restype = ctypes.c_uint64
_lib.treespec_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
_lib.treespec_set_wait_limit_ns.restype = None
_lib.treespec_last_launch_error.argtypes = [ctypes.POINTER(ctypes.c_char_p)]
_lib.treespec_last_launch_error.restype = ctypes.c_int


class TreespecError(RuntimeError):
    def __init__(self, code: int):
        self.code = code
        super().__init__(f"treespec error {code}: {_lib.treespec_error_string(code).decode()}")


def _check(code: int) -> None:
    if code != 0:
        raise TreespecError(code)


def exported_symbols() -> list[str]:
    """Function names declared in include/treespec.h."""
    text = open(HEADER_PATH).read()
    # declarations start in column 0 with a C return type; comment lines never do
    return sorted(set(re.findall(r"^(?:const\s+)?(?:int|size_t|void|uint64_t|uint32_t|char)\s*\*?\s*([a-z_0-9]+)\s*\(",
                                 text, re.M)))


def version() -> int:
    return _lib.treespec_version()


def launch_count() -> int:
    return int(_lib.treespec_launch_count())


def last_launch_error() -> tuple:
    """(cudaError_t code, its name) behind the last launch the CUDA runtime rejected."""
    name = ctypes.c_char_p()
    code = _lib.treespec_last_launch_error(ctypes.byref(name))
    return code, (name.value or b"").decode()


def set_wait_limit_ns(ns: int) -> None:
    """Bound (ns) of the tensor-core kernels' internal waits for later calls; 0 = the default
    2 s.  For tests of the timeout path (see include/treespec.h)."""
    _lib.treespec_set_wait_limit_ns(int(ns))


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream: Optional[torch.cuda.Stream], device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _need_rows(t: torch.Tensor, name: str, device) -> None:
    """float32 rows on `device`, or in pinned host memory (read in place by the kernel)."""
    if not ((t.is_cuda and t.device == device) or (t.device.type == "cpu" and t.is_pinned())):
        raise ValueError(f"{name} must be on {device} or in pinned host memory")
    if t.dtype != torch.float32:
        raise ValueError(f"{name} must be torch.float32, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, device) -> None:
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


@dataclass
class AttnProblem:
    batch: int
    num_nodes: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    max_pages_per_seq: int
    num_pool_pages: int
    dtype: int
    kernel: int = KERNEL_AUTO
    num_splits: int = 0

    def c_shape(self) -> AttnShape:
        return AttnShape(self.batch, self.num_nodes, self.num_q_heads, self.num_kv_heads, self.head_dim,
                         self.page_size, self.max_pages_per_seq, self.num_pool_pages, self.dtype,
                         self.kernel, self.num_splits)


def attn_problem(q: torch.Tensor, k_pages: torch.Tensor, page_table: torch.Tensor, *,
                 kernel: int = KERNEL_AUTO, num_splits: int = 0) -> AttnProblem:
    B, N, Hq, D = q.shape
    P, ps, Hkv, D2 = k_pages.shape
    if D2 != D:
        raise ValueError("head_dim of q and k_pages differ")
    dt = DTYPE_BF16 if q.dtype == torch.bfloat16 else DTYPE_F32
    return AttnProblem(B, N, Hq, Hkv, D, ps, page_table.shape[1], P, dt, kernel, num_splits)


def attn_workspace_bytes(prob: AttnProblem) -> int:
    n = _lib.treespec_attn_workspace_bytes(ctypes.byref(prob.c_shape()))
    if n == 0:
        raise ValueError(f"unsupported attention shape {prob}")
    return int(n)


def attn_plan(prob: AttnProblem) -> AttnPlan:
    plan = AttnPlan()
    _check(_lib.treespec_attn_plan_for(ctypes.byref(prob.c_shape()), ctypes.byref(plan)))
    return plan


def tree_attn_verify(q, k_pages, v_pages, page_table, prefix_lens, tree_parents, out=None, *,
                     kernel: int = KERNEL_AUTO, num_splits: int = 0,
                     workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Tree-attention verification pass; see include/treespec.h for the operation.

    q [B][N][Hq][D], k_pages / v_pages [P][16][Hkv][D] (float32 or bfloat16),
    page_table [B][max_pages] int32, prefix_lens [B] int32, tree_parents [B][N] int32.
    Returns out [B][N][Hq][D] in q's dtype.
    """
    dev = q.device
    dt = q.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise ValueError("q must be float32 or bfloat16")
    _need(q, "q", dt, dev)
    _need(k_pages, "k_pages", dt, dev)
    _need(v_pages, "v_pages", dt, dev)
    _need(page_table, "page_table", torch.int32, dev)
    _need(prefix_lens, "prefix_lens", torch.int32, dev)
    _need(tree_parents, "tree_parents", torch.int32, dev)
    prob = attn_problem(q, k_pages, page_table, kernel=kernel, num_splits=num_splits)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", dt, dev)
    need = attn_workspace_bytes(prob)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _check(_lib.tree_attn_verify(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(prefix_lens), _ptr(tree_parents),
        _ptr(out), ctypes.byref(prob.c_shape()), _ptr(workspace), workspace.numel(),
        _stream_handle(stream, dev)))
    return out


def accept_workspace_bytes(batch: int, num_nodes: int, vocab: int) -> int:
    n = _lib.treespec_accept_workspace_bytes(batch, num_nodes, vocab)
    if n == 0:
        raise ValueError("unsupported accept sizes")
    return int(n)


def tree_accept(target_logits, draft_tokens, draft_probs, tree_parents, uniforms, temperature: float, *,
                accept_path=None, accept_len=None, bonus_token=None, mode: int = ACCEPT_AUTO,
                workspace: Optional[torch.Tensor] = None, stream=None):
    """Accept walk; see include/treespec.h.  Returns (accept_path, accept_len, bonus_token).

    mode: ACCEPT_AUTO, ACCEPT_ALL_ROWS or ACCEPT_PATH_ONLY (tree_accept_with_mode).
    target_logits and draft_probs may be device tensors or pinned host tensors: the
    kernel reads host rows in place over the CPU-GPU link, and the path-only schedule
    reads only the rows on each sequence's walk."""
    dev = draft_tokens.device
    B, N, V = target_logits.shape
    _need_rows(target_logits, "target_logits", dev)
    _need(draft_tokens, "draft_tokens", torch.int32, dev)
    _need(tree_parents, "tree_parents", torch.int32, dev)
    if temperature > 0:
        _need_rows(draft_probs, "draft_probs", dev)
        _need(uniforms, "uniforms", torch.float32, dev)
    if accept_path is None:
        accept_path = torch.empty((B, N), dtype=torch.int32, device=dev)
    if accept_len is None:
        accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    if bonus_token is None:
        bonus_token = torch.empty((B,), dtype=torch.int32, device=dev)
    need = accept_workspace_bytes(B, N, V)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _check(_lib.tree_accept_with_mode(
        _ptr(target_logits), _ptr(draft_tokens), _ptr(draft_probs) if temperature > 0 else None,
        _ptr(tree_parents), _ptr(uniforms) if temperature > 0 else None, float(temperature),
        _ptr(accept_path), _ptr(accept_len), _ptr(bonus_token), B, N, V, int(mode),
        _ptr(workspace), workspace.numel(), _stream_handle(stream, dev)))
    return accept_path, accept_len, bonus_token


def commit_workspace_bytes() -> int:
    return int(_lib.treespec_commit_workspace_bytes())


def tree_kv_commit(k_pages, v_pages, page_table, prefix_lens, accept_path, accept_len, new_prefix_lens=None, *,
                   workspace: Optional[torch.Tensor] = None, stream=None):
    """Move the accepted path's K/V next to each prefix, in place; see include/treespec.h.

    k_pages / v_pages [P][16][Hkv][D] (float32 or bfloat16), page_table [B][max_pages],
    prefix_lens [B], accept_path [B][N], accept_len [B] (int32).  Returns new_prefix_lens
    [B] int32 (prefix + 1 + accept_len, or -1 for a sequence left unchanged)."""
    dev = k_pages.device
    dt = k_pages.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise ValueError("k_pages must be float32 or bfloat16")
    _need(k_pages, "k_pages", dt, dev)
    _need(v_pages, "v_pages", dt, dev)
    for name, t in (("page_table", page_table), ("prefix_lens", prefix_lens), ("accept_path", accept_path),
                    ("accept_len", accept_len)):
        _need(t, name, torch.int32, dev)
    B, N = accept_path.shape
    P, ps, Hkv, D = k_pages.shape
    shape = AttnShape(B, N, Hkv, Hkv, D, ps, page_table.shape[1], P,
                      DTYPE_BF16 if dt == torch.bfloat16 else DTYPE_F32, KERNEL_AUTO, 0)
    if new_prefix_lens is None:
        new_prefix_lens = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(new_prefix_lens, "new_prefix_lens", torch.int32, dev)
    need = commit_workspace_bytes()
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _check(_lib.tree_kv_commit(_ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(prefix_lens), _ptr(accept_path),
                               _ptr(accept_len), _ptr(new_prefix_lens), ctypes.byref(shape), _ptr(workspace),
                               workspace.numel(), _stream_handle(stream, dev)))
    return new_prefix_lens


def draft_workspace_bytes(batch: int, frontier: int, topk: int) -> int:
    n = _lib.treespec_draft_workspace_bytes(batch, frontier, topk)
    if n == 0:
        raise ValueError("unsupported draft-step sizes")
    return int(n)


def tree_draft_step(logprobs, step: int, topk: int, frontier_in, node_parent, node_token, node_score,
                    frontier_out=None, *, workspace: Optional[torch.Tensor] = None, stream=None):
    """One beam-expansion step of the draft tree, in place on the node arrays; see
    include/treespec.h.  logprobs [B][F][V] float32 (F = 1 at step 0, else topk);
    frontier_in [B][F] int32 (the previous step's result; None at step 0); node_parent /
    node_token [B][M] int32, node_score [B][M] float32.  Returns (frontier_out [B][topk],
    workspace)."""
    dev = logprobs.device
    _need(logprobs, "logprobs", torch.float32, dev)
    _need(node_parent, "node_parent", torch.int32, dev)
    _need(node_token, "node_token", torch.int32, dev)
    _need(node_score, "node_score", torch.float32, dev)
    if frontier_in is not None:
        _need(frontier_in, "frontier_in", torch.int32, dev)
    B, F, V = logprobs.shape
    M = node_parent.shape[1]
    if frontier_out is None:
        frontier_out = torch.empty((B, topk), dtype=torch.int32, device=dev)
    _need(frontier_out, "frontier_out", torch.int32, dev)
    need = draft_workspace_bytes(B, F, topk)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _check(_lib.tree_draft_step(_ptr(logprobs), B, F, V, topk, step, _ptr(frontier_in), _ptr(node_parent),
                                _ptr(node_token), _ptr(node_score), M, _ptr(frontier_out), _ptr(workspace),
                                workspace.numel(), _stream_handle(stream, dev)))
    return frontier_out, workspace


def tree_rerank(node_parent, node_token, node_score, num_nodes: int, tree_parents=None, draft_tokens=None, *,
                pool=None, workspace: Optional[torch.Tensor] = None, stream=None):
    """Keep the root and the num_nodes - 1 best nodes (of all, or of `pool` [B][P] int32
    node ids: tree_rerank_pool); returns (tree_parents, draft_tokens) [B][num_nodes] int32.
    See include/treespec.h."""
    dev = node_parent.device
    _need(node_parent, "node_parent", torch.int32, dev)
    _need(node_token, "node_token", torch.int32, dev)
    _need(node_score, "node_score", torch.float32, dev)
    B, M = node_parent.shape
    if tree_parents is None:
        tree_parents = torch.empty((B, num_nodes), dtype=torch.int32, device=dev)
    if draft_tokens is None:
        draft_tokens = torch.empty((B, num_nodes), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(256, dtype=torch.uint8, device=dev)
    if pool is None:
        _check(_lib.tree_rerank(_ptr(node_parent), _ptr(node_token), _ptr(node_score), B, M, num_nodes,
                                _ptr(tree_parents), _ptr(draft_tokens), _ptr(workspace), workspace.numel(),
                                _stream_handle(stream, dev)))
    else:
        _need(pool, "pool", torch.int32, dev)
        _check(_lib.tree_rerank_pool(_ptr(node_parent), _ptr(node_token), _ptr(node_score), _ptr(pool),
                                     pool.shape[1], B, M, num_nodes, _ptr(tree_parents), _ptr(draft_tokens),
                                     _ptr(workspace), workspace.numel(), _stream_handle(stream, dev)))
    return tree_parents, draft_tokens


def read_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise and return the device status word of the last call that used `workspace`."""
    st = ctypes.c_uint32(0)
    _check(_lib.treespec_read_status(_ptr(workspace), ctypes.byref(st),
                                     _stream_handle(stream, workspace.device)))
    return int(st.value)


def raw_library() -> ctypes.CDLL:
    """The loaded C library (for callers that pass raw pointers)."""
    return _lib
