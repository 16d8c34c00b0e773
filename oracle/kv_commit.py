"""Keep the accepted path's K/V, drop the rejected branches.  TEST INFRASTRUCTURE ONLY.

"Tech Radar: SGLang EAGLE-2", section 2 (the verification sequence): after the target's
pass over the tree, the accepted path's KV is retained and the rejected branches are
discarded.  "EAGLE-2 & Lookahead Decoding", section 6 (paged tree KV-cache allocation):
the positions of rejected candidates return to the pool.

Reading (the pages fix no layout): during verification tree node n of a sequence sits at
logical position S + n after its S prefix tokens, node 0 being the root.  Retaining the
accepted path means the sequence becomes the prefix, the root, and the accepted nodes in
path order -- node path[k] moves to position S + 1 + k -- and its length S + 1 + len;
everything after that is free.  All values are copied exactly (no arithmetic).

The positions a commit touches are S (the root, which stays) through S + max(path) (the
deepest source; every destination S + 1 + k lies at or before it because a strictly
increasing path from 1 has path[k] >= k + 1).  Those positions must lie in the page
table: S + 1 + max(path) <= pages * page_size, with max(path) = 0 for an empty path.  The
tree's node count does not enter the bound, so a tree smaller than the batch's N (a row
padded after its last node) commits whenever its own accepted path fits.

A sequence whose prefix length, path or pages are invalid is left untouched and reports
new length -1 with a status flag, as the CUDA entry point does.
"""
from __future__ import annotations

import numpy as np

BAD_PAGE, BAD_LENGTH, BAD_PATH = 2, 4, 64


def kv_commit(k_pages: np.ndarray, v_pages: np.ndarray, page_table: np.ndarray, prefix_lens: np.ndarray,
              accept_path: np.ndarray, accept_len: np.ndarray, num_nodes: int):
    """Returns (k_new, v_new, new_lens, status).  Pools are [P][page_size][Hkv][D]."""
    P, ps = k_pages.shape[0], k_pages.shape[1]
    B, max_pages = page_table.shape
    k_new, v_new = k_pages.copy(), v_pages.copy()
    new_lens = np.full(B, -1, dtype=np.int64)
    status = 0
    for b in range(B):
        S, n = int(prefix_lens[b]), int(accept_len[b])
        bad = 0
        path = [int(x) for x in accept_path[b, :max(n, 0)]] if 0 <= n <= num_nodes - 1 else None
        if path is None or any(x >= num_nodes for x in path) or any(
                x <= prev for prev, x in zip([0] + path[:-1], path)):
            bad |= BAD_PATH
        top = path[-1] if (not bad and path) else 0              # deepest position touched: S + top
        if S < 0 or S + 1 + top > max_pages * ps:
            bad |= BAD_LENGTH
        if bad:
            status |= bad
            continue
        moves = [(S + path[k], S + 1 + k) for k in range(n)]    # (source, destination) positions
        pages = [int(page_table[b, pos // ps]) for mv in moves for pos in mv]
        if any(not 0 <= pg < P for pg in pages):
            status |= BAD_PAGE
            continue
        for src, dst in moves:                                  # every value comes from the old pool
            sp, so = int(page_table[b, src // ps]), src % ps
            dp, do = int(page_table[b, dst // ps]), dst % ps
            k_new[dp, do] = k_pages[sp, so]
            v_new[dp, do] = v_pages[sp, so]
        new_lens[b] = S + 1 + n
    return k_new, v_new, new_lens, status


def logical_rows(pool: np.ndarray, page_table_row: np.ndarray, length: int) -> np.ndarray:
    """The first `length` logical positions of one sequence, gathered through its page table."""
    ps = pool.shape[1]
    return np.stack([pool[int(page_table_row[t // ps]), t % ps] for t in range(length)]) if length else \
        np.zeros((0,) + pool.shape[2:], pool.dtype)
