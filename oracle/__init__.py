"""Plain float64 CPU oracle for the tree-verify path.  TEST INFRASTRUCTURE ONLY.

This package is the independent statement of what the path computes, written
from the method's description; the CUDA library is checked against it.  Only
the test suite, the package smoke check and the bench's CPU-baseline leg may
import it.  It shares no code with the CUDA path and never imports it.

  tree_mask   -- ancestor sets, the dense tree mask M and its 64-bit words
  attention   -- tree attention over a paged KV cache (a definition)
  accept      -- greedy and rejection-sampling accept walks (an algorithm)
  kv_commit   -- keeping the accepted path's K/V after the walk (a definition)
  draft_tree  -- beam expansion by cumulative confidence and the final rerank (an algorithm)

Parity pins (tests that tie each function to something other than itself)
live in tests/test_oracle_*.py.  Unpinned: nothing in these functions; the
pages' "up to 42%" sibling-dedup saving and the entropy thresholds of the
dynamic tree are claims about a different system and are not modelled.
"""
from . import tree_mask, attention, accept, kv_commit, draft_tree  # noqa: F401
