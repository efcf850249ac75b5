"""CPU oracle for tree verification — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct NumPy (float64) statement of what the
verification hot path computes, written from the method descriptions:

* ``attention``  — one target forward over all draft-tree nodes against the
  context KV cache (full, or a SpecPV partial page list), with an explicit
  N x (L' + N) visibility mask (ancestor-or-self inside the tree).
* ``accept``     — greedy (temperature 0) acceptance: the longest accepted
  root path and its bonus token.
* ``commit``     — the KV cache after the accepted path is written to slots
  L .. L + a.
* ``retrieval``  — SpecPV block retrieval: max/min key summaries of 16-token
  pages, block importance against the tree's queries, the partial page list;
  the full/partial schedule and the tree of a full verification that
  re-verifies the buffer of partially verified tokens.
* ``sampling``   — stochastic (temperature > 0) acceptance: speculative
  sampling node by node over the tree, residual draws for the bonus token.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The CUDA library never calls it and
shares no code with it.

Pins: every function here is checked in ``tests/test_oracle_*.py`` against
library routines, closed forms, invariants, the SpecBlock Appendix A.2 mask
example, brute force and (for sampling) the distribution speculative sampling
must reproduce.  Nothing here is "parity unpinned".
"""

from .attention import (  # noqa: F401
    ancestor_or_self_mask,
    bf16_to_f64,
    context_positions,
    tree_verify_attention,
    visibility_mask,
)
from .accept import greedy_accept  # noqa: F401
from .commit import kv_commit  # noqa: F401
from .sampling import inverse_cdf, node_verify, speculative_tree_accept, target_probs  # noqa: F401
from .retrieval import (  # noqa: F401
    extend_partial_lists,
    specpv_schedule,
    block_importance,
    page_regions,
    page_summaries,
    query_block_score,
    retrieve_pages,
    specpv_full_step_trees,
    specpv_full_tree,
)
