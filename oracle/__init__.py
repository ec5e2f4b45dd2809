"""CPU oracle for the self-speculative verification step.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import it.  The product
path (the ``libspecverify`` C-ABI and its Python binding) never imports,
links or calls anything here, and this package imports nothing from the
product path.  Every function is float64 numpy following the pages' own
definitions; see ``specverify_oracle`` for the citations and readings.

Pinning status: every function here is pinned by ``-m "not gpu"`` tests
(golden LA diagram, closed forms, library special cases, brute force,
planted generator expectations).  No function is "parity unpinned".
"""

from .specverify_oracle import (  # noqa: F401
    VP_PAD, VP_ROOT, MODE_GREEDY_TREE, MODE_THRESH_CHAIN,
    la_prefill_mask, la_prefill_attention, la_prefill_vparent, mask_build, verify_attention, gather_paged,
    vocab_reduce, accept, accept_threshold_chain, accept_greedy_tree,
    softmax_t, residual_sample, accept_soft_tree, accept_soft,
    topk_tokens, draft_tree, prune_tree, ss_block_vparent,
    rotate_stream_values, future_gather,
    kv_commit_contiguous, kv_commit_paged,
)
