"""Float64 CPU oracle for MLA chunked-context prefill.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import anything from this package.  The
product path (``mla_chunked_context_gb300``) never imports it, and it imports
nothing from the product path: the two share no code.  The only thing both
sides consume is the seeded input generator module
``mla_chunked_context_gb300.workloads``, which holds no arithmetic of the
method and which this package does not import either (inputs are passed in).

Modules
-------
planner  -- the context-chunk planner and its split search
            (PR #50613 report, "key source snippets": plan_mla_context_chunks,
            aligned_split_len) plus the per-chunk metadata of section
            "implementation breakdown" item 2.
mla      -- gather, W_kv_b up-projection, varlen softmax attention with LSE,
            the LSE merge with prefix_num_tokens (PR #36540 report,
            "implementation breakdown", CUDA kernel layer), the empty-context
            partial (PR #49294 report, test_mask_empty_context; PR #50613
            report, item 3), the chunked prefill loop and an unchunked
            reference over the full context.

Every function is pinned by ``tests/test_oracle_pins.py`` against values the
pages print, closed forms, brute force on tiny inputs, or a library routine
computing the same quantity by another route.  No function here is
"parity unpinned".
"""

from . import planner, mla  # noqa: F401
