"""MLA chunked-context prefill for NVIDIA GB300 (sm_103a).

The computation lives in ``libmla_gb300.so`` (hand-written CUDA kernels behind
a C ABI, ``include/mla_chunked_context.h``).  This package is the thin Python
binding: the functions below carry the C entry points' names and only
marshal arguments; PyTorch provides device memory and streams.
"""

from ._lib import (Chunk, Dims, MlaError, lib, merge_attn_states, mla_chunk_kv_dtype,
                   mla_chunk_workspace_bytes, mla_device_error_flags,
                   mla_chunked_prefill, mla_context_chunk_attn, mla_context_chunk_attn_noalloc,
                   mla_fill_empty_rows,
                   mla_gather_context_rows, mla_has_tcgen05, mla_kv_up_proj,
                   mla_mask_empty_context, mla_plan_context_chunks, mla_prefill_workspace_bytes,
                   mla_varlen_attn, MLA_STATUS_BAD_BLOCK, mla_plan_equal_window_chunks,
                   mla_prefill_equal_window_workspace_bytes, mla_chunked_prefill_equal_window,
                   mla_selftest_bounded_wait, mla_kernel_launches,
                   mla_fused_attn_workspace_bytes, mla_fused_context_attn,
                   mla_fused_attn_plan, mla_prefill_pinned_bytes, mla_profile_begin,
                   mla_profile_end, mla_set_pipeline_overlap, MLA_STATUS_FP16_RANGE)

__all__ = ["Chunk", "Dims", "MlaError", "lib", "merge_attn_states", "mla_chunk_kv_dtype",
           "mla_chunk_workspace_bytes", "mla_device_error_flags",
           "mla_chunked_prefill", "mla_context_chunk_attn", "mla_context_chunk_attn_noalloc",
           "mla_fill_empty_rows",
           "mla_gather_context_rows", "mla_has_tcgen05", "mla_kv_up_proj",
           "mla_mask_empty_context", "mla_plan_context_chunks", "mla_prefill_workspace_bytes",
           "mla_varlen_attn", "MLA_STATUS_BAD_BLOCK", "mla_plan_equal_window_chunks",
           "mla_prefill_equal_window_workspace_bytes", "mla_chunked_prefill_equal_window",
           "mla_selftest_bounded_wait", "mla_kernel_launches", "mla_fused_attn_workspace_bytes",
           "mla_fused_context_attn", "mla_fused_attn_plan", "mla_prefill_pinned_bytes",
           "mla_profile_begin", "mla_profile_end", "mla_set_pipeline_overlap",
           "MLA_STATUS_FP16_RANGE", "ChunkedPrefill"]


class ChunkedPrefill:
    """Holds the device workspace (a torch uint8 tensor) and the pinned host
    metadata scratch for one batch shape and runs ``mla_chunked_prefill`` on
    them."""

    def __init__(self, dims: Dims, context_lens, query_lens, row_budget: int,
                 max_context_chunk: int, split_alignment: int, device="cuda"):
        import torch
        self.dims = dims
        self.context_lens = [int(x) for x in context_lens]
        self.query_lens = [int(x) for x in query_lens]
        self.row_budget = int(row_budget)
        self.max_context_chunk = int(max_context_chunk)
        self.split_alignment = int(split_alignment)
        self.workspace_bytes = mla_prefill_workspace_bytes(
            dims, self.context_lens, self.query_lens, self.row_budget, self.max_context_chunk,
            self.split_alignment)
        self.workspace = torch.empty(max(1, self.workspace_bytes), dtype=torch.uint8,
                                     device=device)
        pinned = mla_prefill_pinned_bytes(dims, self.context_lens, self.query_lens,
                                          self.row_budget, self.max_context_chunk,
                                          self.split_alignment)
        self.pinned = torch.empty(max(16, pinned), dtype=torch.uint8, pin_memory=True)

    def __call__(self, q, new_latent, kv_cache, block_table, w_kv_b, out, out_lse=None,
                 dev_status=None, stream=None):
        mla_chunked_prefill(self.dims, self.context_lens, self.query_lens, self.row_budget,
                            self.max_context_chunk, self.split_alignment, q, new_latent,
                            kv_cache, block_table, w_kv_b, self.workspace, out, out_lse,
                            dev_status, stream, pinned_scratch=self.pinned)
        return out
