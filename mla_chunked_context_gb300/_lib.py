"""ctypes binding of libmla_gb300.so (argument marshalling only).

Every function here has the name of a C-ABI entry point in
``include/mla_chunked_context.h`` and does nothing but check tensor shapes,
pass raw pointers and the current CUDA stream, and turn a negative status into
an exception.  All computation runs in the library's CUDA kernels; there is no
fallback: if the library is missing the first call raises.
"""

from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmla_gb300.so")
HEADER = os.path.join(HERE, "..", "include", "mla_chunked_context.h")

MLA_OK, MLA_ERR_INVALID, MLA_ERR_TOO_SMALL, MLA_ERR_PLANNER_STUCK, MLA_ERR_CUDA, \
    MLA_ERR_UNSUPPORTED = 0, -1, -2, -3, -4, -5
MLA_DTYPE_F32, MLA_DTYPE_BF16, MLA_DTYPE_F16 = 0, 1, 2
MLA_STATUS_BAD_BLOCK, MLA_STATUS_FP16_RANGE = 1, 2

_ERRORS = {MLA_ERR_INVALID: "invalid argument", MLA_ERR_TOO_SMALL: "buffer too small",
           MLA_ERR_PLANNER_STUCK: "planner cannot progress (budget below one aligned split)",
           MLA_ERR_CUDA: "CUDA error", MLA_ERR_UNSUPPORTED: "unsupported dims/dtype"}

EXPORTED = ("mla_plan_context_chunks", "merge_attn_states", "mla_gather_context_rows",
            "mla_kv_up_proj", "mla_varlen_attn", "mla_fill_empty_rows", "mla_mask_empty_context",
            "mla_chunk_workspace_bytes", "mla_context_chunk_attn", "mla_prefill_workspace_bytes",
            "mla_chunked_prefill", "mla_has_tcgen05", "mla_device_error_flags",
            "mla_chunk_kv_dtype", "mla_context_chunk_attn_noalloc",
            "mla_plan_equal_window_chunks", "mla_prefill_equal_window_workspace_bytes",
            "mla_chunked_prefill_equal_window", "mla_selftest_bounded_wait",
            "mla_kernel_launches", "mla_fused_attn_workspace_bytes",
            "mla_fused_context_attn", "mla_fused_attn_plan", "mla_prefill_pinned_bytes",
            "mla_profile_begin", "mla_profile_end", "mla_set_pipeline_overlap")
MLA_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


class MlaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {_ERRORS.get(code, 'error')} ({code})")
        self.code = code


class mla_dims_t(C.Structure):
    _fields_ = [("num_heads", C.c_int32), ("kv_lora_rank", C.c_int32),
                ("qk_rope_dim", C.c_int32), ("qk_nope_dim", C.c_int32), ("v_dim", C.c_int32),
                ("block_size", C.c_int32), ("softmax_scale", C.c_float), ("dtype", C.c_int32)]


class mla_chunk_t(C.Structure):
    _fields_ = [("request_start", C.c_int32), ("request_end", C.c_int32),
                ("entry_offset", C.c_int32), ("rows", C.c_int32),
                ("is_continuation", C.c_int32)]


class mla_launch_record_t(C.Structure):
    _fields_ = [("kernel", C.c_char * 40), ("role", C.c_char * 40), ("stream", C.c_int32),
                ("start_ms", C.c_float), ("ms", C.c_float)]


PADDED_ROWS_FN = C.CFUNCTYPE(C.c_int64, C.c_int64, C.c_void_p)

_lib = None


def lib() -> C.CDLL:
    """Load the library once; raise if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "mla_chunked_context_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        P, I32, I64, SZ = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
        sig = {
            "mla_plan_context_chunks": [P, I32, I32, I32, I32, PADDED_ROWS_FN, P, P, I32, P, P,
                                        I32, P, P],
            "merge_attn_states": [P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, P],
            "mla_gather_context_rows": [P, P, I32, P, I32, I32, P, P, P, I32, P, P, P],
            "mla_kv_up_proj": [P, P, I64, I32, P, P, I32, P, P],
            "mla_varlen_attn": [P, I32, I32, P, P, P, P, I32, P, P, I32, I32, P, I64, P, P, P, P,
                                P],
            "mla_fill_empty_rows": [P, P, I32, I32, I32, I32, P, P],
            "mla_mask_empty_context": [P, P, I32, I32, I32, I32, I32, P, P, P],
            "mla_chunk_workspace_bytes": [P, I32, I32, P],
            "mla_context_chunk_attn": [P, P, P, P, P, I32, P, P, I32, P, I32, P, P, SZ, P, P, P,
                                       P],
            "mla_prefill_workspace_bytes": [P, P, P, I32, I32, I32, I32, P],
            "mla_prefill_pinned_bytes": [P, P, P, I32, I32, I32, I32, P],
            "mla_chunked_prefill": [P, P, P, I32, I32, I32, I32, P, P, P, I32, P, I32, P, P, SZ,
                                    P, P, P, SZ, P, P],
            "mla_profile_begin": [],
            "mla_profile_end": [P, I32, P],
            "mla_has_tcgen05": [],
            "mla_kernel_launches": [P],
            "mla_fused_attn_workspace_bytes": [P, I32, P],
            "mla_fused_attn_plan": [I32, I32, P, P, I32, I32, P, I32, P, I32, P, P, P],
            "mla_fused_context_attn": [P, I32, P, P, P, P, I32, P, P, I64, I32, P, P, P, P, P,
                                       SZ, P, P],
            "mla_device_error_flags": [P],
            "mla_chunk_kv_dtype": [P, P],
            "mla_context_chunk_attn_noalloc": [P, P, P, P, P, I32, P, P, I32, P, I32, P, P, P,
                                               P, P],
            "mla_plan_equal_window_chunks": [P, I32, I32, I32, P, P],
            "mla_selftest_bounded_wait": [I32, P, P],
            "mla_prefill_equal_window_workspace_bytes": [P, P, P, I32, I32, I32, P],
            "mla_chunked_prefill_equal_window": [P, P, P, I32, I32, I32, P, P, P, I32, P, I32, P,
                                                 P, SZ, P, P, P, P],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = C.c_int
        _lib = L
    return _lib


def _check(code: int, where: str):
    if code != MLA_OK:
        raise MlaError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return C.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _i32_host(xs: Sequence[int]):
    arr = (C.c_int32 * max(1, len(xs)))(*[int(x) for x in xs])
    return arr


def dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return MLA_DTYPE_BF16
    if t == torch.float32:
        return MLA_DTYPE_F32
    if t == torch.float16:
        return MLA_DTYPE_F16
    raise ValueError(f"unsupported dtype {t}")


_TORCH_OF = {MLA_DTYPE_F32: torch.float32, MLA_DTYPE_BF16: torch.bfloat16,
             MLA_DTYPE_F16: torch.float16}


@dataclass
class Dims:
    num_heads: int
    kv_lora_rank: int
    qk_rope_dim: int
    qk_nope_dim: int
    v_dim: int
    block_size: int
    softmax_scale: float
    dtype: torch.dtype

    def c(self) -> mla_dims_t:
        return mla_dims_t(self.num_heads, self.kv_lora_rank, self.qk_rope_dim, self.qk_nope_dim,
                          self.v_dim, self.block_size, self.softmax_scale,
                          dtype_code(self.dtype))

    @classmethod
    def of(cls, w) -> "Dims":
        return cls(w.num_heads, w.kv_lora_rank, w.qk_rope_dim, w.qk_nope_dim, w.v_dim,
                   w.block_size, w.softmax_scale, w.torch_dtype)


@dataclass
class Chunk:
    request_start: int
    request_end: int
    starts: list
    seq_lens: list
    rows: int
    is_continuation: bool


# --------------------------------------------------------------------------
def mla_plan_context_chunks(context_lens: Sequence[int], row_budget: int,
                            max_context_chunk: int, split_alignment: int,
                            padded_rows=None) -> list:
    L = lib()
    n = len(context_lens)
    ctx = _i32_host(context_lens)
    nc, ne = C.c_int32(0), C.c_int32(0)
    cb = PADDED_ROWS_FN(lambda x, _ctx: int(padded_rows(int(x)))) if padded_rows else \
        C.cast(None, PADDED_ROWS_FN)
    _check(L.mla_plan_context_chunks(ctx, n, row_budget, max_context_chunk, split_alignment,
                                     cb, None, None, 0, None, None, 0, C.byref(nc),
                                     C.byref(ne)), "mla_plan_context_chunks")
    chunks = (mla_chunk_t * max(1, nc.value))()
    starts = (C.c_int32 * max(1, ne.value))()
    lens = (C.c_int32 * max(1, ne.value))()
    _check(L.mla_plan_context_chunks(ctx, n, row_budget, max_context_chunk, split_alignment,
                                     cb, None, chunks, nc.value, starts, lens, ne.value,
                                     C.byref(nc), C.byref(ne)), "mla_plan_context_chunks")
    out = []
    for i in range(nc.value):
        c = chunks[i]
        k = c.request_end - c.request_start
        out.append(Chunk(c.request_start, c.request_end,
                         [starts[c.entry_offset + j] for j in range(k)],
                         [lens[c.entry_offset + j] for j in range(k)], c.rows,
                         bool(c.is_continuation)))
    return out


def merge_attn_states(out: torch.Tensor, out_lse: Optional[torch.Tensor],
                      prefix_o: torch.Tensor, prefix_lse: torch.Tensor,
                      suffix_o: torch.Tensor, suffix_lse: torch.Tensor,
                      prefix_num_tokens: int, stream=None) -> None:
    T, H, D = suffix_o.shape
    assert prefix_o.shape == suffix_o.shape and out.shape == suffix_o.shape
    assert prefix_lse.shape == (H, T) and suffix_lse.shape == (H, T)
    assert prefix_lse.dtype == torch.float32 and suffix_lse.dtype == torch.float32
    assert prefix_o.dtype == suffix_o.dtype
    for t in (out, prefix_o, suffix_o, prefix_lse, suffix_lse):
        assert t.is_cuda and t.is_contiguous()
    if out_lse is not None:
        assert out_lse.shape == (H, T) and out_lse.dtype == torch.float32
    _check(lib().merge_attn_states(_ptr(out), _ptr(out_lse), _ptr(prefix_o), _ptr(prefix_lse),
                                   _ptr(suffix_o), _ptr(suffix_lse), T, H, D, prefix_num_tokens,
                                   dtype_code(suffix_o.dtype), dtype_code(out.dtype),
                                   _stream(stream)), "merge_attn_states")


def mla_gather_context_rows(dims: Dims, kv_cache, block_table, seq_request, seq_start, cu_rows,
                            total_rows: int, latent_ws, dev_status=None, stream=None) -> None:
    d = dims.c()
    _check(lib().mla_gather_context_rows(C.byref(d), _ptr(kv_cache), kv_cache.shape[0],
                                         _ptr(block_table), block_table.shape[1],
                                         seq_request.numel(), _ptr(seq_request), _ptr(seq_start),
                                         _ptr(cu_rows), total_rows, _ptr(latent_ws),
                                         _ptr(dev_status), _stream(stream)),
           "mla_gather_context_rows")


def mla_kv_up_proj(dims: Dims, latent, rows: int, w_kv_b, kv, dev_status=None,
                   stream=None) -> None:
    """kv's torch dtype (float32 / bfloat16 / float16) selects the output type."""
    d = dims.c()
    _check(lib().mla_kv_up_proj(C.byref(d), _ptr(latent), latent.stride(0), rows, _ptr(w_kv_b),
                                _ptr(kv), dtype_code(kv.dtype), _ptr(dev_status),
                                _stream(stream)), "mla_kv_up_proj")


def mla_varlen_attn(dims: Dims, causal: bool, q_loc: Sequence[int], k_loc: Sequence[int], q,
                    kv, latent, o, lse, accumulate: Optional[Sequence[int]] = None,
                    stream=None, q_loc_dev=None, k_loc_dev=None, accumulate_dev=None,
                    kv_rows: Optional[int] = None, dev_status=None) -> None:
    """q_loc / k_loc (and accumulate) are host sequences; they are copied to
    the device here unless device copies are passed as *_dev tensors.  kv is
    head-major [H, kv_rows, Dn+Dv]; kv_rows defaults to k_loc[-1]."""
    n = len(q_loc) - 1
    dev = q.device
    ql = q_loc_dev if q_loc_dev is not None else torch.tensor(list(q_loc), dtype=torch.int32,
                                                              device=dev)
    kl = k_loc_dev if k_loc_dev is not None else torch.tensor(list(k_loc), dtype=torch.int32,
                                                              device=dev)
    acc = accumulate_dev
    if acc is None and accumulate:
        acc = torch.tensor(list(accumulate), dtype=torch.int32, device=dev)
    d = dims.c()
    rows = int(k_loc[-1]) if kv_rows is None else int(kv_rows)
    _check(lib().mla_varlen_attn(C.byref(d), int(causal), n, _ptr(ql), _ptr(kl),
                                 _i32_host(q_loc), _i32_host(k_loc), q.shape[0], _ptr(q),
                                 _ptr(kv), dtype_code(kv.dtype), rows, _ptr(latent),
                                 latent.stride(0), _ptr(acc), _ptr(o), _ptr(lse),
                                 _ptr(dev_status), _stream(stream)), "mla_varlen_attn")


def mla_fused_attn_workspace_bytes(dims: Dims, num_tokens: int) -> int:
    d = dims.c()
    n = C.c_size_t(0)
    _check(lib().mla_fused_attn_workspace_bytes(C.byref(d), int(num_tokens), C.byref(n)),
           "mla_fused_attn_workspace_bytes")
    return int(n.value)


def mla_fused_context_attn(dims: Dims, q_loc: Sequence[int], k_loc: Sequence[int], q, latent,
                           w_kv_b, o, lse, accumulate: Optional[Sequence[int]] = None,
                           workspace=None, stream=None, q_loc_dev=None, k_loc_dev=None,
                           accumulate_dev=None, dev_status=None) -> None:
    """Context attention with the up-projection fused in: latent rows
    [k_loc[i], k_loc[i+1]) are sequence i's keys.  workspace: a uint8 device
    tensor of mla_fused_attn_workspace_bytes bytes (allocated here if None)."""
    n = len(q_loc) - 1
    dev = q.device
    ql = q_loc_dev if q_loc_dev is not None else torch.tensor(list(q_loc), dtype=torch.int32,
                                                              device=dev)
    kl = k_loc_dev if k_loc_dev is not None else torch.tensor(list(k_loc), dtype=torch.int32,
                                                              device=dev)
    acc = accumulate_dev
    if acc is None and accumulate:
        acc = torch.tensor(list(accumulate), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(mla_fused_attn_workspace_bytes(dims, q.shape[0]),
                                dtype=torch.uint8, device=dev)
    d = dims.c()
    _check(lib().mla_fused_context_attn(C.byref(d), n, _ptr(ql), _ptr(kl), _i32_host(q_loc),
                                        _i32_host(k_loc), q.shape[0], _ptr(q), _ptr(latent),
                                        latent.stride(0), latent.shape[0], _ptr(w_kv_b),
                                        _ptr(acc), _ptr(o), _ptr(lse), _ptr(workspace),
                                        workspace.numel(), _ptr(dev_status), _stream(stream)),
           "mla_fused_context_attn")


def mla_fused_attn_plan(num_heads: int, q_loc: Sequence[int], k_loc: Sequence[int],
                        clusters: int, split_slots: int):
    """The fused kernel's work split (host only): (bounds, items, groups)
    with items as (sequence, key tiles, first tile, slot info) tuples."""
    L = lib()
    n = len(q_loc) - 1
    ql, kl = _i32_host(q_loc), _i32_host(k_loc)
    nc, ni, ng = C.c_int32(0), C.c_int32(0), C.c_int32(0)
    _check(L.mla_fused_attn_plan(num_heads, n, ql, kl, clusters, split_slots, None, 0, None, 0,
                                 C.byref(nc), C.byref(ni), C.byref(ng)), "mla_fused_attn_plan")
    b = (C.c_int32 * (nc.value + 1))()
    it = (C.c_int32 * max(1, 4 * ni.value))()
    _check(L.mla_fused_attn_plan(num_heads, n, ql, kl, clusters, split_slots, b, nc.value + 1,
                                 it, ni.value, C.byref(nc), C.byref(ni), C.byref(ng)),
           "mla_fused_attn_plan")
    items = [tuple(it[4 * i:4 * i + 4]) for i in range(ni.value)]
    return list(b), items, ng.value


def mla_fill_empty_rows(o, lse, slices: Sequence, stream=None) -> None:
    T, H, Dv = o.shape
    flat = [int(x) for s in slices for x in s]
    sl = torch.tensor(flat or [0, 0], dtype=torch.int32, device=o.device)
    _check(lib().mla_fill_empty_rows(_ptr(o), _ptr(lse), T, H, Dv, len(slices), _ptr(sl),
                                     _stream(stream)), "mla_fill_empty_rows")


def mla_mask_empty_context(lse, o, query_start_loc, context_start_loc, stream=None) -> None:
    T, H, D = o.shape
    R = query_start_loc.numel() - 1
    _check(lib().mla_mask_empty_context(_ptr(lse), _ptr(o), dtype_code(o.dtype), T, H, D, R,
                                        _ptr(query_start_loc), _ptr(context_start_loc),
                                        _stream(stream)), "mla_mask_empty_context")


def mla_chunk_workspace_bytes(dims: Dims, max_rows: int, max_entries: int) -> int:
    d = dims.c()
    b = C.c_size_t(0)
    _check(lib().mla_chunk_workspace_bytes(C.byref(d), max_rows, max_entries, C.byref(b)),
           "mla_chunk_workspace_bytes")
    return b.value


def mla_context_chunk_attn(dims: Dims, chunk: Chunk, query_start_loc: Sequence[int], q,
                           kv_cache, block_table, w_kv_b, workspace, o_partial, lse_partial,
                           dev_status=None, stream=None) -> None:
    d = dims.c()
    n = chunk.request_end - chunk.request_start
    c = mla_chunk_t(chunk.request_start, chunk.request_end, 0, chunk.rows,
                    int(chunk.is_continuation))
    _check(lib().mla_context_chunk_attn(
        C.byref(d), C.byref(c), _i32_host(chunk.starts), _i32_host(chunk.seq_lens),
        _i32_host(query_start_loc), q.shape[0], _ptr(q), _ptr(kv_cache), kv_cache.shape[0],
        _ptr(block_table), block_table.shape[1], _ptr(w_kv_b), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(o_partial), _ptr(lse_partial),
        _ptr(dev_status), _stream(stream)), "mla_context_chunk_attn")
    assert n >= 1


def mla_context_chunk_attn_noalloc(dims: Dims, chunk: Chunk, query_start_loc: Sequence[int], q,
                                   kv_cache, block_table, w_kv_b, o_partial, lse_partial,
                                   dev_status=None, stream=None) -> None:
    """mla_context_chunk_attn with the library's own device scratch array
    (for callers that cannot allocate device memory; see the C header)."""
    d = dims.c()
    c = mla_chunk_t(chunk.request_start, chunk.request_end, 0, chunk.rows,
                    int(chunk.is_continuation))
    _check(lib().mla_context_chunk_attn_noalloc(
        C.byref(d), C.byref(c), _i32_host(chunk.starts), _i32_host(chunk.seq_lens),
        _i32_host(query_start_loc), q.shape[0], _ptr(q), _ptr(kv_cache), kv_cache.shape[0],
        _ptr(block_table), block_table.shape[1], _ptr(w_kv_b), _ptr(o_partial),
        _ptr(lse_partial), _ptr(dev_status), _stream(stream)), "mla_context_chunk_attn_noalloc")


def mla_prefill_workspace_bytes(dims: Dims, context_lens, query_lens, row_budget: int,
                                max_context_chunk: int, split_alignment: int) -> int:
    d = dims.c()
    b = C.c_size_t(0)
    _check(lib().mla_prefill_workspace_bytes(C.byref(d), _i32_host(context_lens),
                                             _i32_host(query_lens), len(context_lens),
                                             row_budget, max_context_chunk, split_alignment,
                                             C.byref(b)), "mla_prefill_workspace_bytes")
    return b.value


def mla_prefill_pinned_bytes(dims: Dims, context_lens, query_lens, row_budget: int,
                             max_context_chunk: int, split_alignment: int) -> int:
    d = dims.c()
    b = C.c_size_t(0)
    _check(lib().mla_prefill_pinned_bytes(C.byref(d), _i32_host(context_lens),
                                          _i32_host(query_lens), len(context_lens), row_budget,
                                          max_context_chunk, split_alignment, C.byref(b)),
           "mla_prefill_pinned_bytes")
    return b.value


def mla_chunked_prefill(dims: Dims, context_lens, query_lens, row_budget: int,
                        max_context_chunk: int, split_alignment: int, q, new_latent, kv_cache,
                        block_table, w_kv_b, workspace, out, out_lse=None, dev_status=None,
                        stream=None, pinned_scratch=None) -> None:
    """pinned_scratch: optional page-locked uint8 host tensor of at least
    mla_prefill_pinned_bytes bytes for the metadata upload."""
    d = dims.c()
    pin = _ptr(pinned_scratch)
    pin_bytes = 0 if pinned_scratch is None else pinned_scratch.numel() * \
        pinned_scratch.element_size()
    _check(lib().mla_chunked_prefill(
        C.byref(d), _i32_host(context_lens), _i32_host(query_lens), len(context_lens),
        row_budget, max_context_chunk, split_alignment, _ptr(q), _ptr(new_latent),
        _ptr(kv_cache), kv_cache.shape[0], _ptr(block_table), block_table.shape[1],
        _ptr(w_kv_b), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out),
        _ptr(out_lse), pin, pin_bytes, _ptr(dev_status), _stream(stream)),
        "mla_chunked_prefill")


def mla_has_tcgen05() -> bool:
    return bool(lib().mla_has_tcgen05())


def mla_set_pipeline_overlap(on: bool) -> bool:
    """Overlap the chunk pipeline's gathers and up-projections with the
    attention on side streams (True, the default) or run every kernel of a
    prefill on the caller's stream in order (False); returns the previous
    setting."""
    L = lib()
    L.mla_set_pipeline_overlap.restype = C.c_int32
    return bool(L.mla_set_pipeline_overlap(C.c_int32(1 if on else 0)))


def mla_profile_begin() -> None:
    """Record CUDA events around every kernel this thread's calls enqueue."""
    _check(lib().mla_profile_begin(), "mla_profile_begin")


def mla_profile_end(cap: int = 8192) -> list:
    """Stop profiling; (kernel, stream, start_ms, ms, role) per launch, in
    launch order."""
    recs = (mla_launch_record_t * cap)()
    n = C.c_int32(0)
    _check(lib().mla_profile_end(recs, cap, C.byref(n)), "mla_profile_end")
    return [(recs[i].kernel.decode(), recs[i].stream, recs[i].start_ms, recs[i].ms,
             recs[i].role.decode()) for i in range(n.value)]


def mla_kernel_launches() -> int:
    """Kernels the library has enqueued since it was loaded (all threads)."""
    n = C.c_uint64(0)
    _check(lib().mla_kernel_launches(C.byref(n)), "mla_kernel_launches")
    return n.value


def mla_device_error_flags() -> int:
    f = C.c_int32(0)
    _check(lib().mla_device_error_flags(C.byref(f)), "mla_device_error_flags")
    return f.value


def mla_chunk_kv_dtype(dims: Dims) -> torch.dtype:
    d = dims.c()
    k = C.c_int32(0)
    _check(lib().mla_chunk_kv_dtype(C.byref(d), C.byref(k)), "mla_chunk_kv_dtype")
    return _TORCH_OF[k.value]


def mla_plan_equal_window_chunks(context_lens: Sequence[int], row_budget: int,
                                 split_alignment: int):
    """(window, number of chunks) of the old equal-window scheme."""
    w, n = C.c_int32(0), C.c_int32(0)
    _check(lib().mla_plan_equal_window_chunks(_i32_host(context_lens), len(context_lens),
                                              row_budget, split_alignment, C.byref(w),
                                              C.byref(n)), "mla_plan_equal_window_chunks")
    return w.value, n.value


def mla_prefill_equal_window_workspace_bytes(dims: Dims, context_lens, query_lens,
                                             row_budget: int, split_alignment: int) -> int:
    d = dims.c()
    b = C.c_size_t(0)
    _check(lib().mla_prefill_equal_window_workspace_bytes(
        C.byref(d), _i32_host(context_lens), _i32_host(query_lens), len(context_lens),
        row_budget, split_alignment, C.byref(b)), "mla_prefill_equal_window_workspace_bytes")
    return b.value


def mla_chunked_prefill_equal_window(dims: Dims, context_lens, query_lens, row_budget: int,
                                     split_alignment: int, q, new_latent, kv_cache, block_table,
                                     w_kv_b, workspace, out, out_lse=None, dev_status=None,
                                     stream=None) -> None:
    d = dims.c()
    _check(lib().mla_chunked_prefill_equal_window(
        C.byref(d), _i32_host(context_lens), _i32_host(query_lens), len(context_lens),
        row_budget, split_alignment, _ptr(q), _ptr(new_latent), _ptr(kv_cache),
        kv_cache.shape[0], _ptr(block_table), block_table.shape[1], _ptr(w_kv_b),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), _ptr(out_lse),
        _ptr(dev_status), _stream(stream)), "mla_chunked_prefill_equal_window")


def mla_selftest_bounded_wait(limit_us: int, gave_up, stream=None) -> None:
    """Run the bounded-wait self test (gave_up: device int32 tensor)."""
    _check(lib().mla_selftest_bounded_wait(int(limit_us), _ptr(gave_up), _stream(stream)),
           "mla_selftest_bounded_wait")
