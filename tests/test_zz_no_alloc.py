"""The no-alloc chunk entry point against the workspace one.

mla_context_chunk_attn_noalloc is for callers that cannot allocate device
memory themselves (for example a plugin whose host framework owns every
device allocation and gives it no workspace): it runs the same chunk pipeline
with its scratch in a library-owned device array.  This test calls it through
the C ABI for every chunk of a multi-chunk batch, twice in a row (the array
keeps the previous call's contents), and checks each result against
mla_context_chunk_attn with a caller-provided workspace, within the
attention tolerance the other parity tests use.  It also checks that a chunk
too large for the array is refused with MLA_ERR_TOO_SMALL.

The file name makes pytest collect it last; it needs nothing from other tests.
"""

import numpy as np
import pytest
import torch

import mla_chunked_context_gb300 as M
from mla_chunked_context_gb300 import _lib
from mla_chunked_context_gb300 import workloads as W
from oracle import planner as P

pytestmark = pytest.mark.gpu


def _close(got, ref, atol, rtol):
    g = got.double().cpu().numpy()
    r = ref.double().cpu().numpy()
    both_nan = np.isnan(g) & np.isnan(r)
    both_ninf = np.isneginf(g) & np.isneginf(r)
    with np.errstate(invalid="ignore"):
        d = np.where(both_nan | both_ninf, 0.0, np.abs(g - r))
    lim = atol + rtol * np.abs(np.where(np.isfinite(r), r, 0.0))
    assert (d <= lim).all(), f"{int((~(d <= lim)).sum())} values outside tolerance"


def test_noalloc_matches_workspace_entry_two_calls():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required")
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    w = W.scaled(W.workload("uniform"), context_lens=[200, 0, 900, 50],
                 query_lens=[20, 5, 130, 9], num_heads=8, row_budget=512,
                 max_context_chunk=512, split_alignment=64, seed=46)
    x = W.make_inputs(w)
    g = {k: v.to(dev) for k, v in x.items()}
    d = M.Dims.of(w)
    T, H, Dv = w.num_tokens, w.num_heads, w.v_dim
    qsl = P.query_start_loc(w.query_lens)
    empty = P.empty_token_slices(w.context_lens, w.query_lens)
    chunks = M.mla_plan_context_chunks(w.context_lens, w.row_budget, w.max_context_chunk,
                                       w.split_alignment)
    assert len(chunks) >= 2 and any(c.is_continuation for c in chunks)

    def run(call):
        o = torch.full((T, H, Dv), float("nan"), device=dev)
        lse = torch.full((H, T), float("nan"), device=dev)
        M.mla_fill_empty_rows(o, lse, empty)
        for c in chunks:
            call(c, o, lse)
        torch.cuda.synchronize()
        return o, lse

    ws = torch.empty(M.mla_chunk_workspace_bytes(d, max(c.rows for c in chunks),
                                                 max(c.request_end - c.request_start
                                                     for c in chunks)),
                     dtype=torch.uint8, device=dev)
    ref_o, ref_l = run(lambda c, o, l: M.mla_context_chunk_attn(
        d, c, qsl, g["q"], g["kv_cache"], g["block_table"], g["w_kv_b"], ws, o, l))
    # every row of the partial is written (the last request has context, so
    # no token lies past prefix_num_tokens): a row both paths left unwritten
    # would otherwise compare equal as NaN against NaN
    assert not torch.isnan(ref_o).any() and not torch.isnan(ref_l).any()
    for _ in range(2):
        got_o, got_l = run(lambda c, o, l: M.mla_context_chunk_attn_noalloc(
            d, c, qsl, g["q"], g["kv_cache"], g["block_table"], g["w_kv_b"], o, l))
        assert not torch.isnan(got_o).any() and not torch.isnan(got_l).any()
        _close(got_o, ref_o, 2e-2, 2e-2)
        _close(got_l, ref_l, 1e-3, 0.0)
    assert M.mla_device_error_flags() == 0

    # a chunk whose workspace exceeds the array is refused before any launch
    big = M.Chunk(2, 3, [0], [900000], 900000, False)
    bt = torch.zeros(4, 900000 // w.block_size + 1, dtype=torch.int32, device=dev)
    with pytest.raises(M.MlaError) as e:
        M.mla_context_chunk_attn_noalloc(d, big, qsl, g["q"], g["kv_cache"], bt, g["w_kv_b"],
                                         ref_o, ref_l)
    assert e.value.code == _lib.MLA_ERR_TOO_SMALL
