"""The C ABI's contract on the GPU: the fp16 range status bit, refused
(misaligned) operands, the pinned metadata scratch, and the per-launch
profile.  Expected values come only from oracle/ (or from the library's own
other entry point where two paths must agree bit for bit)."""

import numpy as np
import pytest
import torch

import mla_chunked_context_gb300 as M
from mla_chunked_context_gb300 import _lib
from mla_chunked_context_gb300 import workloads as W
from oracle import mla as O

pytestmark = [pytest.mark.gpu,
              pytest.mark.filterwarnings("ignore::RuntimeWarning")]

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA GPU required for -m gpu tests")
    M.lib()
    torch.cuda.set_device(0)


@pytest.fixture(autouse=True)
def _no_device_errors():
    yield
    assert M.mla_device_error_flags() == 0, "a tensor-core kernel gave up waiting"


def f64(t):
    return t.detach().to("cpu").double().numpy()


def _small_batch(seed=90, heads=4):
    # DeepSeek-V3 head shape, a request split across chunks, a context-free one
    return W.scaled(W.workload("uniform"), context_lens=[0, 300, 700], query_lens=[4, 130, 9],
                    num_heads=heads, row_budget=512, max_context_chunk=512, seed=seed)


def _prefill(w, x, pinned=True):
    g = {k: v.to(DEV) for k, v in x.items()}
    T = w.num_tokens
    out = torch.full((T, w.num_heads, w.v_dim), float("nan"), dtype=w.torch_dtype, device=DEV)
    lse = torch.full((w.num_heads, T), float("nan"), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    d = M.Dims.of(w)
    args = (w.context_lens, w.query_lens, w.row_budget, w.max_context_chunk, w.split_alignment)
    ws = torch.empty(M.mla_prefill_workspace_bytes(d, *args), dtype=torch.uint8, device=DEV)
    pin = None
    if pinned:
        pin = torch.empty(M.mla_prefill_pinned_bytes(d, *args), dtype=torch.uint8,
                          pin_memory=True)
    M.mla_chunked_prefill(d, *args, g["q"], g["new_latent"], g["kv_cache"], g["block_table"],
                          g["w_kv_b"], ws, out, lse, status, pinned_scratch=pin)
    torch.cuda.synchronize()
    return out, lse, status.item()


def _oracle(w, x):
    n = {k: (f64(v) if v.is_floating_point() else v.numpy()) for k, v in x.items()}
    d = O.MlaDims(w.num_heads, w.kv_lora_rank, w.qk_rope_dim, w.qk_nope_dim, w.v_dim,
                  w.block_size, w.softmax_scale)
    ro, rl, _ = O.chunked_prefill(n["q"], n["new_latent"], n["kv_cache"], n["block_table"],
                                  n["w_kv_b"], w.context_lens, w.query_lens, d, w.row_budget,
                                  w.max_context_chunk, w.split_alignment)
    return ro, rl


def _matches(out, lse, ro, rl):
    o, l = f64(out), f64(lse)
    if np.isnan(o).any() or np.isnan(l).any():
        return False
    okl = np.where(np.isneginf(l) & np.isneginf(rl), True, np.abs(l - rl) <= 1e-3)
    return bool((np.abs(o - ro) <= 2e-2 + 2e-2 * np.abs(ro)).all() and okl.all())


# -------------------------------------------------------- fp16 range bit --
def test_fp16_range_of_q_nope_sets_status():
    """A few q_nope entries of 1e5 (representable in bf16, beyond fp16's
    65504): the tensor-core path rounds q_nope to fp16, so the result cannot
    be trusted, and the status bit says so (never NaN with status 0)."""
    w = _small_batch()
    x = W.make_inputs(w)
    x["q"][5, 1, 7] = 1e5
    x["q"][140, 3, 100] = -1e5
    out, lse, status = _prefill(w, x)
    assert status & _lib.MLA_STATUS_FP16_RANGE
    # the per-step attention converts q_nope in the kernel: same bit
    g = {k: v.to(DEV) for k, v in x.items()}
    kv = torch.zeros(w.num_heads, 64, 256, dtype=torch.float16, device=DEV)
    lat = torch.zeros(64, 576, dtype=torch.bfloat16, device=DEV)
    o = torch.empty(w.num_tokens, w.num_heads, 128, device=DEV)
    l = torch.empty(w.num_heads, w.num_tokens, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    T = w.num_tokens
    M.mla_varlen_attn(M.Dims.of(w), False, [0, T], [0, 64], g["q"], kv, lat, o, l, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & _lib.MLA_STATUS_FP16_RANGE


def test_fp16_range_of_kv_sets_status():
    """W_kv_b scaled so that up-projected K/V exceed 65504: the fp16 K/V of
    the tensor-core path overflow; the prefill either still matches the
    oracle or reports MLA_STATUS_FP16_RANGE (here it must report it), and the
    per-step GEMM reports it as well."""
    w = _small_batch(seed=91)
    x = W.make_inputs(w)
    x["w_kv_b"] = (x["w_kv_b"].float() * 1e5).to(torch.bfloat16)
    out, lse, status = _prefill(w, x)
    assert status & _lib.MLA_STATUS_FP16_RANGE
    ro, rl = _oracle(w, x)
    assert (status & _lib.MLA_STATUS_FP16_RANGE) or _matches(out, lse, ro, rl)
    g = {k: v.to(DEV) for k, v in x.items()}
    kv = torch.empty(w.num_tokens, w.num_heads * 256, dtype=torch.float16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    M.mla_kv_up_proj(M.Dims.of(w), g["new_latent"], w.num_tokens, g["w_kv_b"], kv, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & _lib.MLA_STATUS_FP16_RANGE
    # in range: the bit stays clear and the result matches the oracle
    x2 = W.make_inputs(w)
    out2, lse2, status2 = _prefill(w, x2)
    assert status2 == 0
    assert _matches(out2, lse2, *_oracle(w, x2))


# ------------------------------------------------- refused operands --
def test_misaligned_operands_are_refused_on_the_gpu():
    """An offset view (2 bytes off a 16-byte boundary) of q, or of a merge
    output, is refused with an error code; nothing runs on a slower path."""
    w = _small_batch(seed=92)
    x = W.make_inputs(w)
    g = {k: v.to(DEV) for k, v in x.items()}
    T, H = w.num_tokens, w.num_heads
    flat = torch.empty(T * H * 192 + 8, dtype=torch.bfloat16, device=DEV)
    q_odd = flat[1:1 + T * H * 192].view(T, H, 192)
    q_odd.copy_(g["q"])
    kv = torch.zeros(H, 64, 256, dtype=torch.float16, device=DEV)
    lat = torch.zeros(64, 576, dtype=torch.bfloat16, device=DEV)
    o = torch.empty(T, H, 128, device=DEV)
    l = torch.empty(H, T, device=DEV)
    with pytest.raises(M.MlaError) as e:
        M.mla_varlen_attn(M.Dims.of(w), False, [0, T], [0, 64], q_odd, kv, lat, o, l)
    assert e.value.code == _lib.MLA_ERR_UNSUPPORTED
    buf = torch.empty(T * H * 128 + 8, device=DEV)
    out_odd = buf[1:1 + T * H * 128].view(T, H, 128)
    so = torch.zeros(T, H, 128, device=DEV)
    sl = torch.zeros(H, T, device=DEV)
    with pytest.raises(M.MlaError) as e:
        M.merge_attn_states(out_odd, None, so, sl, so, sl, T)
    assert e.value.code == _lib.MLA_ERR_INVALID


# ------------------------------------------------- pinned metadata --
def test_pinned_and_pageable_metadata_give_the_same_result():
    """mla_chunked_prefill with the caller's pinned scratch and without it
    (pageable upload) computes the same numbers, bit for bit, call after
    call on one pinned buffer."""
    w = _small_batch(seed=93, heads=8)
    x = W.make_inputs(w)
    a_out, a_lse, sa = _prefill(w, x, pinned=False)
    b_out, b_lse, sb = _prefill(w, x, pinned=True)
    assert sa == 0 and sb == 0
    assert torch.equal(a_out, b_out) and torch.equal(a_lse, b_lse)
    pf = M.ChunkedPrefill(M.Dims.of(w), w.context_lens, w.query_lens, w.row_budget,
                          w.max_context_chunk, w.split_alignment, device=DEV)
    g = {k: v.to(DEV) for k, v in x.items()}
    outs = []
    for _ in range(3):
        out = torch.empty_like(a_out)
        pf(g["q"], g["new_latent"], g["kv_cache"], g["block_table"], g["w_kv_b"], out)
        outs.append(out)
    torch.cuda.synchronize()
    for out in outs:
        assert torch.equal(out, a_out)
    ro, rl = _oracle(w, x)
    assert _matches(a_out, a_lse, ro, rl)


# ------------------------------------------------- per-launch profile --
def test_profile_records_every_launch_of_a_prefill():
    """mla_profile_begin/_end around a prefill: one record per kernel the
    library enqueued (the launch counter agrees), with the tcgen05 kernels
    named, positive durations, and the gathers and GEMMs on side streams."""
    w = _small_batch(seed=94, heads=8)
    x = W.make_inputs(w)
    _prefill(w, x)                       # warm: streams, attributes
    n0 = M.mla_kernel_launches()
    M.mla_profile_begin()
    out, lse, status = _prefill(w, x)
    recs = M.mla_profile_end()
    launched = M.mla_kernel_launches() - n0
    assert status == 0
    assert len(recs) == launched > 0
    names = [r[0] for r in recs]
    assert "up_proj_tc_kernel" in names and "gather_bulk_kernel" in names
    assert any(n.startswith("attn_tc") for n in names)
    assert all(r[3] > 0 for r in recs) and all(r[2] >= 0 for r in recs)
    streams = {r[0]: r[1] for r in recs}
    assert streams["gather_bulk_kernel"] != streams["up_proj_tc_kernel"]
    # profiling off again: nothing is recorded
    _prefill(w, x)
    M.mla_profile_begin()
    assert M.mla_profile_end() == []


# ------------------------------------------------- pipeline overlap --
def test_serial_and_overlapped_pipeline_are_identical():
    """With the pipeline's overlap switched off every kernel of a prefill
    runs on the caller's stream, in the same order; the numbers are the
    same, bit for bit, and the setting comes back."""
    w = _small_batch(seed=95, heads=8)
    x = W.make_inputs(w)
    a_out, a_lse, sa = _prefill(w, x)
    prev = M.mla_set_pipeline_overlap(False)
    try:
        M.mla_profile_begin()
        b_out, b_lse, sb = _prefill(w, x)
        recs = M.mla_profile_end()
    finally:
        assert M.mla_set_pipeline_overlap(prev) is False
    assert prev is True
    assert sa == 0 and sb == 0
    assert torch.equal(a_out, b_out) and torch.equal(a_lse, b_lse)
    assert len(recs) > 3 and len({r[1] for r in recs}) == 1
    M.mla_profile_begin()
    _prefill(w, x)
    recs = M.mla_profile_end()
    assert len({r[1] for r in recs}) == 3  # caller's, gathers, up-projections
