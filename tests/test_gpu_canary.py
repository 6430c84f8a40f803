"""Canary regions around every buffer the library writes: each output is a
view into a larger allocation whose guard regions before and after hold a
sentinel, and the calls must leave the guards exactly as they were (a write
past either end of an output, a workspace or a status word would change
them).  Outputs start as NaN, so a row the call should have written and did
not is caught as well.  Expected values come from oracle/."""

import math

import numpy as np
import pytest
import torch

import mla_chunked_context_gb300 as M
from mla_chunked_context_gb300 import workloads as W
from oracle import mla as O

pytestmark = [pytest.mark.gpu,
              pytest.mark.filterwarnings("ignore::RuntimeWarning")]

DEV = "cuda:0"
SENTINEL = -1232.0    # exact in float32, bfloat16 and float16
GUARD = 64            # elements on either side (128-256 B: views stay 16-byte aligned)


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


def guarded(shape, dtype, fill=float("nan")):
    n = math.prod(shape)
    buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=dtype, device=DEV)
    view = buf[GUARD:GUARD + n].view(*shape)
    view.fill_(fill)
    return buf, view


def guarded_bytes(nbytes):
    buf = torch.full((nbytes + 2 * 4096,), 0xA5, dtype=torch.uint8, device=DEV)
    return buf, buf[4096:4096 + nbytes]


def intact(buf):
    if buf.dtype == torch.uint8:
        g = 4096
        return bool((buf[:g] == 0xA5).all() and (buf[-g:] == 0xA5).all())
    return bool((buf[:GUARD] == SENTINEL).all() and (buf[-GUARD:] == SENTINEL).all())


def f64(t):
    return t.detach().to("cpu").double().numpy()


def assert_close(got, ref, atol, rtol=0.0, what=""):
    both_inf = np.isneginf(got) & np.isneginf(ref)
    bad = ~both_inf & ~(np.abs(got - ref) <= atol + rtol * np.abs(ref))
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} off"


def _oracle_prefill(w, x):
    n = {k: (f64(v) if v.is_floating_point() else v.numpy()) for k, v in x.items()}
    d = O.MlaDims(w.num_heads, w.kv_lora_rank, w.qk_rope_dim, w.qk_nope_dim, w.v_dim,
                  w.block_size, w.softmax_scale)
    ro, rl, _ = O.chunked_prefill(n["q"], n["new_latent"], n["kv_cache"], n["block_table"],
                                  n["w_kv_b"], w.context_lens, w.query_lens, d, w.row_budget,
                                  w.max_context_chunk, w.split_alignment)
    return ro, rl


@pytest.mark.parametrize("case", ["deepseek", "split", "tiny"])
def test_prefill_writes_only_its_outputs(case):
    """mla_chunked_prefill: output, output LSE, workspace and status word all
    guarded.  deepseek: the tensor-core path (a continued request, one
    without context); split: few queries over a long context, so the
    context attention splits its units over their keys into the workspace's
    scratch slots; tiny: the float32 CUDA-core path."""
    if case == "tiny":
        w = W.workload("tiny")
    elif case == "split":
        w = W.scaled(W.workload("uniform"), context_lens=[9000, 0], query_lens=[70, 5],
                     num_heads=4, row_budget=4096, max_context_chunk=4096, seed=61)
    else:
        w = W.scaled(W.workload("uniform"), context_lens=[0, 300, 700], query_lens=[4, 130, 9],
                     num_heads=8, row_budget=512, max_context_chunk=512, seed=60)
    x = W.make_inputs(w)
    g = {k: v.to(DEV) for k, v in x.items()}
    T, H = w.num_tokens, w.num_heads
    d = M.Dims.of(w)
    args = (w.context_lens, w.query_lens, w.row_budget, w.max_context_chunk, w.split_alignment)
    ob, out = guarded((T, H, w.v_dim), w.torch_dtype)
    lb, lse = guarded((H, T), torch.float32)
    sb, status = guarded((1,), torch.int32, fill=0)
    wb, ws = guarded_bytes(M.mla_prefill_workspace_bytes(d, *args))
    M.mla_chunked_prefill(d, *args, g["q"], g["new_latent"], g["kv_cache"], g["block_table"],
                          g["w_kv_b"], ws, out, lse, status)
    torch.cuda.synchronize()
    assert intact(ob) and intact(lb) and intact(sb) and intact(wb)
    assert status.item() == 0
    ro, rl = _oracle_prefill(w, x)
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("heads", [4, 64])
def test_varlen_attention_writes_only_its_outputs(causal, heads):
    """mla_varlen_attn (4 heads: a CTA per unit; 64 heads and short
    sequences: the looping kernel) with O and LSE guarded; ragged sequences
    end inside a query tile."""
    w = W.scaled(W.workload("uniform"), num_heads=heads, seed=62)
    ql = [130, 77, 3, 200]
    kl = ql if causal else [300, 129, 40, 700]
    q_loc = [0] + list(np.cumsum(ql))
    k_loc = [0] + list(np.cumsum(kl))
    T, R = q_loc[-1], k_loc[-1]
    torch.manual_seed(62)
    q = torch.randn(T, heads, 192).to(torch.bfloat16)
    kv = (0.45 * torch.randn(heads, R, 256)).to(torch.float16)
    lat = torch.randn(R, 576).to(torch.bfloat16)
    ob, o = guarded((T, heads, 128), torch.float32)
    lb, lse = guarded((heads, T), torch.float32)
    M.mla_varlen_attn(M.Dims.of(w), causal, q_loc, k_loc, q.to(DEV), kv.to(DEV), lat.to(DEV),
                      o, lse)
    torch.cuda.synchronize()
    assert intact(ob) and intact(lb)
    kvr = f64(kv).transpose(1, 0, 2)
    for i in range(len(ql)):
        a, b, c, e = q_loc[i], q_loc[i + 1], k_loc[i], k_loc[i + 1]
        vis = np.tril(np.ones((b - a, e - c), dtype=bool)) if causal else None
        ro, rl = O.attention_with_lse(f64(q[a:b]), kvr[c:e, :, :128], f64(lat[c:e, 512:]),
                                      kvr[c:e, :, 128:], w.softmax_scale, visible=vis)
        assert_close(f64(o[a:b]), ro, 2e-2, 2e-2, what=f"O seq {i}")
        assert_close(f64(lse[:, a:b]), rl, 1e-3, what=f"LSE seq {i}")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_merge_writes_only_its_outputs(out_dtype):
    T, H, D = 333, 8, 128
    torch.manual_seed(63)
    po = torch.randn(T, H, D, device=DEV)
    so = torch.randn(T, H, D, device=DEV)
    pl = torch.randn(H, T, device=DEV)
    sl = torch.randn(H, T, device=DEV)
    pl[:, ::7] = float("-inf")
    ob, out = guarded((T, H, D), out_dtype)
    lb, lse = guarded((H, T), torch.float32)
    M.merge_attn_states(out, lse, po, pl, so, sl, 300)
    torch.cuda.synchronize()
    assert intact(ob) and intact(lb)
    ref_o, ref_l = O.merge_attn_states(f64(po), f64(pl), f64(so), f64(sl), 300)
    tol = 1e-5 if out_dtype == torch.float32 else 2 ** -8
    assert_close(f64(out), ref_o, tol, tol, what="O")
    assert_close(f64(lse), ref_l, 1e-5, what="LSE")


@pytest.mark.parametrize("rows", [300, 8192 + 77])
def test_up_projection_writes_only_its_output(rows):
    """mla_kv_up_proj with a ragged last row tile: the fp16 K/V output and
    the status word guarded."""
    w = W.scaled(W.workload("uniform"), num_heads=8, seed=64)
    torch.manual_seed(64)
    lat = torch.randn(rows, 576, device=DEV).to(torch.bfloat16)
    wkv = (torch.randn(8 * 256, 512, device=DEV) * 0.02).to(torch.bfloat16)
    kb, kv = guarded((8, rows, 256), torch.float16)
    sb, st = guarded((1,), torch.int32, fill=0)
    M.mla_kv_up_proj(M.Dims.of(w), lat, rows, wkv, kv, dev_status=st)
    torch.cuda.synchronize()
    assert intact(kb) and intact(sb) and st.item() == 0
    ref = np.einsum("rk,hck->hrc", f64(lat[:, :512]), f64(wkv).reshape(8, 256, 512))
    assert_close(f64(kv), ref, 2e-2, 2e-3, what="K/V")


def test_gather_writes_only_its_workspace():
    w = W.scaled(W.workload("uniform"), context_lens=[1, 37, 70, 129, 300],
                 query_lens=[1] * 5, num_heads=2, seed=65)
    x = W.make_inputs(w)
    g = {k: v.to(DEV) for k, v in x.items()}
    rows = sum(w.context_lens)
    req = torch.arange(5, dtype=torch.int32, device=DEV)
    st = torch.zeros(5, dtype=torch.int32, device=DEV)
    cu = torch.tensor([0] + list(np.cumsum(w.context_lens)), dtype=torch.int32, device=DEV)
    wb, ws = guarded((rows, w.latent_dim), w.torch_dtype)
    sb, status = guarded((1,), torch.int32, fill=0)
    M.mla_gather_context_rows(M.Dims.of(w), g["kv_cache"], g["block_table"], req, st, cu, rows,
                              ws, status)
    torch.cuda.synchronize()
    assert intact(wb) and intact(sb) and status.item() == 0
    assert not torch.isnan(ws).any()
