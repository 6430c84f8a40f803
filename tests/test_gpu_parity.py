"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Tolerances (written here, applied elementwise):
  * merge, float32 in/out:   |gpu - oracle| <= 1e-5 (O and LSE)
  * merge, bf16 in/out:      within one bf16 rounding of the float64 result
                             (|d| <= 2^-8 |ref| + 1e-6)
  * attention / prefill:     O: |d| <= 2e-2 + 2e-2 |ref|;  LSE: |d| <= 1e-3
  * gather, planner:         bit-exact
  * up-projection (bf16 out): |d| <= 2e-3 + 8e-3 |ref|
Inputs come from mla_chunked_context_gb300.workloads (seeded, host-drawn);
expected values come only from oracle/.
"""

import math

import numpy as np
import pytest
import torch

import mla_chunked_context_gb300 as M
from mla_chunked_context_gb300 import workloads as W
from oracle import mla as O
from oracle import planner as P

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


def assert_close(got, ref, atol, rtol=0.0, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    both_ninf = np.isneginf(got) & np.isneginf(ref)
    d = np.where(both_ninf, 0.0, np.abs(got - ref))
    lim = atol + rtol * np.abs(np.where(np.isfinite(ref), ref, 0.0))
    bad = ~(d <= lim)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; "
                             f"first {idx.tolist()} got {got[tuple(idx.T)]} ref {ref[tuple(idx.T)]}")


def dims_of(w):
    return M.Dims.of(w)


def to_dev(x):
    return {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in x.items()}


def np_inputs(x):
    return {k: (f64(v) if v.is_floating_point() else v.numpy()) for k, v in x.items()
            if torch.is_tensor(v)}


def odims(w):
    return O.MlaDims(w.num_heads, w.kv_lora_rank, w.qk_rope_dim, w.qk_nope_dim, w.v_dim,
                     w.block_size, w.softmax_scale)


# ------------------------------------------------------ failure detection --
def test_bounded_wait_gives_up_and_context_survives():
    """A wait that nothing satisfies runs out after its limit, sets the error
    bit and returns; the device keeps working afterwards."""
    if not M.mla_has_tcgen05():
        pytest.skip("the bounded waits live in the sm_103a kernels")
    assert M.mla_device_error_flags() == 0
    gave_up = torch.zeros(1, dtype=torch.int32, device=DEV)
    M.mla_selftest_bounded_wait(2000, gave_up)            # 2 ms limit
    torch.cuda.synchronize()
    assert gave_up.item() == 1
    assert M.mla_device_error_flags() == 1               # MLA_DEVICE_ERR_WAIT_TIMEOUT
    assert M.mla_device_error_flags() == 0               # read-and-clear
    m, x = _merge_case(64, 2, 8, 32, "f32", 35)          # the context still works
    out, lse = _run_merge(x, torch.float32)
    assert not torch.isnan(out).any()


# ------------------------------------------------------------------ merge --
def _merge_case(T, H, D, pnt, dtype, seed):
    m = W.MergeWorkload(num_tokens=T, num_heads=H, head_dim=D, prefix_num_tokens=pnt,
                        dtype=dtype, seed=seed, both_empty=4)
    return m, W.make_merge_inputs(m, poison=True)


def _run_merge(x, out_dtype, with_lse=True):
    g = {k: v.to(DEV) for k, v in x.items() if torch.is_tensor(v)}
    T, H, D = g["suffix_o"].shape
    out = torch.full((T, H, D), float("nan"), dtype=out_dtype, device=DEV)
    out_lse = torch.full((H, T), float("nan"), device=DEV) if with_lse else None
    M.merge_attn_states(out, out_lse, g["prefix_o"], g["prefix_lse"], g["suffix_o"],
                        g["suffix_lse"], x["prefix_num_tokens"])
    torch.cuda.synchronize()
    return out, out_lse


def test_merge_fp32_tight():
    m, x = _merge_case(300, 4, 16, 200, "f32", 31)
    out, lse = _run_merge(x, torch.float32)
    ro, rl = O.merge_attn_states(f64(x["prefix_o"]), f64(x["prefix_lse"]), f64(x["suffix_o"]),
                                 f64(x["suffix_lse"]), m.prefix_num_tokens)
    assert not torch.isnan(out).any()
    assert_close(f64(out), ro, 1e-5, what="O")
    assert_close(f64(lse), rl, 1e-5, what="LSE")
    for t, h in x["both_empty"]:
        assert (out[t, h] == 0).all() and math.isinf(lse[h, t].item())


def test_merge_bf16_one_rounding():
    m, x = _merge_case(1024, 16, 128, 768, "bf16", 32)
    out, lse = _run_merge(x, torch.bfloat16)
    ro, rl = O.merge_attn_states(f64(x["prefix_o"]), f64(x["prefix_lse"]), f64(x["suffix_o"]),
                                 f64(x["suffix_lse"]), m.prefix_num_tokens)
    assert_close(f64(out), ro, 1e-6, 2.0 ** -8, what="O")
    assert_close(f64(lse), rl, 1e-5, what="LSE")
    # tokens at or past prefix_num_tokens: the suffix, bit for bit
    assert torch.equal(out[768:].cpu(), x["suffix_o"][768:])


@pytest.mark.slow
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_merge_full_size_every_row(dtype):
    """The full standalone merge (8192 tokens x 128 heads x 128, 15% empty
    prefix tokens, 4 both-empty rows, NaN prefix past prefix_num_tokens 6144)
    against the oracle on every one of its 1,048,576 (token, head) rows:
    bf16 within one rounding of the float64 result, float32 within 1e-5;
    rows at or past the threshold are the suffix bit for bit."""
    m = W.MergeWorkload(dtype=dtype)
    x = W.make_merge_inputs(m, poison=True)
    out_dtype = torch.bfloat16 if dtype == "bf16" else torch.float32
    out, lse = _run_merge(x, out_dtype)
    pnt = m.prefix_num_tokens
    assert not torch.isnan(out).any().item() and not torch.isnan(lse).any().item()
    assert torch.equal(out[pnt:].cpu(), x["suffix_o"][pnt:])
    assert torch.equal(lse[:, pnt:].cpu(), x["suffix_lse"][:, pnt:])
    for t, h in x["both_empty"]:
        assert (out[t, h] == 0).all() and math.isinf(lse[h, t].item()) and lse[h, t] < 0
    # the rows below the threshold, compared in full (in slices of tokens to
    # bound the oracle's host memory)
    tol = (1e-6, 2.0 ** -8) if dtype == "bf16" else (1e-5, 0.0)
    for a in range(0, pnt, 1024):
        b = min(pnt, a + 1024)
        ro, rl = O.merge_attn_states(f64(x["prefix_o"][a:b]), f64(x["prefix_lse"][:, a:b]),
                                     f64(x["suffix_o"][a:b]), f64(x["suffix_lse"][:, a:b]),
                                     b - a)
        assert_close(f64(out[a:b]), ro, *tol, what=f"O tokens {a}:{b}")
        assert_close(f64(lse[:, a:b]), rl, 1e-5, what=f"LSE tokens {a}:{b}")


def test_merge_in_place_on_suffix():
    m, x = _merge_case(257, 8, 64, 100, "f32", 33)
    g = {k: v.to(DEV) for k, v in x.items() if torch.is_tensor(v)}
    ro, _ = O.merge_attn_states(f64(x["prefix_o"]), f64(x["prefix_lse"]), f64(x["suffix_o"]),
                                f64(x["suffix_lse"]), 100)
    M.merge_attn_states(g["suffix_o"], None, g["prefix_o"], g["prefix_lse"], g["suffix_o"],
                        g["suffix_lse"], 100)
    torch.cuda.synchronize()
    assert_close(f64(g["suffix_o"]), ro, 1e-5, what="in-place O")


def test_merge_empty_batch_and_zero_prefix():
    z = torch.empty(0, 2, 8, device=DEV)
    zl = torch.empty(2, 0, device=DEV)
    M.merge_attn_states(z, zl, z, zl, z, zl, 0)
    m, x = _merge_case(64, 2, 8, 0, "f32", 34)
    out, lse = _run_merge(x, torch.float32)
    assert torch.equal(out.cpu(), x["suffix_o"]) and torch.equal(lse.cpu(), x["suffix_lse"])


# ---------------------------------------------------- empty-context rows --
def test_mask_empty_context_page_shape():
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "mask_empty_context.json")))
    H, T, D = g["num_heads"], g["num_tokens"], g["head_dim"]
    lo, hi = g["masked_rows"]
    gen = torch.Generator().manual_seed(3)
    lse = torch.randn(H, T, generator=gen)
    out = torch.randn(T, H, D, generator=gen)
    out[lo:hi] = float("nan")
    qsl = torch.tensor(P.query_start_loc(g["query_lens"]), dtype=torch.int32)
    csl = torch.tensor(P.query_start_loc(g["context_lens"]), dtype=torch.int32)
    rl, ro = O.mask_empty_context(lse.double().numpy(), out.double().numpy(), qsl.numpy(),
                                  csl.numpy())
    dl, do = lse.to(DEV), out.to(DEV)
    M.mla_mask_empty_context(dl, do, qsl.to(DEV), csl.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(f64(dl), rl) and np.array_equal(f64(do), ro)
    # the partial initialisation of the chunked scheme gives the same rows
    o2 = torch.full((T, H, D), float("nan"), device=DEV)
    l2 = torch.full((H, T), float("nan"), device=DEV)
    M.mla_fill_empty_rows(o2, l2, P.empty_token_slices(g["context_lens"], g["query_lens"]))
    torch.cuda.synchronize()
    assert (o2[lo:hi] == 0).all() and torch.isneginf(l2[:, lo:hi]).all()
    assert torch.isnan(o2[:lo]).all() and torch.isnan(l2[:, hi:]).all()


# ---------------------------------------------------------------- gather --
def _gather_case(w, plan):
    x = W.make_inputs(w)
    g = to_dev(x)
    n = plan.request_end - plan.request_start
    req = torch.arange(plan.request_start, plan.request_end, dtype=torch.int32, device=DEV)
    st = torch.tensor(plan.starts, dtype=torch.int32, device=DEV)
    cu = torch.tensor([0] + list(np.cumsum(plan.seq_lens)), dtype=torch.int32, device=DEV)
    rows = int(sum(plan.seq_lens))
    ws = torch.full((rows, w.latent_dim), float("nan"), dtype=w.torch_dtype, device=DEV)
    return x, g, req, st, cu, rows, ws, n


@pytest.mark.parametrize("name", ["tiny", "deepseek"])
def test_gather_bit_exact(name):
    if name == "tiny":
        w = W.workload("tiny")
    else:
        w = W.scaled(W.workload("uniform"), context_lens=[0, 300, 1000, 5, 700],
                     query_lens=[1, 1, 1, 1, 1], num_heads=2, seed=40)
    plans = P.plan_mla_context_chunks(w.context_lens, 512, 512, 16)
    for plan in plans:
        x, g, req, st, cu, rows, ws, n = _gather_case(w, plan)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        M.mla_gather_context_rows(M.Dims.of(w), g["kv_cache"], g["block_table"], req, st, cu,
                                  rows, ws, status)
        torch.cuda.synchronize()
        ref = O.gather_chunk(f64(x["kv_cache"]), x["block_table"].numpy(), plan, w.block_size)
        assert np.array_equal(f64(ws), ref)
        assert status.item() == 0


def test_gather_windows_runs_and_adjacent_blocks():
    """The bulk-copy gather cuts the workspace into 32-row windows and copies
    runs of rows that are consecutive in the cache: sequences of 1..70 rows
    starting mid-block, a request whose physical blocks follow one another
    in memory (runs that cross block boundaries), and a partial last window;
    bit-exact against the oracle's row-by-row gather."""
    w = W.scaled(W.workload("uniform"), context_lens=[1, 37, 70, 129, 5, 300, 2, 64],
                 query_lens=[1] * 8, num_heads=2, seed=39)
    x = W.make_inputs(w)
    # request 5 (300 rows, 5 blocks) moved to 5 new physical blocks that
    # follow one another in memory, holding the same rows
    bt = x["block_table"].clone()
    nblk = x["kv_cache"].shape[0]
    x["kv_cache"] = torch.cat([x["kv_cache"], x["kv_cache"][bt[5, :5].long()]], 0)
    bt[5, :5] = torch.arange(nblk, nblk + 5, dtype=torch.int32)
    x["block_table"] = bt
    g = to_dev(x)
    starts = [0, 3, 60, 0, 1, 17, 1, 0]                  # mid-block starts
    lens = [1, 34, 10, 129, 4, 283, 1, 64]
    assert all(s + n <= c for s, n, c in zip(starts, lens, w.context_lens))
    from oracle.planner import ChunkPlan
    plan = ChunkPlan(0, 8, starts, lens)
    req = torch.arange(8, dtype=torch.int32, device=DEV)
    st = torch.tensor(starts, dtype=torch.int32, device=DEV)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=DEV)
    rows = int(sum(lens))
    assert rows % 32 != 0
    ws = torch.full((rows, w.latent_dim), float("nan"), dtype=w.torch_dtype, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    M.mla_gather_context_rows(M.Dims.of(w), g["kv_cache"], g["block_table"], req, st, cu, rows,
                              ws, status)
    torch.cuda.synchronize()
    ref = O.gather_chunk(f64(x["kv_cache"]), bt.numpy(), plan, w.block_size)
    assert not np.isnan(ref).any()          # only rows inside the contexts
    assert np.array_equal(f64(ws), ref)
    assert status.item() == 0


def test_gather_bad_block_sets_status():
    w = W.workload("tiny")
    plan = P.plan_mla_context_chunks(w.context_lens, 128, 128, 16)[0]
    x, g, req, st, cu, rows, ws, n = _gather_case(w, plan)
    bt = g["block_table"].clone()
    bt[1, 2] = 10 ** 6                      # request 1, rows 32..47
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    M.mla_gather_context_rows(M.Dims.of(w), g["kv_cache"], bt, req, st, cu, rows, ws, status)
    torch.cuda.synchronize()
    assert status.item() == M.MLA_STATUS_BAD_BLOCK
    assert (ws[32:48] == 0).all()
    ref = O.gather_chunk(f64(x["kv_cache"]), x["block_table"].numpy(), plan, w.block_size)
    assert np.array_equal(f64(ws[:32]), ref[:32]) and np.array_equal(f64(ws[48:]), ref[48:])


# ----------------------------------------------------------- up-projection --
# one rounding of the f32 accumulation to the output type, plus f32 ordering
UP_TOL = {torch.bfloat16: (2e-3, 8e-3), torch.float16: (1e-4, 1.5e-3),
          torch.float32: (1e-4, 1e-4)}


@pytest.mark.parametrize("kv_dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("rows,heads", [(300, 8), (128, 2), (1, 2), (4099, 16)])
def test_up_proj_deepseek(rows, heads, kv_dtype):
    w = W.scaled(W.workload("uniform"), num_heads=heads, seed=41)
    gen = torch.Generator().manual_seed(rows)
    lat = torch.randn(rows, w.latent_dim, generator=gen).to(torch.bfloat16)
    wkv = (torch.randn(heads * 256, 512, generator=gen) * 0.02).to(torch.bfloat16)
    kv = torch.full((rows, heads * 256), float("nan"), dtype=kv_dtype, device=DEV)
    M.mla_kv_up_proj(M.Dims.of(w), lat.to(DEV), rows, wkv.to(DEV), kv)
    torch.cuda.synchronize()
    kn, v = O.up_project(f64(lat), f64(wkv), odims(w))
    ref = np.concatenate([kn, v], axis=2).transpose(1, 0, 2)   # head-major [H, rows, 256]
    assert_close(f64(kv).reshape(heads, rows, 256), ref, *UP_TOL[kv_dtype], what="kv")


def test_up_proj_deepseek_float32_out_is_refused():
    """The DeepSeek-shaped bf16 up-projection runs on the tcgen05 GEMM only,
    which writes 16-bit K/V: a float32 output is refused, not handed to the
    CUDA-core GEMM."""
    w = W.scaled(W.workload("uniform"), num_heads=2, seed=41)
    lat = torch.zeros(64, w.latent_dim, dtype=torch.bfloat16, device=DEV)
    wkv = torch.zeros(2 * 256, 512, dtype=torch.bfloat16, device=DEV)
    kv = torch.empty(64, 2 * 256, dtype=torch.float32, device=DEV)
    with pytest.raises(M.MlaError) as e:
        M.mla_kv_up_proj(M.Dims.of(w), lat, 64, wkv, kv)
    assert e.value.code == -5


def test_up_proj_fp32_tiny():
    w = W.workload("tiny")
    x = W.make_inputs(w)
    lat = x["new_latent"]
    kv = torch.empty(lat.shape[0], w.num_heads * 64, device=DEV)
    M.mla_kv_up_proj(M.Dims.of(w), lat.to(DEV), lat.shape[0], x["w_kv_b"].to(DEV), kv)
    torch.cuda.synchronize()
    kn, v = O.up_project(f64(lat), f64(x["w_kv_b"]), odims(w))
    ref = np.concatenate([kn, v], axis=2).transpose(1, 0, 2)
    assert_close(f64(kv).reshape(w.num_heads, lat.shape[0], 64), ref, 1e-5, 1e-5,
                 what="kv fp32")


# -------------------------------------------------------------- attention --
def _attn_inputs(w, n_rows, T, seed, kv_dtype=None):
    gen = torch.Generator().manual_seed(seed)
    H = w.num_heads
    q = torch.randn(T, H, w.qk_dim, generator=gen).to(w.torch_dtype)
    # head-major [H, rows, Dn+Dv], as mla_kv_up_proj writes it
    kv = (0.45 * torch.randn(H, n_rows, w.qk_nope_dim + w.v_dim, generator=gen)).to(
        kv_dtype or w.torch_dtype)
    lat = torch.randn(n_rows, w.latent_dim, generator=gen).to(w.torch_dtype)
    return q, kv, lat


def _oracle_attn(w, q, kv, lat, q_loc, k_loc, causal):
    H, Dn, Dv, L = w.num_heads, w.qk_nope_dim, w.v_dim, w.kv_lora_rank
    T = q.shape[0]
    kvr = f64(kv).transpose(1, 0, 2)            # [rows, H, Dn+Dv]
    o = np.full((T, H, Dv), np.nan)
    lse = np.full((H, T), np.nan)
    for i in range(len(q_loc) - 1):
        a, b, c, e = q_loc[i], q_loc[i + 1], k_loc[i], k_loc[i + 1]
        if a == b:
            continue
        vis = np.tril(np.ones((b - a, e - c), dtype=bool)) if causal else None
        o[a:b], lse[:, a:b] = O.attention_with_lse(
            f64(q[a:b]), kvr[c:e, :, :Dn], f64(lat[c:e, L:]), kvr[c:e, :, Dn:],
            w.softmax_scale, visible=vis)
    return o, lse


@pytest.mark.parametrize("kind", ["deepseek", "tiny"])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_attention(kind, causal):
    """deepseek: fp16 K/V (the tcgen05 kernel on GB300); tiny: float32
    storage (the CUDA-core kernel)."""
    kv_dtype = {"deepseek": torch.float16}.get(kind)
    if kind != "tiny":
        w = W.scaled(W.workload("uniform"), num_heads=4, seed=42)
        if causal:
            ql = [1, 130, 77, 256, 129]
            kl = ql
        else:
            ql = [1, 130, 77, 3, 200]
            kl = [5, 300, 129, 1000, 64]
    else:
        w = W.workload("tiny")
        ql = [3, 16, 5]
        kl = ql if causal else [64, 128, 37]
    q_loc = [0] + list(np.cumsum(ql))
    k_loc = [0] + list(np.cumsum(kl))
    q, kv, lat = _attn_inputs(w, k_loc[-1], q_loc[-1], 7, kv_dtype)
    o = torch.full((q_loc[-1], w.num_heads, w.v_dim), float("nan"), device=DEV)
    lse = torch.full((w.num_heads, q_loc[-1]), float("nan"), device=DEV)
    M.mla_varlen_attn(M.Dims.of(w), causal, q_loc, k_loc, q.to(DEV), kv.to(DEV), lat.to(DEV),
                      o, lse)
    torch.cuda.synchronize()
    ro, rl = _oracle_attn(w, q, kv, lat, q_loc, k_loc, causal)
    assert_close(f64(o), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_attention_multi_tile(causal):
    """Sequences of 3, 5 and 2 query tiles, several tiles of a sequence and
    head side by side (sharing K/V through L2); causal tiles see a growing
    number of key tiles."""
    w = W.scaled(W.workload("uniform"), num_heads=2, seed=45)
    ql = [300, 520, 129]
    kl = ql if causal else [700, 1030, 64]
    q_loc = [0] + list(np.cumsum(ql))
    k_loc = [0] + list(np.cumsum(kl))
    q, kv, lat = _attn_inputs(w, k_loc[-1], q_loc[-1], 9, torch.float16)
    o = torch.full((q_loc[-1], w.num_heads, w.v_dim), float("nan"), device=DEV)
    lse = torch.full((w.num_heads, q_loc[-1]), float("nan"), device=DEV)
    M.mla_varlen_attn(M.Dims.of(w), causal, q_loc, k_loc, q.to(DEV), kv.to(DEV), lat.to(DEV),
                      o, lse)
    torch.cuda.synchronize()
    ro, rl = _oracle_attn(w, q, kv, lat, q_loc, k_loc, causal)
    assert_close(f64(o), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_attention_many_units_several_tiles(causal):
    """Several (query tile, head) units per SM with several key tiles each
    (the one-CTA kernel, a CTA per unit, many waves): a sequence without
    keys in between (O=0, LSE=-inf), odd and ragged tile counts; non-causal
    also a second, accumulating pass over the same keys (LSE + ln 2)."""
    w = W.scaled(W.workload("uniform"), num_heads=64 if not causal else 16, seed=48)
    ql = [300, 520, 129, 200] if not causal else [2000, 900]
    kl = [700, 1030, 0, 2000] if not causal else ql
    q_loc = [0] + list(np.cumsum(ql))
    k_loc = [0] + list(np.cumsum(kl))
    q, kv, lat = _attn_inputs(w, k_loc[-1], q_loc[-1], 12, torch.float16)
    o = torch.full((q_loc[-1], w.num_heads, w.v_dim), float("nan"), device=DEV)
    lse = torch.full((w.num_heads, q_loc[-1]), float("nan"), device=DEV)
    d = M.Dims.of(w)
    gq, gkv, glat = q.to(DEV), kv.to(DEV), lat.to(DEV)
    M.mla_profile_begin()
    M.mla_varlen_attn(d, causal, q_loc, k_loc, gq, gkv, glat, o, lse)
    names = [r[0] for r in M.mla_profile_end()]
    torch.cuda.synchronize()
    assert "attn_tc_kernel" in names
    ro, rl = _oracle_attn(w, q, kv, lat, q_loc, k_loc, causal)
    assert_close(f64(o), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")
    if not causal:
        acc = [1] * len(ql)
        M.mla_varlen_attn(d, False, q_loc, k_loc, gq, gkv, glat, o, lse, accumulate=acc)
        torch.cuda.synchronize()
        rl2 = np.where(np.isfinite(rl), rl + np.log(2.0), rl)
        assert_close(f64(o), ro, 2e-2, 2e-2, what="O accumulated")
        assert_close(f64(lse), rl2, 1e-3, what="LSE accumulated")


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_attention_many_short_units(causal):
    """Many more (query tile, head) units than SMs, each of one or two key
    tiles; context sequences without keys between them write O=0,
    LSE=-inf; a second pass over the same keys accumulates (LSE + ln 2)."""
    w = W.scaled(W.workload("uniform"), num_heads=64, seed=46)
    ql = [130, 1, 200, 77, 256, 3, 129, 40]
    kl = ql if causal else [100, 0, 250, 129, 0, 5, 256, 1]
    q_loc = [0] + list(np.cumsum(ql))
    k_loc = [0] + list(np.cumsum(kl))
    q, kv, lat = _attn_inputs(w, k_loc[-1], q_loc[-1], 10, torch.float16)
    o = torch.full((q_loc[-1], w.num_heads, w.v_dim), float("nan"), device=DEV)
    lse = torch.full((w.num_heads, q_loc[-1]), float("nan"), device=DEV)
    d = M.Dims.of(w)
    gq, gkv, glat = q.to(DEV), kv.to(DEV), lat.to(DEV)
    M.mla_varlen_attn(d, causal, q_loc, k_loc, gq, gkv, glat, o, lse)
    torch.cuda.synchronize()
    ro, rl = _oracle_attn(w, q, kv, lat, q_loc, k_loc, causal)  # keyless: O=0, LSE=-inf
    assert_close(f64(o), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")
    if not causal:
        # the same keys again, accumulated: the result is attention over the
        # keys twice (LSE + ln 2, same O), keyless rows unchanged
        acc = [1] * len(ql)
        M.mla_varlen_attn(d, False, q_loc, k_loc, gq, gkv, glat, o, lse, accumulate=acc)
        torch.cuda.synchronize()
        rl2 = np.where(np.isfinite(rl), rl + np.log(2.0), rl)
        assert_close(f64(o), ro, 2e-2, 2e-2, what="O accumulated")
        assert_close(f64(lse), rl2, 1e-3, what="LSE accumulated")


@pytest.mark.parametrize("heads,ql,kl", [(4, [130, 5], [1000, 300]),
                                         (64, [130, 1, 77, 40, 9, 128], [500, 3, 129, 256, 64, 400])])
def test_varlen_attention_running_max_rescales(heads, ql, kl):
    """Keys whose K_nope grows every 64 keys, so the running max of a row
    rises by more than 2^8 again and again, inside a tile and from tile to
    tile: O is rescaled (after the previous P.V) and, in the looping kernel,
    the first half of a tile's P is rescaled when the second half raises the
    max.  4 heads: one CTA per unit; 64 heads and short sequences: the
    looping kernel."""
    w = W.scaled(W.workload("uniform"), num_heads=heads, seed=47)
    q_loc = [0] + list(np.cumsum(ql))
    k_loc = [0] + list(np.cumsum(kl))
    q, kv, lat = _attn_inputs(w, k_loc[-1], q_loc[-1], 11, torch.float16)
    grow = torch.ones(k_loc[-1])
    for i in range(len(kl)):
        j = torch.arange(kl[i], dtype=torch.float32)
        grow[k_loc[i]:k_loc[i + 1]] = 1.0 + 1.5 * (j // 64)
    kv = kv.float()
    kv[:, :, :128] *= grow[None, :, None]
    kv = kv.to(torch.float16)
    o = torch.full((q_loc[-1], heads, w.v_dim), float("nan"), device=DEV)
    lse = torch.full((heads, q_loc[-1]), float("nan"), device=DEV)
    M.mla_varlen_attn(M.Dims.of(w), False, q_loc, k_loc, q.to(DEV), kv.to(DEV), lat.to(DEV), o,
                      lse)
    torch.cuda.synchronize()
    ro, rl = _oracle_attn(w, q, kv, lat, q_loc, k_loc, False)
    # the scores really do grow by more than 2^8 (base 2) between the first
    # and the last 64 keys of the longest sequence
    kvr = f64(kv).transpose(1, 0, 2)
    qn = f64(q[:ql[0]])
    s = np.einsum("mhd,nhd->hmn", qn[:, :, :128], kvr[:kl[0], :, :128]) * w.softmax_scale
    assert (s[:, :, -64:].max(axis=2) - s[:, :, :64].max(axis=2)).mean() / math.log(2) > 8
    assert_close(f64(o), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


def test_varlen_attention_accumulate():
    """Chunk 2 continues the requests of chunk 1 and merges into its partial;
    the result equals attention over both key ranges at once."""
    w = W.scaled(W.workload("uniform"), num_heads=2, seed=43)
    ql = [7, 140]
    k1, k2 = [100, 260], [60, 131]
    q_loc = [0] + list(np.cumsum(ql))
    q, kv, lat = _attn_inputs(w, sum(k1) + sum(k2), q_loc[-1], 8, torch.float16)
    # key rows: chunk-1 rows of both requests, then chunk-2 rows of both
    loc1 = [0, k1[0], k1[0] + k1[1]]
    loc2 = [loc1[-1], loc1[-1] + k2[0], loc1[-1] + k2[0] + k2[1]]
    o = torch.full((q_loc[-1], 2, 128), float("nan"), device=DEV)
    lse = torch.full((2, q_loc[-1]), float("nan"), device=DEV)
    d = M.Dims.of(w)
    gq, gkv, glat = q.to(DEV), kv.to(DEV), lat.to(DEV)
    M.mla_varlen_attn(d, False, q_loc, loc1, gq, gkv, glat, o, lse, kv_rows=551)
    M.mla_varlen_attn(d, False, q_loc, loc2, gq, gkv, glat, o, lse, accumulate=[1, 1],
                      kv_rows=551)
    torch.cuda.synchronize()
    idx = [np.r_[0:100, 360:420], np.r_[100:360, 420:551]]
    kvr = f64(kv).transpose(1, 0, 2)
    for i in range(2):
        a, b = q_loc[i], q_loc[i + 1]
        ro, rl = O.attention_with_lse(f64(q[a:b]), kvr[idx[i], :, :128], f64(lat[idx[i], 512:]),
                                      kvr[idx[i], :, 128:], w.softmax_scale)
        assert_close(f64(o[a:b]), ro, 2e-2, 2e-2, what="O")
        assert_close(f64(lse[:, a:b]), rl, 1e-3, what="LSE")


# ------------------------------------------- fused up-projection (f2) --
def _fused_inputs(w, n_rows, T, seed):
    gen = torch.Generator().manual_seed(seed)
    H = w.num_heads
    q = torch.randn(T, H, w.qk_dim, generator=gen).to(w.torch_dtype)
    lat = torch.randn(n_rows, w.latent_dim, generator=gen).to(w.torch_dtype)
    wkv = (0.02 * torch.randn(H * (w.qk_nope_dim + w.v_dim), w.kv_lora_rank,
                              generator=gen)).to(w.torch_dtype)
    return q, lat, wkv


def _oracle_fused(w, q, lat, wkv, q_loc, k_loc, key_rows=None):
    """(O, LSE) of each sequence over its latent rows, up-projected by the
    oracle; key_rows[i] overrides the rows of sequence i."""
    L = w.kv_lora_rank
    kn, v = O.up_project(f64(lat), f64(wkv), odims(w))
    T, H = q.shape[0], w.num_heads
    o = np.full((T, H, w.v_dim), np.nan)
    lse = np.full((H, T), np.nan)
    la = f64(lat)
    for i in range(len(q_loc) - 1):
        a, b = q_loc[i], q_loc[i + 1]
        rows = key_rows[i] if key_rows is not None else np.arange(k_loc[i], k_loc[i + 1])
        if a == b or len(rows) == 0:
            continue
        o[a:b], lse[:, a:b] = O.attention_with_lse(f64(q[a:b]), kn[rows], la[rows, L:], v[rows],
                                                   w.softmax_scale)
    return o, lse


def _fused_case(heads, ql, kl, seed):
    w = W.scaled(W.workload("uniform"), num_heads=heads, seed=seed)
    q_loc = [0] + [int(x) for x in np.cumsum(ql)]
    k_loc = [0] + [int(x) for x in np.cumsum(kl)]
    q, lat, wkv = _fused_inputs(w, k_loc[-1], q_loc[-1], seed)
    return w, q_loc, k_loc, q, lat, wkv


@pytest.mark.parametrize("heads", [16, 128])
def test_fused_context_attention(heads):
    """Up-projection fused into the attention: ragged sequences of 1-128
    queries and 1-8 key tiles (tails of 5, 44, 1 and 104 keys); a sequence
    without queries and one without keys leave their rows untouched.  The
    (head, sequence, key tile) space is cut into one range per cluster, so
    some (head, sequence) units are split between clusters and merged."""
    ql = [1, 128, 77, 5, 0, 100]
    kl = [5, 300, 129, 1000, 64, 0]
    w, q_loc, k_loc, q, lat, wkv = _fused_case(heads, ql, kl, 50)
    T = q_loc[-1]
    o = torch.full((T, heads, w.v_dim), 7.0, device=DEV)
    lse = torch.full((heads, T), 3.0, device=DEV)
    M.mla_fused_context_attn(M.Dims.of(w), q_loc, k_loc, q.to(DEV), lat.to(DEV), wkv.to(DEV),
                             o, lse)
    torch.cuda.synchronize()
    ro, rl = _oracle_fused(w, q, lat, wkv, q_loc, k_loc)
    keyless = slice(q_loc[5], q_loc[6])
    ro[keyless], rl[:, keyless] = 7.0, 3.0   # untouched
    assert_close(f64(o), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


def test_fused_context_attention_split_and_accumulate():
    """One long sequence over 16 heads, its 40 key tiles cut over many
    clusters per head (up to 16 scratch slots), in two chunks: the second
    accumulates into the first's partial; the result is attention over
    both chunks' keys."""
    heads, nq = 16, 99
    k1, k2 = 2500, 2620
    w, _, _, q, lat, wkv = _fused_case(heads, [nq], [k1 + k2], 51)
    o = torch.full((nq, heads, w.v_dim), float("nan"), device=DEV)
    lse = torch.full((heads, nq), float("nan"), device=DEV)
    d = M.Dims.of(w)
    gq, glat, gw = q.to(DEV), lat.to(DEV), wkv.to(DEV)
    M.mla_fused_context_attn(d, [0, nq], [0, k1], gq, glat, gw, o, lse)
    torch.cuda.synchronize()
    ro1, rl1 = _oracle_fused(w, q, lat, wkv, [0, nq], [0, k1])
    assert_close(f64(o), ro1, 2e-2, 2e-2, what="O chunk 1")
    assert_close(f64(lse), rl1, 1e-3, what="LSE chunk 1")
    M.mla_fused_context_attn(d, [0, nq], [k1, k1 + k2], gq, glat, gw, o, lse, accumulate=[1])
    torch.cuda.synchronize()
    ro, rl = _oracle_fused(w, q, lat, wkv, [0, nq], [0, k1 + k2])
    assert_close(f64(o), ro, 2e-2, 2e-2, what="O accumulated")
    assert_close(f64(lse), rl, 1e-3, what="LSE accumulated")


@pytest.mark.parametrize("heads,seed", [(16, 52), (4, 53)])
def test_fused_context_attention_many_sequences(heads, seed):
    """40 sequences of 1-128 queries and 130-420 keys.  16 heads (seed 52):
    six sequences are cut between clusters and merged from scratch slots;
    4 heads (seed 53): more cut units than scratch slots, so the cluster
    ranges end on unit boundaries instead."""
    rng = np.random.default_rng(seed)
    ql = [int(x) for x in rng.integers(1, 129, 40)]
    kl = [int(x) for x in rng.integers(130, 421, 40)]
    w, q_loc, k_loc, q, lat, wkv = _fused_case(heads, ql, kl, seed)
    T = q_loc[-1]
    o = torch.full((T, heads, w.v_dim), float("nan"), device=DEV)
    lse = torch.full((heads, T), float("nan"), device=DEV)
    M.mla_fused_context_attn(M.Dims.of(w), q_loc, k_loc, q.to(DEV), lat.to(DEV), wkv.to(DEV),
                             o, lse)
    torch.cuda.synchronize()
    ro, rl = _oracle_fused(w, q, lat, wkv, q_loc, k_loc)
    assert_close(f64(o), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


@pytest.mark.parametrize("heads,ql,kl", [(1, [1, 128], [1, 128]), (7, [57], [3000]),
                                         (3, [57], [3000])])
def test_fused_context_attention_edge_heads(heads, ql, kl):
    """One head with a one-key and a one-full-tile sequence (two clusters,
    one tile each); 7 heads of one 24-tile sequence cut into up to 12 pieces
    each, cluster ranges crossing head boundaries; 3 heads of it: more
    pieces than scratch slots, so one cluster per head and most idle."""
    w, q_loc, k_loc, q, lat, wkv = _fused_case(heads, ql, kl, 54)
    T = q_loc[-1]
    o = torch.full((T, heads, w.v_dim), float("nan"), device=DEV)
    lse = torch.full((heads, T), float("nan"), device=DEV)
    M.mla_fused_context_attn(M.Dims.of(w), q_loc, k_loc, q.to(DEV), lat.to(DEV), wkv.to(DEV),
                             o, lse)
    torch.cuda.synchronize()
    ro, rl = _oracle_fused(w, q, lat, wkv, q_loc, k_loc)
    assert_close(f64(o), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


def test_fused_context_attention_rejects_two_query_tiles():
    w, q_loc, k_loc, q, lat, wkv = _fused_case(16, [129], [300], 53)
    o = torch.zeros(129, 16, 128, device=DEV)
    lse = torch.zeros(16, 129, device=DEV)
    with pytest.raises(M.MlaError) as e:
        M.mla_fused_context_attn(M.Dims.of(w), q_loc, k_loc, q.to(DEV), lat.to(DEV),
                                 wkv.to(DEV), o, lse)
    assert e.value.code == -5


# ---------------------------------------------------------- whole prefill --
def _run_prefill(w, x):
    g = to_dev(x)
    T = w.num_tokens
    out = torch.full((T, w.num_heads, w.v_dim), float("nan"), dtype=w.torch_dtype, device=DEV)
    out_lse = torch.full((w.num_heads, T), float("nan"), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pf = M.ChunkedPrefill(M.Dims.of(w), w.context_lens, w.query_lens, w.row_budget,
                          w.max_context_chunk, w.split_alignment, device=DEV)
    pf(g["q"], g["new_latent"], g["kv_cache"], g["block_table"], g["w_kv_b"], out, out_lse,
       status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return out, out_lse


def _oracle_prefill(w, x):
    n = np_inputs(x)
    return O.chunked_prefill(n["q"], n["new_latent"], n["kv_cache"], n["block_table"],
                             n["w_kv_b"], w.context_lens, w.query_lens, odims(w), w.row_budget,
                             w.max_context_chunk, w.split_alignment)


def test_prefill_tiny_workload():
    w = W.workload("tiny")
    x = W.make_inputs(w)
    out, lse = _run_prefill(w, x)
    ro, rl, _ = _oracle_prefill(w, x)
    assert not torch.isnan(out).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")
    # float32 storage: far inside the contract
    assert_close(f64(out), ro, 1e-4, 1e-4, what="O fp32")


@pytest.mark.parametrize("budget", [512, 2048])
def test_prefill_deepseek_shapes_multichunk(budget):
    w = W.scaled(W.workload("uniform"), context_lens=[0, 300, 1000, 5, 0, 700, 64],
                 query_lens=[3, 130, 1, 40, 7, 200, 0], num_heads=8, row_budget=budget,
                 max_context_chunk=budget, split_alignment=64, seed=44)
    x = W.make_inputs(w)
    out, lse = _run_prefill(w, x)
    ro, rl, plans = _oracle_prefill(w, x)
    assert len(plans) >= 2
    assert not torch.isnan(out).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


def test_prefill_key_split_and_pipeline():
    # few (request, query tile, head) units and long contexts: the context
    # attention splits them over their keys (2 splits of 16+ key tiles) and
    # merges the splits, also into a continued request's stored partial
    # (second chunk of request 0; request 3 has two query tiles); the chunks
    # run through the two-buffer pipeline (gathers and up-projections on
    # their own streams)
    w = W.scaled(W.workload("uniform"), context_lens=[8192, 3, 0, 5000],
                 query_lens=[100, 20, 5, 130], num_heads=16, row_budget=4096,
                 max_context_chunk=4096, split_alignment=64, seed=51)
    x = W.make_inputs(w)
    out, lse = _run_prefill(w, x)
    ro, rl, plans = _oracle_prefill(w, x)
    assert len(plans) == 5 and plans[1].is_continuation and plans[4].is_continuation
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


def test_prefill_multi_tile_key_split():
    # requests of three and two query tiles over long contexts: several
    # query tiles of a request, each split over its keys into scratch slots
    # and merged, also into the stored partial of each continued request
    # (budget 4096: two chunks each); the new-token attention runs with the
    # final merge
    w = W.scaled(W.workload("uniform"), context_lens=[8192, 5000], query_lens=[300, 256],
                 num_heads=4, row_budget=4096, max_context_chunk=4096, split_alignment=64,
                 seed=55)
    x = W.make_inputs(w)
    M.mla_profile_begin()
    out, lse = _run_prefill(w, x)
    names = [r[0] for r in M.mla_profile_end()]
    assert "attn_tc_kernel" in names and "split_combine_kernel" in names
    ro, rl, plans = _oracle_prefill(w, x)
    assert len(plans) >= 4 and any(p.is_continuation for p in plans)
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


def test_prefill_groups_small_chunks_into_one_launch_set():
    # three chunks, separated only by context-free requests and together
    # within the budget, run as one execution group: one gather, one
    # up-projection and one attention launch for all of them
    w = W.scaled(W.workload("uniform"), context_lens=[100, 0, 50, 0, 30],
                 query_lens=[5, 7, 130, 3, 9], num_heads=4, row_budget=4096,
                 max_context_chunk=4096, split_alignment=64, seed=52)
    x = W.make_inputs(w)
    n0 = M.mla_kernel_launches()
    out, lse = _run_prefill(w, x)
    launched = M.mla_kernel_launches() - n0
    ro, rl, plans = _oracle_prefill(w, x)
    assert len(plans) == 3
    # fill of context-free rows + gather + up-projection + attention of the
    # group + new-token up-projection + new-token attention, and on the
    # tensor-core path the query preparation (its new-token attention merges
    # in its epilogue), on the CUDA-core path a separate merge
    assert launched == 7
    assert not torch.isnan(out).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


def test_prefill_long_new_tokens_loop_path():
    """Long runs of new tokens (8.5 causal key tiles per unit on average)
    with prepared queries: the new-token attention and the final merge run
    on the looping kernel (its limit for prepared queries is above the one
    for the caller's queries); a request with context, one without, one
    with context after it; compared in full."""
    ctx, ql = [300, 0, 130], [2048, 700, 1100]
    w = W.scaled(W.workload("uniform"), context_lens=ctx, query_lens=ql, num_heads=16,
                 row_budget=1024, max_context_chunk=512, split_alignment=64, seed=59)
    x = W.make_inputs(w)
    M.mla_profile_begin()
    out, lse = _run_prefill(w, x)
    names = [r[0] for r in M.mla_profile_end()]
    assert names[-1] == "attn_tc_loop_kernel"
    ro, rl, _ = _oracle_prefill(w, x)
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


def test_prefill_loop_path_continuation_chunks():
    """Context chunks of 1024 keys (8 key tiles per unit) over 64 heads and a
    few query tiles: with prepared queries the group attention runs on the
    looping kernel, and the later chunks of a split request accumulate into
    its partial there; compared in full."""
    ctx, ql = [2500, 1800, 0, 2200], [300, 260, 50, 280]
    w = W.scaled(W.workload("uniform"), context_lens=ctx, query_lens=ql, num_heads=64,
                 row_budget=2048, max_context_chunk=1024, split_alignment=64, seed=61)
    x = W.make_inputs(w)
    M.mla_profile_begin()
    out, lse = _run_prefill(w, x)
    names = [r[0] for r in M.mla_profile_end()]
    assert names.count("attn_tc_loop_kernel") >= 2
    ro, rl, plans = _oracle_prefill(w, x)
    assert any(p.is_continuation for p in plans)
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


def test_prefill_last_group_with_new_tokens_in_one_launch():
    """Short last group: its context attention and the new-token attention
    run as one looping-kernel launch (each unit walks its request's context
    rows of that group, then its own new tokens causally).  Every kind of
    request: context only in earlier groups (A, its partial merged in the
    epilogue), continued into the last group (B, merged), context only in
    the last group (C, E: nothing to merge), none (D); compared in full."""
    ctx, ql = [1500, 900, 200, 0, 150], [99, 130, 60, 20, 200]
    w = W.scaled(W.workload("uniform"), context_lens=ctx, query_lens=ql, num_heads=64,
                 row_budget=1024, max_context_chunk=1024, split_alignment=64, seed=67)
    x = W.make_inputs(w)
    plans = M.mla_plan_context_chunks(ctx, w.row_budget, w.max_context_chunk,
                                      w.split_alignment)
    # chunks: A | A's rest + B | B's rest + C | E; the last execution group
    # is the last two (B's continuation with C, then E)
    assert [c.is_continuation for c in plans] == [False, True, True, False]
    assert plans[2].request_start == 1 and plans[2].rows + plans[3].rows <= w.row_budget
    M.mla_profile_begin()
    out, lse = _run_prefill(w, x)
    recs = M.mla_profile_end()
    roles = [r[4] for r in recs]
    assert recs[-1][0] == "attn_tc_loop_kernel"
    assert recs[-1][4] == "a6-a10 last context group + new tokens"
    assert "a9-a10 new-token attention + merge" not in roles
    ro, rl, _ = _oracle_prefill(w, x)
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


@pytest.mark.parametrize("ctx,ql,heads,budget,split", [
    ([4800, 0, 5000, 4500], [250, 10, 200, 400], 96, 6144, False),
    ([6000, 9000], [300, 300], 64, 8192, True)])
def test_prefill_persistent_attention(ctx, ql, heads, budget, split):
    """Context groups of 384-576 (query tile, head) units of 18-27 key tiles
    with prepared queries take the persistent one-unit kernel (a CTA per SM
    walking several units); the last group continues a request: accumulating
    into the stored partial in the kernel's epilogue, or writing key-split
    scratch slots that split_combine merges into it; compared on every token
    for six heads (oracle runs on those heads' W_kv_b rows and query
    columns), every head checked for NaN."""
    w = W.scaled(W.workload("uniform"), context_lens=ctx, query_lens=ql, num_heads=heads,
                 row_budget=budget, max_context_chunk=budget, split_alignment=64, seed=63)
    x = W.make_inputs(w)
    M.mla_profile_begin()
    out, lse = _run_prefill(w, x)
    rec = M.mla_profile_end()
    names = [r[0] for r in rec]
    assert "attn_tc_persist_kernel" in names
    assert ("split_combine_kernel" in names) or not split
    assert not torch.isnan(out).any().item() and not torch.isnan(lse).any().item()
    H, Dn, Dv = w.num_heads, w.qk_nope_dim, w.v_dim
    q = x["q"].float().numpy()
    lat = x["new_latent"].float().numpy()
    cache = x["kv_cache"].float().numpy()
    bt = x["block_table"].numpy()
    wk = x["w_kv_b"].float().numpy()
    d1 = O.MlaDims(1, w.kv_lora_rank, w.qk_rope_dim, Dn, Dv, w.block_size, w.softmax_scale)
    for h in (0, 1, 37, 50, H - 2, H - 1):
        ro, rl, _ = O.chunked_prefill(q[:, h:h + 1], lat, cache, bt,
                                      wk[h * (Dn + Dv):(h + 1) * (Dn + Dv)], w.context_lens,
                                      w.query_lens, d1, w.row_budget, w.max_context_chunk,
                                      w.split_alignment)
        assert_close(f64(out[:, h]), ro[:, 0], 2e-2, 2e-2, what=f"O head {h}")
        assert_close(f64(lse[h]), rl[0], 1e-3, what=f"LSE head {h}")


@pytest.mark.parametrize("seed", [73, 74, 75, 76])
def test_prefill_final_launch_edge_cases(seed):
    """The final launch with the last group's context over ragged shapes,
    compared in full.  Seed 73 is fixed: the last group holds a context of
    exactly one key tile (128 rows) and a request with one new token, an
    earlier group a request with context but no new tokens, and
    context-free requests sit between and after the groups.  The others
    draw 10 requests (context 0-700 rows, 0-260 new tokens) and take
    whichever final launch their plan gives."""
    if seed == 73:
        ctx, ql = [256, 700, 0, 128, 390, 0], [40, 0, 130, 200, 1, 77]
    else:
        rng = np.random.default_rng(seed)
        ctx = [int(c) if rng.random() > 0.25 else 0 for c in rng.integers(1, 700, 10)]
        ql = [int(q) for q in rng.integers(0, 260, 10)]
    w = W.scaled(W.workload("uniform"), context_lens=ctx, query_lens=ql, num_heads=32,
                 row_budget=1024, max_context_chunk=512, split_alignment=64, seed=seed)
    x = W.make_inputs(w)
    M.mla_profile_begin()
    out, lse = _run_prefill(w, x)
    recs = M.mla_profile_end()
    if seed == 73:
        assert recs[-1][0] == "attn_tc_loop_kernel"
        assert recs[-1][4] == "a6-a10 last context group + new tokens"
    ro, rl, _ = _oracle_prefill(w, x)
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


def test_prefill_last_group_with_new_tokens_persistent():
    """A long last group (a 3544-row continuation, 28 key tiles) with the
    new tokens over 96 heads: the final launch takes the persistent kernel
    (about 23 key tiles per unit), each unit walking the group's context
    rows and then its new tokens causally; the continued request merges
    with its first chunk's partial, the other has no context in that group
    but its own partial; compared on every token for six heads, every head
    checked for NaN."""
    ctx, ql = [600, 7000], [100, 300]
    w = W.scaled(W.workload("uniform"), context_lens=ctx, query_lens=ql, num_heads=96,
                 row_budget=4096, max_context_chunk=4096, split_alignment=64, seed=71)
    x = W.make_inputs(w)
    plans = M.mla_plan_context_chunks(ctx, w.row_budget, w.max_context_chunk,
                                      w.split_alignment)
    assert [c.is_continuation for c in plans] == [False, True]
    M.mla_profile_begin()
    out, lse = _run_prefill(w, x)
    recs = M.mla_profile_end()
    assert recs[-1][0] == "attn_tc_persist_kernel"
    assert recs[-1][4] == "a6-a10 last context group + new tokens"
    assert not torch.isnan(out).any().item() and not torch.isnan(lse).any().item()
    H, Dn, Dv = w.num_heads, w.qk_nope_dim, w.v_dim
    q = x["q"].float().numpy()
    lat = x["new_latent"].float().numpy()
    cache = x["kv_cache"].float().numpy()
    bt = x["block_table"].numpy()
    wk = x["w_kv_b"].float().numpy()
    d1 = O.MlaDims(1, w.kv_lora_rank, w.qk_rope_dim, Dn, Dv, w.block_size, w.softmax_scale)
    for h in (0, 1, 37, 50, H - 2, H - 1):
        ro, rl, _ = O.chunked_prefill(q[:, h:h + 1], lat, cache, bt,
                                      wk[h * (Dn + Dv):(h + 1) * (Dn + Dv)], w.context_lens,
                                      w.query_lens, d1, w.row_budget, w.max_context_chunk,
                                      w.split_alignment)
        assert_close(f64(out[:, h]), ro[:, 0], 2e-2, 2e-2, what=f"O head {h}")
        assert_close(f64(lse[h]), rl[0], 1e-3, what=f"LSE head {h}")


def test_prefill_persistent_new_token_attention():
    """A request with 4200 new tokens (33 query tiles, 17 causal key tiles
    per unit on average, past the looping kernel's limit) over 16 heads:
    the new-token attention with the final merge runs on the persistent
    one-unit kernel (causal masking, the context partial merged in its
    epilogue, bf16 output); a second request without context; compared in
    full."""
    w = W.scaled(W.workload("uniform"), context_lens=[300, 0], query_lens=[4200, 90],
                 num_heads=16, row_budget=4096, max_context_chunk=4096, split_alignment=64,
                 seed=67)
    x = W.make_inputs(w)
    M.mla_profile_begin()
    out, lse = _run_prefill(w, x)
    names = [r[0] for r in M.mla_profile_end()]
    assert names[-1] == "attn_tc_persist_kernel"
    ro, rl, _ = _oracle_prefill(w, x)
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


def test_prefill_many_short_requests_loop_path():
    # 64 heads and many short requests: more (query tile, head) units than
    # SMs with few key tiles each, so the group attention and the new-token
    # attention (with the final merge) run on the looping kernel, with the
    # prepared queries; a continuation (budget 256), context-free requests
    # between and after the ones with context; compared in full
    rng = np.random.default_rng(53)
    ctx = [int(x) for x in rng.integers(0, 300, size=12)]
    ctx[3] = 0
    ctx[7] = 0
    ctx[1] = 600                       # split over three chunks of 256
    ctx += [0, 0]                      # context-free tail
    ql = [int(x) for x in rng.integers(1, 200, size=len(ctx))]
    w = W.scaled(W.workload("uniform"), context_lens=ctx, query_lens=ql, num_heads=64,
                 row_budget=1024, max_context_chunk=256, split_alignment=64, seed=53)
    x = W.make_inputs(w)
    out, lse = _run_prefill(w, x)
    ro, rl, plans = _oracle_prefill(w, x)
    assert any(p.is_continuation for p in plans)
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


@pytest.mark.parametrize("seed", [61, 62, 63])
def test_prefill_random_batches(seed):
    # seeded random batches over the execution paths at once: random context
    # and query lengths (some zero), random budget and split cap, 32 heads
    # (enough units for the looping attention, few enough for key splits when
    # a request is long), compared in full with the oracle
    rng = np.random.default_rng(seed)
    R = int(rng.integers(4, 14))
    ctx = [int(x) if rng.random() > 0.25 else 0 for x in rng.integers(1, 1500, size=R)]
    ctx[int(rng.integers(0, R))] = int(rng.integers(3000, 6000))   # one long request
    ql = [int(x) if rng.random() > 0.1 else 0 for x in rng.integers(1, 300, size=R)]
    ql[0] = max(ql[0], 1)
    budget = int(rng.choice([512, 1024, 2048, 4096, 8192]))
    mcc = int(rng.choice([budget, max(64, budget // 4)]))
    w = W.scaled(W.workload("uniform"), context_lens=ctx, query_lens=ql, num_heads=32,
                 row_budget=budget, max_context_chunk=mcc, split_alignment=64, seed=seed)
    x = W.make_inputs(w)
    out, lse = _run_prefill(w, x)
    ro, rl, _ = _oracle_prefill(w, x)
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


EDGE_CASES = {
    # no request has context: the output is the new-token attention alone
    "no_context": dict(context_lens=[0, 0, 0], query_lens=[5, 1, 130]),
    # only the last request has context; a context-free head of the batch
    "context_last": dict(context_lens=[0, 0, 77], query_lens=[3, 2, 9]),
    # a request with context but no new tokens, one with a single context row
    "zero_query": dict(context_lens=[300, 1, 64, 129], query_lens=[0, 1, 2, 128]),
    # one request spread over five chunks (continuations), budget = alignment
    "many_continuations": dict(context_lens=[320, 5], query_lens=[17, 3], row_budget=64,
                               max_context_chunk=64),
    # a context-free tail after the last request with context
    "empty_tail": dict(context_lens=[200, 0, 0], query_lens=[4, 6, 1]),
}


@pytest.mark.parametrize("case", sorted(EDGE_CASES))
def test_prefill_edge_cases(case):
    kw = dict(row_budget=512, max_context_chunk=512)
    kw.update(EDGE_CASES[case])
    w = W.scaled(W.workload("uniform"), num_heads=4, split_alignment=64, seed=48, **kw)
    x = W.make_inputs(w)
    out, lse = _run_prefill(w, x)
    ro, rl, _ = _oracle_prefill(w, x)
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


def test_prefill_no_new_tokens_is_a_no_op():
    w = W.scaled(W.workload("uniform"), context_lens=[100, 0], query_lens=[0, 0], num_heads=2,
                 row_budget=512, max_context_chunk=512, seed=49)
    x = W.make_inputs(w)
    g = to_dev(x)
    d = M.Dims.of(w)
    ws = torch.empty(max(1, M.mla_prefill_workspace_bytes(d, w.context_lens, w.query_lens, 512,
                                                          512, 64)), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty(0, 2, 128, dtype=torch.bfloat16, device=DEV)
    M.mla_chunked_prefill(d, w.context_lens, w.query_lens, 512, 512, 64, g["q"], g["new_latent"],
                          g["kv_cache"], g["block_table"], g["w_kv_b"], ws, out)
    torch.cuda.synchronize()


def test_chunk_entry_composes_to_prefill():
    """mla_context_chunk_attn per chunk + fill + new-token attention + merge
    gives what mla_chunked_prefill gives (which, on the tensor-core path,
    merges inside the new-token attention: equal up to one bf16 rounding)."""
    w = W.scaled(W.workload("uniform"), context_lens=[200, 0, 900, 50],
                 query_lens=[20, 5, 130, 9], num_heads=4, row_budget=512,
                 max_context_chunk=512, split_alignment=64, seed=45)
    x = W.make_inputs(w)
    g = to_dev(x)
    out_ref, lse_ref = _run_prefill(w, x)
    d = M.Dims.of(w)
    T, H = w.num_tokens, w.num_heads
    qsl = P.query_start_loc(w.query_lens)
    chunks = M.mla_plan_context_chunks(w.context_lens, 512, 512, 64)
    op = torch.full((T, H, 128), float("nan"), device=DEV)
    lp = torch.full((H, T), float("nan"), device=DEV)
    M.mla_fill_empty_rows(op, lp, P.empty_token_slices(w.context_lens, w.query_lens))
    ws = torch.empty(M.mla_chunk_workspace_bytes(d, max(c.rows for c in chunks), 8),
                     dtype=torch.uint8, device=DEV)
    for c in chunks:
        M.mla_context_chunk_attn(d, c, qsl, g["q"], g["kv_cache"], g["block_table"],
                                 g["w_kv_b"], ws, op, lp)
    kvs = torch.empty(T, H * 256, dtype=M.mla_chunk_kv_dtype(d), device=DEV)
    M.mla_kv_up_proj(d, g["new_latent"], T, g["w_kv_b"], kvs)
    os_ = torch.empty(T, H, 128, device=DEV)
    ls = torch.empty(H, T, device=DEV)
    M.mla_varlen_attn(d, True, qsl, qsl, g["q"], kvs, g["new_latent"], os_, ls)
    out = torch.empty(T, H, 128, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(H, T, device=DEV)
    M.merge_attn_states(out, lse, op, lp, os_, ls,
                        P.prefix_num_tokens(w.context_lens, w.query_lens))
    torch.cuda.synchronize()
    assert_close(f64(out), f64(out_ref), 1e-6, 2.0 ** -7, what="O")
    assert_close(f64(lse), f64(lse_ref), 1e-5, what="LSE")


def _run_equal_window(w, x):
    g = to_dev(x)
    T = w.num_tokens
    out = torch.full((T, w.num_heads, w.v_dim), float("nan"), dtype=w.torch_dtype, device=DEV)
    out_lse = torch.full((w.num_heads, T), float("nan"), device=DEV)
    d = M.Dims.of(w)
    ws = torch.empty(M.mla_prefill_equal_window_workspace_bytes(
        d, w.context_lens, w.query_lens, w.row_budget, w.split_alignment),
        dtype=torch.uint8, device=DEV)
    M.mla_chunked_prefill_equal_window(d, w.context_lens, w.query_lens, w.row_budget,
                                       w.split_alignment, g["q"], g["new_latent"], g["kv_cache"],
                                       g["block_table"], g["w_kv_b"], ws, out, out_lse)
    torch.cuda.synchronize()
    return out, out_lse


@pytest.mark.parametrize("kind", ["tiny", "deepseek"])
def test_equal_window_comparator_matches_oracle(kind):
    """The old equal-window scheme (kept as a comparator) gives the oracle's
    result for that scheme, which equals the per-request packing's."""
    if kind == "tiny":
        w = W.scaled(W.workload("tiny"), row_budget=64, max_context_chunk=64)
    else:
        w = W.scaled(W.workload("uniform"), context_lens=[0, 300, 1000, 5, 0, 700, 64],
                     query_lens=[3, 130, 1, 40, 7, 200, 0], num_heads=8, row_budget=1024,
                     max_context_chunk=1024, split_alignment=64, seed=47)
    x = W.make_inputs(w)
    out, lse = _run_equal_window(w, x)
    n = np_inputs(x)
    ro, rl, chunks = O.equal_window_prefill(n["q"], n["new_latent"], n["kv_cache"],
                                            n["block_table"], n["w_kv_b"], w.context_lens,
                                            w.query_lens, odims(w), w.row_budget,
                                            w.split_alignment)
    assert chunks > 1
    assert not torch.isnan(out).any()
    assert_close(f64(out), ro, 2e-2, 2e-2, what="O")
    assert_close(f64(lse), rl, 1e-3, what="LSE")


# ------------------------------------- full sizes, every token of 3 heads --
@pytest.mark.slow
@pytest.mark.parametrize("name", ["uniform", "hetero", "long"])
def test_prefill_full_size_every_token_three_heads(name):
    """The full workloads through mla_chunked_prefill (the launch
    configuration bench.py times), compared element by element with the
    oracle on every token for heads 0, H-1 and one seeded head: the oracle's
    chunked prefill run on those heads' W_kv_b rows and query columns (heads
    are independent in MLA attention, so a one-head oracle run is that head's
    exact reference).  Every other head is checked for NaN."""
    w = W.workload(name)
    x = W.make_inputs(w)
    out, lse = _run_prefill(w, x)
    T, H = w.num_tokens, w.num_heads
    Dn, Dv = w.qk_nope_dim, w.v_dim
    assert not torch.isnan(out).any().item() and not torch.isnan(lse).any().item()
    heads = sorted({0, H - 1, int(np.random.default_rng(77 + len(name)).integers(1, H - 1))})
    q = x["q"].float().numpy()
    lat = x["new_latent"].float().numpy()
    cache = x["kv_cache"].float().numpy()
    bt = x["block_table"].numpy()
    wk = x["w_kv_b"].float().numpy()
    d1 = O.MlaDims(1, w.kv_lora_rank, w.qk_rope_dim, Dn, Dv, w.block_size, w.softmax_scale)
    for h in heads:
        ro, rl, _ = O.chunked_prefill(q[:, h:h + 1], lat, cache, bt,
                                      wk[h * (Dn + Dv):(h + 1) * (Dn + Dv)], w.context_lens,
                                      w.query_lens, d1, w.row_budget, w.max_context_chunk,
                                      w.split_alignment)
        assert_close(f64(out[:, h]), ro[:, 0], 2e-2, 2e-2, what=f"O head {h}")
        assert_close(f64(lse[h]), rl[0], 1e-3, what=f"LSE head {h}")
