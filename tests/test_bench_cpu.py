"""Host logic of bench.py (no GPU): the per-step split of the launch
records, the overlap-attributed time, the in-step rooflines and the
tensor-target bar, on synthetic launch records."""

import math

import pytest

import bench
from mla_chunked_context_gb300 import workloads as W
from oracle import planner as P


def _rec(kernel, stream, start, ms, role):
    return (kernel, stream, start, ms, role)


def test_attributed_time_shares_overlap_and_sums_to_busy_time():
    rs = [_rec("a", 0, 0.0, 2.0, "x"), _rec("b", 1, 1.0, 2.0, "y"), _rec("c", 0, 4.0, 1.0, "x")]
    at = bench.attributed_ms(rs)
    # [0,1) x alone, [1,2) x and y, [2,3) y alone, [4,5) x alone; idle [3,4)
    assert math.isclose(at["x"], 1.0 + 0.5 + 1.0)
    assert math.isclose(at["y"], 0.5 + 1.0)
    assert math.isclose(sum(at.values()), 4.0)


def test_split_steps_needs_equal_steps():
    rs = [_rec("k", 0, float(i), 1.0, "r") for i in range(6)]
    assert [len(s) for s in bench.split_steps(rs, 3)] == [2, 2, 2]
    with pytest.raises(RuntimeError):
        bench.split_steps(rs, 4)


def test_breakdown_bar_and_rooflines():
    w = W.workload("uniform")
    plans = P.plan_mla_context_chunks(w.context_lens, w.row_budget, w.max_context_chunk,
                                      w.split_alignment)
    fl = bench.flops_of(w, plans)
    peaks = dict(hbm_gbs=6000.0, bf16_tflops=2000.0, bf16_tflops_sustained=1800.0,
                 source="test")
    one = [_rec("gather", 1, 0.0, 0.1, bench.ROLE_GATHER),
           _rec("gemm", 2, 0.1, 1.5, bench.ROLE_UP),
           _rec("attn", 0, 1.6, 2.5, bench.ROLE_ATTN),
           _rec("gemm", 2, 1.7, 0.2, bench.ROLE_UP_NEW),
           _rec("attn", 0, 4.1, 0.6, bench.ROLE_ATTN_NEW)]
    two = [(k, s, t + 10.0, ms, r) for k, s, t, ms, r in one]
    br = bench.breakdown_of(one + two, 2, w, plans, peaks)
    bar = br["target_bar"]
    assert math.isclose(bar["a4_a7_span_ms"], 4.1)
    assert math.isclose(bar["tflops"], (fl["up_proj_ctx"] + fl["attn_ctx"]) / 4.1e-3 / 1e12)
    up = br["rooflines"]["up_proj"]
    assert math.isclose(up["ms_per_step"], 1.7) and up["launches_per_step"] == 2
    assert math.isclose(up["achieved"], (fl["up_proj_ctx"] + fl["up_proj_new"]) / 1.7e-3 / 1e12)
    g = br["rooflines"]["gather"]
    assert g["unit"] == "GB/s" and math.isclose(
        g["achieved"], 2 * fl["context_rows"] * 576 * 2 / 0.1e-3 / 1e9)
    assert [e["kernel"] for e in br["timeline_first_step"]] == ["gather", "gemm", "attn", "gemm",
                                                               "attn"]


def _plans(w):
    return P.plan_mla_context_chunks(w.context_lens, w.row_budget, w.max_context_chunk,
                                     w.split_alignment)


def test_execution_groups_follow_the_prefill():
    """Chunks run together until a continuation or the row budget ends the
    group: the hetero batch's four long-request chunks alone, its seven
    small chunks together; the uniform batch in one group."""
    w = W.workload("hetero")
    assert [len(g) for g in bench.execution_groups(_plans(w), w.row_budget)] == [1, 1, 1, 1, 7]
    w = W.workload("uniform")
    assert [len(g) for g in bench.execution_groups(_plans(w), w.row_budget)] == [1]


def test_last_group_work_splits_the_context_attention():
    """The final launch's FLOPs are the last group's context attention plus
    the new-token attention, the rest stay with the context attention; its
    bytes are fewer than those of the two launches it replaces."""
    w = W.workload("hetero")
    plans = _plans(w)
    fl = bench.flops_of(w, plans)
    last_fl, last_by, ctx_fl, ctx_by = bench.last_group_work(w, plans)
    assert math.isclose(last_fl + ctx_fl, fl["attn_ctx"] + fl["attn_new"], rel_tol=1e-12)
    assert ctx_fl < fl["attn_ctx"] and ctx_by < fl["attn_ctx_bytes"]
    last_ctx_by = fl["attn_ctx_bytes"] - ctx_by
    assert last_by < last_ctx_by + fl["attn_new_bytes"]
    # the queries once, the new tokens' and the group's K/V, the output
    H, Dn, Dv, Pd = w.num_heads, w.qk_nope_dim, w.v_dim, w.qk_rope_dim
    rows = sum(sum(c.seq_lens) for c in bench.execution_groups(plans, w.row_budget)[-1])
    T = w.num_tokens
    assert last_by >= (T * H * (Dn + Pd) * 2 + (T + rows) * (H * (Dn + Dv) * 2 + Pd * 2)
                       + T * H * (Dv * 2 + 4))


def test_breakdown_with_the_final_launch_role():
    """With the last group's context attention in the final launch, that
    launch is its own roofline class and the context attention class counts
    the other groups only."""
    w = W.workload("hetero")
    plans = _plans(w)
    peaks = dict(hbm_gbs=6000.0, bf16_tflops=2000.0, bf16_tflops_sustained=1800.0,
                 source="test")
    one = [_rec("gather", 1, 0.0, 0.1, bench.ROLE_GATHER),
           _rec("gemm", 2, 0.1, 1.5, bench.ROLE_UP),
           _rec("attn", 0, 1.6, 2.5, bench.ROLE_ATTN),
           _rec("gemm", 2, 1.7, 0.2, bench.ROLE_UP_NEW),
           _rec("loop", 0, 4.1, 0.5, bench.ROLE_LAST)]
    br = bench.breakdown_of(one, 1, w, plans, peaks)
    last_fl, last_by, ctx_fl, ctx_by = bench.last_group_work(w, plans)
    rl = br["rooflines"]
    assert "new_token_attention_merge" not in rl
    assert rl["context_attention"]["flops_per_step"] == ctx_fl
    assert rl["context_attention"]["bytes_per_step"] == ctx_by
    fin = rl["last_group_and_new_token_attention"]
    assert fin["flops_per_step"] == last_fl and fin["bytes_per_step"] == last_by
    assert math.isclose(fin["ms_per_step"], 0.5)
    # the bar's span ends with the final launch
    assert math.isclose(br["target_bar"]["a4_a7_span_ms"], 4.6)
