"""Host logic of bench.py (no GPU): the per-step split of the launch
records, the overlap-attributed time, the in-step rooflines and the
spec bar, on synthetic launch records."""

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
    bar = br["north_star_bar"]
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
