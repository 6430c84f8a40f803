"""Host-side checks of the C ABI (no GPU needed): the library loads and
exports every function the header declares; the C++ planner matches the
oracle planner bit for bit; argument checks return their error codes before
anything touches a GPU."""

import ctypes as C
import os
import re

import numpy as np
import pytest

import mla_chunked_context_gb300 as M
from mla_chunked_context_gb300 import _lib, build, workloads as W
from oracle import planner as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session", autouse=True)
def built_library():
    srcs = [os.path.join(build.CSRC, f) for f in os.listdir(build.CSRC)]
    hdr = os.path.join(ROOT, "include", "mla_chunked_context.h")
    newest = max(os.path.getmtime(p) for p in srcs + [hdr])
    if not os.path.exists(build.LIB) or os.path.getmtime(build.LIB) < newest:
        build.build()
    return build.LIB


def header_functions():
    text = open(os.path.join(ROOT, "include", "mla_chunked_context.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^int\s+(\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol():
    names = header_functions()
    assert len(names) >= 12
    assert set(names) == set(_lib.EXPORTED)
    L = C.CDLL(build.LIB)
    for n in names:
        assert hasattr(L, n), n


def _same(c_plans, o_plans):
    assert len(c_plans) == len(o_plans)
    for a, b in zip(c_plans, o_plans):
        assert (a.request_start, a.request_end, a.starts, a.seq_lens, a.is_continuation) == \
               (b.request_start, b.request_end, b.starts, b.seq_lens, b.is_continuation)
        assert a.rows == sum(b.seq_lens)


def test_c_planner_worked_example_and_workloads():
    for a in (1, 16, 64, 256):
        _same(M.mla_plan_context_chunks([768, 512, 512], 1024, 1024, a),
              P.plan_mla_context_chunks([768, 512, 512], 1024, 1024, a))
    for name in ("tiny", "uniform", "hetero", "long"):
        w = W.workload(name)
        _same(M.mla_plan_context_chunks(w.context_lens, w.row_budget, w.max_context_chunk,
                                        w.split_alignment),
              P.plan_mla_context_chunks(w.context_lens, w.row_budget, w.max_context_chunk,
                                        w.split_alignment))


def test_c_planner_fuzz_bit_exact():
    rng = np.random.default_rng(21)
    for _ in range(10000):
        n = int(rng.integers(1, 14))
        ctx = [int(x) if rng.random() > 0.25 else 0 for x in rng.integers(1, 5000, size=n)]
        align = int(rng.choice([1, 2, 16, 64, 128]))
        budget = int(rng.integers(align, 6000))
        mcc = int(rng.choice([budget, max(align, budget // 3), 10 ** 9]))
        _same(M.mla_plan_context_chunks(ctx, budget, mcc, align),
              P.plan_mla_context_chunks(ctx, budget, mcc, align))


def test_c_planner_padded_rows_callback():
    rows_of = lambda x: (x + 3) // 4  # noqa: E731
    rng = np.random.default_rng(22)
    for _ in range(300):
        ctx = [int(x) for x in rng.integers(0, 5000, size=int(rng.integers(1, 8)))]
        budget = int(rng.integers(64, 2000))
        a = M.mla_plan_context_chunks(ctx, budget, 10 ** 9, 16, rows_of)
        b = P.plan_mla_context_chunks(ctx, budget, 10 ** 9, 16, rows_of)
        assert len(a) == len(b)
        for x, y in zip(a, b):
            assert (x.starts, x.seq_lens) == (y.starts, y.seq_lens)
            assert x.rows == sum(rows_of(s + l) - rows_of(s) for s, l in zip(y.starts, y.seq_lens))


def test_c_planner_errors():
    with pytest.raises(M.MlaError) as e:
        M.mla_plan_context_chunks([100], 8, 8, 16)
    assert e.value.code == _lib.MLA_ERR_PLANNER_STUCK
    with pytest.raises(M.MlaError) as e:
        M.mla_plan_context_chunks([-1], 8, 8, 1)
    assert e.value.code == _lib.MLA_ERR_INVALID
    with pytest.raises(M.MlaError) as e:
        M.mla_plan_context_chunks([5], 0, 8, 1)
    assert e.value.code == _lib.MLA_ERR_INVALID
    assert M.mla_plan_context_chunks([0, 0], 8, 8, 1) == []
    # caps too small
    L = _lib.lib()
    ctx = _lib._i32_host([10, 10])
    chunks = (_lib.mla_chunk_t * 1)()
    s = (C.c_int32 * 1)()
    l = (C.c_int32 * 1)()
    nc, ne = C.c_int32(0), C.c_int32(0)
    rc = L.mla_plan_context_chunks(ctx, 2, 10, 10, 1, C.cast(None, _lib.PADDED_ROWS_FN), None,
                                   chunks, 1, s, l, 1, C.byref(nc), C.byref(ne))
    assert rc == _lib.MLA_ERR_TOO_SMALL and nc.value == 2 and ne.value == 2


def test_workspace_queries():
    w = W.workload("uniform")
    dims = _lib.Dims.of(w)
    b = M.mla_prefill_workspace_bytes(dims, w.context_lens, w.query_lens, w.row_budget,
                                      w.max_context_chunk, w.split_alignment)
    T, H = w.num_tokens, w.num_heads
    rows = 65536
    kv_es = M.mla_chunk_kv_dtype(dims).itemsize
    split = 16 * H * 128 * (128 + 1) * 4        # key-split scratch of the context attention

    def lower(sets, rows, T):
        # buffer sets, prepared queries, new-token K/V, partials, split scratch
        return (sets * (rows * 576 * 2 + rows * H * 256 * kv_es) + T * H * 192 * 2 +
                T * H * 256 * kv_es + 2 * T * H * 128 * 4 + split)
    # one chunk: one buffer set
    assert lower(1, rows, T) <= b <= lower(1, rows, T) + 64 * 1024 * 1024
    # several chunks: two buffer sets for the pipeline
    h = W.workload("hetero")
    bh = M.mla_prefill_workspace_bytes(dims, h.context_lens, h.query_lens, h.row_budget,
                                       h.max_context_chunk, h.split_alignment)
    lo = lower(2, h.row_budget, h.num_tokens)
    assert lo <= bh <= lo + 64 * 1024 * 1024
    cb = M.mla_chunk_workspace_bytes(dims, 1000, 10)
    assert cb >= 1000 * 576 * 2 + 1000 * H * 256 * 2


def test_argument_errors_before_any_launch():
    L = _lib.lib()
    w = W.workload("tiny")
    d = _lib.Dims.of(w).c()
    # null outputs / inputs
    assert L.merge_attn_states(None, None, None, None, None, None, 4, 2, 8, 0, 1, 1, None) == \
        _lib.MLA_ERR_INVALID
    assert L.merge_attn_states(None, None, None, None, None, None, 4, 2, 12, 0, 1, 1, None) == \
        _lib.MLA_ERR_INVALID          # head_dim not a multiple of 8
    assert L.mla_kv_up_proj(C.byref(d), None, 80, 5, None, None, 0, None) == \
        _lib.MLA_ERR_INVALID
    assert L.mla_kv_up_proj(C.byref(d), None, 80, 5, None, None, 7, None) == \
        _lib.MLA_ERR_INVALID          # unknown K/V dtype
    bad = _lib.Dims.of(w)
    bad.v_dim = 12
    assert L.mla_kv_up_proj(C.byref(bad.c()), None, 80, 5, None, None, 0, None) == \
        _lib.MLA_ERR_UNSUPPORTED
    ctx, ql = _lib._i32_host(w.context_lens), _lib._i32_host(w.query_lens)
    rc = L.mla_chunked_prefill(C.byref(d), ctx, ql, 4, w.row_budget, w.max_context_chunk,
                               w.split_alignment, None, None, None, 0, None, 1, None, None, 0,
                               None, None, None, None)
    assert rc == _lib.MLA_ERR_INVALID
    # a budget below one aligned split
    rc = L.mla_chunked_prefill(C.byref(d), ctx, ql, 4, 8, 8, 16, None, None, None, 0, None, 1,
                               None, None, 0, None, None, None, None)
    assert rc == _lib.MLA_ERR_PLANNER_STUCK
    # workspace too small (non-null pointers that are never dereferenced)
    fake = C.c_void_p(16)
    rc = L.mla_chunked_prefill(C.byref(d), ctx, ql, 4, w.row_budget, w.max_context_chunk,
                               w.split_alignment, fake, fake, fake, 100, fake, 100, fake, fake,
                               16, fake, None, None, None)
    assert rc == _lib.MLA_ERR_TOO_SMALL
    # a context longer than the block table can address
    rc = L.mla_chunked_prefill(C.byref(d), ctx, ql, 4, w.row_budget, w.max_context_chunk,
                               w.split_alignment, fake, fake, fake, 100, fake, 2, fake, fake,
                               1 << 40, fake, None, None, None)
    assert rc == _lib.MLA_ERR_INVALID


def test_c_equal_window_planner_matches_oracle():
    rng = np.random.default_rng(23)
    for _ in range(2000):
        n = int(rng.integers(1, 12))
        ctx = [int(x) if rng.random() > 0.3 else 0 for x in rng.integers(1, 5000, size=n)]
        if not any(ctx):
            assert M.mla_plan_equal_window_chunks(ctx, 4096, 16) == (0, 0)
            continue
        align = int(rng.choice([1, 16, 64]))
        budget = int(rng.integers(align * n, 9000))
        win, starts, _, _ = P.plan_equal_window_chunks(ctx, budget, align)
        assert M.mla_plan_equal_window_chunks(ctx, budget, align) == (win, len(starts))
    w = W.workload("hetero")
    assert M.mla_plan_equal_window_chunks(w.context_lens, w.row_budget, w.split_alignment) == \
        (1280, 103)
    with pytest.raises(M.MlaError) as e:
        M.mla_plan_equal_window_chunks([5, 5, 5], 2, 1)
    assert e.value.code == _lib.MLA_ERR_PLANNER_STUCK


def test_fused_entry_host_checks():
    """mla_fused_context_attn: workspace size, argument errors, and the
    shape limit (at most 128 queries per sequence), all returned before
    anything is launched."""
    L = _lib.lib()
    w = W.workload("uniform")
    dims = _lib.Dims.of(w)
    d = dims.c()
    T, H = 512, w.num_heads
    need = T * H * 192 * 2 + 16 * H * 128 * (128 + 1) * 4
    got = M.mla_fused_attn_workspace_bytes(dims, T)
    assert need <= got <= need + 4096
    fake = C.c_void_p(16)
    ql, kl = _lib._i32_host([0, 100]), _lib._i32_host([0, 300])

    def call(q_loc, k_loc, q=fake, latent_ld=576, rows=300, n=1):
        return L.mla_fused_context_attn(C.byref(d), n, fake, fake, q_loc, k_loc, T, q, fake,
                                        latent_ld, rows, fake, None, fake, fake, fake, 1 << 30,
                                        None)
    assert call(ql, kl, q=None) == _lib.MLA_ERR_INVALID
    assert call(ql, kl, latent_ld=500) == _lib.MLA_ERR_INVALID
    assert call(ql, kl, rows=299) == _lib.MLA_ERR_INVALID            # keys past the latent rows
    assert call(_lib._i32_host([100, 0]), kl) == _lib.MLA_ERR_INVALID
    assert call(ql, kl, n=0) == _lib.MLA_OK                            # nothing to do
    # a sequence of two query tiles is refused whatever the GPU
    assert call(_lib._i32_host([0, 129]), kl) == _lib.MLA_ERR_UNSUPPORTED
