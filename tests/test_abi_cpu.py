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
    return sorted(set(re.findall(r"^(?:int|int32_t)\s+(\w+)\s*\(", text, flags=re.M)))


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
    assert L.mla_kv_up_proj(C.byref(d), None, 80, 5, None, None, 0, None, None) == \
        _lib.MLA_ERR_INVALID
    assert L.mla_kv_up_proj(C.byref(d), None, 80, 5, None, None, 7, None, None) == \
        _lib.MLA_ERR_INVALID          # unknown K/V dtype
    bad = _lib.Dims.of(w)
    bad.v_dim = 12
    assert L.mla_kv_up_proj(C.byref(bad.c()), None, 80, 5, None, None, 0, None, None) == \
        _lib.MLA_ERR_UNSUPPORTED
    ctx, ql = _lib._i32_host(w.context_lens), _lib._i32_host(w.query_lens)
    rc = L.mla_chunked_prefill(C.byref(d), ctx, ql, 4, w.row_budget, w.max_context_chunk,
                               w.split_alignment, None, None, None, 0, None, 1, None, None, 0,
                               None, None, None, 0, None, None)
    assert rc == _lib.MLA_ERR_INVALID
    # a budget below one aligned split
    rc = L.mla_chunked_prefill(C.byref(d), ctx, ql, 4, 8, 8, 16, None, None, None, 0, None, 1,
                               None, None, 0, None, None, None, 0, None, None)
    assert rc == _lib.MLA_ERR_PLANNER_STUCK
    # workspace too small (non-null pointers that are never dereferenced)
    fake = C.c_void_p(16)
    rc = L.mla_chunked_prefill(C.byref(d), ctx, ql, 4, w.row_budget, w.max_context_chunk,
                               w.split_alignment, fake, fake, fake, 100, fake, 100, fake, fake,
                               16, fake, None, None, 0, None, None)
    assert rc == _lib.MLA_ERR_TOO_SMALL
    # a context longer than the block table can address
    rc = L.mla_chunked_prefill(C.byref(d), ctx, ql, 4, w.row_budget, w.max_context_chunk,
                               w.split_alignment, fake, fake, fake, 100, fake, 2, fake, fake,
                               1 << 40, fake, None, None, 0, None, None)
    assert rc == _lib.MLA_ERR_INVALID


def test_alignment_and_dispatch_errors_before_any_launch():
    """Pointer alignment and the no-fallback rule: a misaligned O for the
    merge, a misaligned workspace or cache, and a DeepSeek-shaped bf16 call
    whose operands the tensor-core kernels cannot take all return an error
    code before anything is enqueued (fake pointers, never dereferenced)."""
    L = _lib.lib()
    ok, odd = C.c_void_p(256), C.c_void_p(256 + 8)
    # merge: O pointers 16-byte aligned, LSE pointers 4-byte aligned
    for args in ((odd, ok, ok), (ok, odd, ok), (ok, ok, odd)):
        out, po, so = args
        assert L.merge_attn_states(out, None, po, ok, so, ok, 4, 2, 8, 2, 1, 1, None) == \
            _lib.MLA_ERR_INVALID
    assert L.merge_attn_states(ok, None, ok, C.c_void_p(258), ok, ok, 4, 2, 8, 2, 1, 1,
                               None) == _lib.MLA_ERR_INVALID
    # a prefix that is never read (prefix_num_tokens = 0) needs no alignment
    assert L.merge_attn_states(ok, None, odd, None, ok, C.c_void_p(258), 4, 2, 8, 0, 1, 1,
                               None) == _lib.MLA_ERR_INVALID      # suffix LSE still checked
    w = W.workload("uniform")
    d = _lib.Dims.of(w).c()
    # gather: cache and workspace move as 16-byte pieces
    assert L.mla_gather_context_rows(C.byref(d), odd, 10, ok, 4, 1, ok, ok, ok, 64, ok, None,
                                     None) == _lib.MLA_ERR_INVALID
    # the tensor-core shape never takes the CUDA-core kernels: a misaligned
    # operand (or no tcgen05 GPU, as here) is MLA_ERR_UNSUPPORTED
    assert L.mla_kv_up_proj(C.byref(d), odd, 576, 64, ok, ok, _lib.MLA_DTYPE_F16, None,
                            None) == _lib.MLA_ERR_UNSUPPORTED
    assert L.mla_kv_up_proj(C.byref(d), ok, 576, 64, ok, ok, _lib.MLA_DTYPE_F32, None,
                            None) == _lib.MLA_ERR_UNSUPPORTED      # F32 K/V: not on that path
    ql, kl = _lib._i32_host([0, 4]), _lib._i32_host([0, 64])
    for q, kv_dtype in ((odd, _lib.MLA_DTYPE_F16), (ok, _lib.MLA_DTYPE_BF16)):
        assert L.mla_varlen_attn(C.byref(d), 0, 1, ok, ok, ql, kl, 4, q, ok, kv_dtype, 64, ok,
                                 576, None, ok, ok, None, None) == _lib.MLA_ERR_UNSUPPORTED
    ctx, qn = _lib._i32_host(w.context_lens), _lib._i32_host(w.query_lens)
    n = len(w.context_lens)
    big = 1 << 40

    def prefill(q=ok, ws=ok, cache=ok, pinned=None, pinned_bytes=0):
        return L.mla_chunked_prefill(C.byref(d), ctx, qn, n, w.row_budget, w.max_context_chunk,
                                     w.split_alignment, q, ok, cache, 100, ok, 1 << 20, ok, ws,
                                     big, ok, None, pinned, pinned_bytes, None, None)
    assert prefill(ws=odd) == _lib.MLA_ERR_INVALID
    assert prefill(cache=odd) == _lib.MLA_ERR_INVALID
    assert prefill(q=odd) == _lib.MLA_ERR_UNSUPPORTED
    # pinned metadata scratch below mla_prefill_pinned_bytes
    need = M.mla_prefill_pinned_bytes(_lib.Dims.of(w), w.context_lens, w.query_lens,
                                      w.row_budget, w.max_context_chunk, w.split_alignment)
    assert need > 0
    assert prefill(pinned=ok, pinned_bytes=need - 4) == _lib.MLA_ERR_TOO_SMALL


def test_pinned_bytes_counts_the_metadata():
    """The metadata of one prefill: per execution group (n requests) 5n + 2
    ints, two ints per empty-token slice, R + 1 query offsets, and the last
    group's context-row offsets (R + 1) and merge flags (R) over all
    requests."""
    w = W.workload("tiny")
    dims = _lib.Dims.of(w)
    got = M.mla_prefill_pinned_bytes(dims, w.context_lens, w.query_lens, w.row_budget,
                                     w.max_context_chunk, w.split_alignment)
    # tiny: the plan's chunks run as groups; bound it by one group per chunk
    plans = M.mla_plan_context_chunks(w.context_lens, w.row_budget, w.max_context_chunk,
                                      w.split_alignment)
    R = len(w.context_lens)
    empty = len(P.empty_token_slices(w.context_lens, w.query_lens))
    hi = (sum(5 * (c.request_end - c.request_start) + 2 for c in plans) + 2 * empty + R + 1
          + 2 * R + 1)
    assert 0 < got <= 4 * hi


def test_profile_with_no_launches():
    """mla_profile_begin / _end with nothing launched in between: no
    records, no CUDA call needed."""
    M.mla_profile_begin()
    assert M.mla_profile_end() == []


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
                                        None, None)
    assert call(ql, kl, q=None) == _lib.MLA_ERR_INVALID
    assert call(ql, kl, latent_ld=500) == _lib.MLA_ERR_INVALID
    assert call(ql, kl, rows=299) == _lib.MLA_ERR_INVALID            # keys past the latent rows
    assert call(_lib._i32_host([100, 0]), kl) == _lib.MLA_ERR_INVALID
    assert call(ql, kl, n=0) == _lib.MLA_OK                            # nothing to do
    # a sequence of two query tiles is refused whatever the GPU
    assert call(_lib._i32_host([0, 129]), kl) == _lib.MLA_ERR_UNSUPPORTED


def _walk_fused_plan(H, bounds, items):
    """Decode every cluster's range the way the fused kernel does; return
    the coverage count per flattened position and the (slot, head) writes."""
    tph = sum(t for _, t, _, _ in items)
    N = H * tph
    P = len(bounds) - 1
    starts = [tb for _, _, tb, _ in items]

    def pair_of(x):
        lo, hi = 0, P - 1
        while lo < hi:
            mid = (lo + hi + 1) >> 1
            if bounds[mid] <= x:
                lo = mid
            else:
                hi = mid - 1
        return lo
    cover = np.zeros(N, dtype=np.int64)
    writes = {}
    for c in range(P):
        f, f1 = bounds[c], bounds[c + 1]
        while f < f1:
            h, r = divmod(f, tph)
            i = max(k for k in range(len(items)) if starts[k] <= r)
            seq, tiles, tb, info = items[i]
            kt0 = r - tb
            kt1 = min(tiles, kt0 + (f1 - f))
            assert 0 <= kt0 < kt1 <= tiles
            cover[h * tph + tb + kt0:h * tph + tb + kt1] += 1
            sb, maxp = (info & 0xffff) - 1, info >> 16
            if sb >= 0:
                slot = sb + c - pair_of(h * tph + tb)
                assert sb <= slot < sb + maxp
                writes[(slot, h)] = writes.get((slot, h), 0) + 1
                if kt1 == tiles:       # the last piece clears the head's unused slots
                    for s2 in range(slot + 1, sb + maxp):
                        writes[(s2, h)] = writes.get((s2, h), 0) + 1
            f += kt1 - kt0
    return cover, writes


def test_fused_plan_covers_every_tile_once():
    """The fused kernel's work split (C++ host planner): every (head,
    sequence, key tile) lands in exactly one cluster; each cut item's scratch
    slots are written exactly once per head (a piece or a clear); the slot
    and group limits hold; equal shares when nothing is snapped."""
    rng = np.random.default_rng(7)
    cases = [(128, [99], [32768], 76, 16), (16, [1, 128, 77, 5, 0, 100],
                                            [5, 300, 129, 1000, 64, 0], 76, 16),
             (4, [1] * 40, [300] * 40, 76, 16), (1, [1, 128], [1, 128], 76, 16),
             (3, [57], [3000], 76, 16), (7, [57], [3000], 76, 0)]
    for _ in range(60):
        n = int(rng.integers(1, 30))
        H = int(rng.choice([1, 2, 3, 16, 128]))
        ql = [int(x) for x in rng.integers(0, 129, n)]
        kl = [int(x) for x in rng.integers(0, 4000, n) * (rng.random(n) < 0.8)]
        cases.append((H, ql, kl, int(rng.choice([1, 2, 7, 76, 300])),
                      int(rng.choice([0, 4, 16]))))
    for H, ql, kl, clusters, slots in cases:
        q_loc = [0] + [int(x) for x in np.cumsum(ql)]
        k_loc = [0] + [int(x) for x in np.cumsum(kl)]
        bounds, items, groups = M.mla_fused_attn_plan(H, q_loc, k_loc, clusters, slots)
        want = [i for i in range(len(ql)) if ql[i] > 0 and kl[i] > 0]
        assert [it[0] for it in items] == want
        if not want:
            continue
        tiles = [(kl[i] + 127) // 128 for i in want]
        assert [it[1] for it in items] == tiles
        assert [it[2] for it in items] == [int(x) for x in np.cumsum([0] + tiles[:-1])]
        N = H * sum(tiles)
        P = len(bounds) - 1
        assert P == min(clusters, 128, N) and bounds[0] == 0 and bounds[-1] == N
        assert all(a <= b for a, b in zip(bounds, bounds[1:]))
        cover, writes = _walk_fused_plan(H, bounds, items)
        assert (cover == 1).all()
        cut = [it for it in items if it[3]]
        assert len(cut) == groups <= 16
        assert sum(it[3] >> 16 for it in cut) <= slots
        for seq, _, _, info in cut:
            sb, maxp = (info & 0xffff) - 1, info >> 16
            for h in range(H):
                for s in range(sb, sb + maxp):
                    assert writes.get((s, h), 0) == 1, (H, ql, kl, seq, h, s)
        if bounds == [c * N // P for c in range(P + 1)]:
            assert max(b - a for a, b in zip(bounds, bounds[1:])) <= -(-N // P)
    with pytest.raises(M.MlaError) as e:
        M.mla_fused_attn_plan(16, [0, 129], [0, 300], 76, 16)
    assert e.value.code == _lib.MLA_ERR_UNSUPPORTED
