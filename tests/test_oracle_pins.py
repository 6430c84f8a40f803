"""Pins of the float64 oracle against what the pages and the mathematics fix.

No test here compares the oracle with itself: each one checks it against a
value printed on the pages (tests/golden), a closed form, brute force on tiny
inputs, or a library routine computing the same quantity another way
(torch's CPU scaled_dot_product_attention, the pages' own reference for the
chunked-context backends in the PR #50613 report, item 5).
The mutation tests at the end plant plausible mistakes in copies of oracle
functions and check that a pin fails for each.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import mla as O
from oracle import planner as P
from mla_chunked_context_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- planner --
def _plans_as_dicts(plans):
    return [dict(request_start=p.request_start, request_end=p.request_end,
                 starts=list(p.starts), seq_lens=list(p.seq_lens),
                 is_continuation=bool(p.is_continuation)) for p in plans]


def test_planner_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "planner_worked_example.json")))
    for a in g["alignments"]:
        plans = P.plan_mla_context_chunks(g["context_lens"], g["row_budget"],
                                          g["row_budget"], a)
        assert _plans_as_dicts(plans) == g["chunks"], a


def check_plan_invariants(ctx, plans, budget, rows_of=lambda x: x):
    """Invariants of the PR #50613 report, item 2 and the test names of
    test_mla_context_chunks.py: every context row gathered exactly once (no
    overlap, no hole), no chunk over the workspace, no context-free request
    in a chunk, a continuation only at a chunk's first request, chunks in
    request order."""
    covered = [0] * len(ctx)          # next row each request expects
    last_req = -1
    for p in plans:
        assert p.request_end - p.request_start == len(p.starts) == len(p.seq_lens)
        assert p.request_start >= last_req
        rows = 0
        for i, r in enumerate(range(p.request_start, p.request_end)):
            assert ctx[r] > 0
            assert p.seq_lens[i] > 0
            if i > 0:
                assert p.starts[i] == 0
            assert p.starts[i] == covered[r]          # no overlap, no hole
            covered[r] += p.seq_lens[i]
            assert covered[r] <= ctx[r]
            rows += rows_of(p.starts[i] + p.seq_lens[i]) - rows_of(p.starts[i])
        assert rows <= budget
        assert p.is_continuation == (p.starts[0] > 0)
        last_req = p.request_end - 1
    assert covered == list(ctx)


def test_planner_invariants_fuzz():
    rng = np.random.default_rng(7)
    for _ in range(3000):
        n = int(rng.integers(1, 12))
        ctx = [int(x) if rng.random() > 0.25 else 0
               for x in rng.integers(1, 3000, size=n)]
        align = int(rng.choice([1, 2, 16, 64]))
        budget = int(rng.integers(align, 4000))
        mcc = int(rng.choice([budget, budget // 2 + align, 10 ** 9]))
        plans = P.plan_mla_context_chunks(ctx, budget, mcc, align)
        check_plan_invariants(ctx, plans, budget)


def test_planner_invariants_padded_rows():
    # A padding function of the context-parallel kind (rows local to one of
    # 4 ranks); the budget applies to padded rows.
    rows_of = lambda x: (x + 3) // 4  # noqa: E731
    rng = np.random.default_rng(8)
    for _ in range(500):
        n = int(rng.integers(1, 8))
        ctx = [int(x) for x in rng.integers(0, 5000, size=n)]
        budget = int(rng.integers(64, 2000))
        plans = P.plan_mla_context_chunks(ctx, budget, 10 ** 9, 16, rows_of)
        check_plan_invariants(ctx, plans, budget, rows_of)


def test_planner_minimal_chunk_count():
    """With alignment 1 and no padding every chunk but a run's last is filled
    to the budget, so a run of requests with context between two empty ones
    needs exactly ceil(rows / budget) chunks (the "minimises chunks" claim of
    test_tail_splitting_minimizes_chunks), counted here by brute force."""
    rng = np.random.default_rng(9)
    for _ in range(2000):
        n = int(rng.integers(1, 10))
        ctx = [int(x) if rng.random() > 0.3 else 0 for x in rng.integers(1, 500, size=n)]
        budget = int(rng.integers(1, 700))
        plans = P.plan_mla_context_chunks(ctx, budget, budget, 1)
        want, run = 0, 0
        for c in ctx + [0]:
            if c == 0:
                want += -(-run // budget)
                run = 0
            else:
                run += c
        assert len(plans) == want


def test_planner_overflow_without_split_closes_chunk():
    # 1020 rows fill the chunk; 10 more cannot be split at alignment 16 and
    # must not be appended whole (1030 > 1024): they open the next chunk.
    plans = P.plan_mla_context_chunks([1020, 10], 1024, 1024, 16)
    assert _plans_as_dicts(plans) == [
        dict(request_start=0, request_end=1, starts=[0], seq_lens=[1020], is_continuation=False),
        dict(request_start=1, request_end=2, starts=[0], seq_lens=[10], is_continuation=False)]


def test_planner_budget_below_alignment_is_stuck():
    with pytest.raises(P.PlannerStuck):
        P.plan_mla_context_chunks([100], 8, 8, 16)


def test_planner_aligned_split_len_definition():
    # plain enumeration of every candidate length on tiny cases
    for start in range(0, 40, 7):
        for remaining in range(1, 70):
            for avail in range(0, 50, 3):
                for a in (1, 4, 16):
                    got = P.aligned_split_len(start, remaining, avail, 32, a)
                    ok = [x for x in range(0, remaining) if x % a == 0 and x <= 32 and x <= avail]
                    assert got == max(ok)


def test_planner_derived_workload_plans():
    t = W.workload("tiny")
    plans = P.plan_mla_context_chunks(t.context_lens, t.row_budget, t.max_context_chunk,
                                      t.split_alignment)
    assert _plans_as_dicts(plans) == [
        dict(request_start=1, request_end=3, starts=[0, 0], seq_lens=[64, 64], is_continuation=False),
        dict(request_start=2, request_end=3, starts=[64], seq_lens=[128], is_continuation=True),
        dict(request_start=2, request_end=4, starts=[192, 0], seq_lens=[8, 37], is_continuation=True)]
    u = W.workload("uniform")
    assert len(P.plan_mla_context_chunks(u.context_lens, 65536, 65536, 64)) == 1
    lg = W.workload("long")
    plans = P.plan_mla_context_chunks(lg.context_lens, 65536, 65536, 64)
    assert len(plans) == 4 and not any(p.is_continuation for p in plans)


# --------------------------------------------------------------- metadata --
def test_metadata_on_mask_test_shape(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "mask_empty_context.json")))
    lo, hi = g["masked_rows"]
    assert P.empty_token_slices(g["context_lens"], g["query_lens"]) == [(lo, hi)]
    assert P.prefix_num_tokens(g["context_lens"], g["query_lens"]) == g["num_tokens"]
    # a context-free tail is passed through, not merged
    assert P.prefix_num_tokens([5, 0, 0], [2, 3, 4]) == 2
    assert P.prefix_num_tokens([0, 0], [2, 3]) == 0


def test_chunk_metadata_offsets():
    plan = P.ChunkPlan(2, 5, [7, 0, 0], [3, 1, 2], True)
    m = P.chunk_metadata(plan, [1, 2, 3, 4, 5, 6])
    assert m.cu_seq_lens == [0, 3, 4, 6]
    assert m.token_to_seq == [0, 0, 0, 1, 2, 2]
    assert m.token_slice == (3, 15)
    assert m.max_seq_len == 3


# ----------------------------------------------------------------- gather --
def test_gather_reads_rows_in_logical_order():
    bs, R = 4, 3
    ctx = [5, 0, 9]
    nblk = [(c + bs - 1) // bs for c in ctx]
    phys = np.random.default_rng(1).permutation(sum(nblk))
    bt = np.zeros((R, max(nblk)), dtype=np.int32)
    cache = np.full((sum(nblk), bs, 3), np.nan)
    k = 0
    for r in range(R):
        for b in range(nblk[r]):
            bt[r, b] = phys[k]
            k += 1
            for s in range(bs):
                cache[bt[r, b], s] = [r, b * bs + s, 7.0]
    plan = P.ChunkPlan(0, 3, [2, 0, 0], [3, 0, 9], True)
    plan.seq_lens[1] = 0
    ws = O.gather_chunk(cache, bt, plan, bs)
    want = [[0, j, 7] for j in range(2, 5)] + [[2, j, 7] for j in range(9)]
    np.testing.assert_array_equal(ws, np.array(want, dtype=float))


# ------------------------------------------------------------ up-project --
def test_up_project_brute_force():
    rng = np.random.default_rng(2)
    d = O.MlaDims(num_heads=3, kv_lora_rank=5, qk_rope_dim=2, qk_nope_dim=4, v_dim=3,
                  block_size=4, softmax_scale=1.0)
    lat = rng.standard_normal((6, 7))
    w = rng.standard_normal((3 * 7, 5))
    kn, v = O.up_project(lat, w, d)
    for n in range(6):
        for h in range(3):
            for j in range(4):
                want = math.fsum(lat[n, l] * w[h * 7 + j, l] for l in range(5))
                assert abs(kn[n, h, j] - want) < 1e-12
            for j in range(3):
                want = math.fsum(lat[n, l] * w[h * 7 + 4 + j, l] for l in range(5))
                assert abs(v[n, h, j] - want) < 1e-12


# -------------------------------------------------------------- attention --
def _rand_attn(rng, m=5, n=7, H=3, Dn=4, P_=2, Dv=3):
    return (rng.standard_normal((m, H, Dn + P_)), rng.standard_normal((n, H, Dn)),
            rng.standard_normal((n, P_)), rng.standard_normal((n, H, Dv)))


def test_attention_single_key_closed_form():
    rng = np.random.default_rng(3)
    q, kn, kp, v = _rand_attn(rng, n=1)
    o, lse = O.attention_with_lse(q, kn, kp, v, 0.3)
    for m in range(q.shape[0]):
        for h in range(q.shape[1]):
            s = 0.3 * (math.fsum(q[m, h, :4] * kn[0, h]) + math.fsum(q[m, h, 4:] * kp[0]))
            assert abs(lse[h, m] - s) < 1e-12
    np.testing.assert_allclose(o, np.broadcast_to(v[0], o.shape), atol=1e-12)


def test_attention_identical_keys_and_zero_query():
    rng = np.random.default_rng(4)
    q, kn, kp, v = _rand_attn(rng, n=6)
    kn[:] = kn[0]
    kp[:] = kp[0]
    o, lse = O.attention_with_lse(q, kn, kp, v, 0.7)
    o1, l1 = O.attention_with_lse(q, kn[:1], kp[:1], v[:1], 0.7)
    np.testing.assert_allclose(lse, l1 + math.log(6), atol=1e-12)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=0), o.shape), atol=1e-12)
    q0 = np.zeros_like(q)
    q, kn, kp, v = _rand_attn(rng, n=9)
    o, lse = O.attention_with_lse(q0[:, :, :], kn, kp, v, 0.5)
    np.testing.assert_allclose(lse, math.log(9), atol=1e-12)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=0), o.shape), atol=1e-12)


def test_attention_no_keys_is_zero_and_neg_inf():
    rng = np.random.default_rng(5)
    q, kn, kp, v = _rand_attn(rng, n=4)
    vis = np.zeros((5, 4), dtype=bool)
    vis[2, 1] = True
    o, lse = O.attention_with_lse(q, kn, kp, v, 1.0, visible=vis)
    assert not np.isnan(o).any()
    for m in (0, 1, 3, 4):
        assert np.all(np.isneginf(lse[:, m])) and np.all(o[m] == 0)
    o0, l0 = O.attention_with_lse(q, kn[:0], kp[:0], v[:0], 1.0)
    assert np.all(o0 == 0) and np.all(np.isneginf(l0))


def test_attention_lse_brute_force():
    rng = np.random.default_rng(6)
    q, kn, kp, v = _rand_attn(rng, m=3, n=5, H=2)
    o, lse = O.attention_with_lse(q, kn, kp, v, 0.9)
    for m in range(3):
        for h in range(2):
            s = [0.9 * (math.fsum(q[m, h, d] * kn[j, h, d] for d in range(4))
                        + math.fsum(q[m, h, 4 + p] * kp[j, p] for p in range(2)))
                 for j in range(5)]
            z = math.fsum(math.exp(x) for x in s)
            assert abs(lse[h, m] - math.log(z)) < 1e-12
            for d in range(3):
                want = math.fsum(math.exp(s[j]) / z * v[j, h, d] for j in range(5))
                assert abs(o[m, h, d] - want) < 1e-12


def sdpa_reference(q, kn, kp, v, scale, visible=None):
    """torch CPU float64 scaled_dot_product_attention on concat(K_nope, k_pe)."""
    m, H, _ = q.shape
    n = kn.shape[0]
    k = np.concatenate([kn, np.broadcast_to(kp[:, None, :], (n, H, kp.shape[1]))], axis=2)
    tq = torch.from_numpy(np.ascontiguousarray(q.transpose(1, 0, 2)))[None]
    tk = torch.from_numpy(np.ascontiguousarray(k.transpose(1, 0, 2)))[None]
    tv = torch.from_numpy(np.ascontiguousarray(v.transpose(1, 0, 2)))[None]
    mask = None if visible is None else torch.from_numpy(np.asarray(visible, dtype=bool))
    out = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    return out[0].numpy().transpose(1, 0, 2)


def check_attention_vs_sdpa(attn):
    rng = np.random.default_rng(10)
    q, kn, kp, v = _rand_attn(rng, m=6, n=11, H=4, Dn=8, P_=4, Dv=5)
    vis = np.ones((6, 11), dtype=bool)
    vis[:, 5:] = np.tril(np.ones((6, 6), dtype=bool))      # context + causal
    for mask in (None, vis):
        o, _ = attn(q, kn, kp, v, 0.35, visible=mask)
        np.testing.assert_allclose(o, sdpa_reference(q, kn, kp, v, 0.35, mask), atol=1e-12)


def test_attention_matches_sdpa():
    check_attention_vs_sdpa(O.attention_with_lse)


# ------------------------------------------------------------------ merge --
def test_merge_both_empty_is_zero_not_nan():
    T, H, D = 4, 2, 3
    pO = np.full((T, H, D), np.nan)
    sO = np.full((T, H, D), np.nan)
    L = np.full((H, T), -np.inf)
    o, l = O.merge_attn_states(pO, L, sO, L, T)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_merge_identity_and_passthrough():
    rng = np.random.default_rng(11)
    T, H, D = 6, 3, 4
    pO, sO = rng.standard_normal((T, H, D)), rng.standard_normal((T, H, D))
    pL, sL = rng.standard_normal((H, T)), rng.standard_normal((H, T))
    garbage = np.full((T, H, D), np.nan)
    ninf = np.full((H, T), -np.inf)
    o, l = O.merge_attn_states(garbage, ninf, sO, sL, T)
    assert np.array_equal(o, sO) and np.array_equal(l, sL)
    o, l = O.merge_attn_states(pO, pL, garbage, ninf, T)
    assert np.array_equal(o, pO) and np.array_equal(l, pL)
    # tokens at or past prefix_num_tokens copy the suffix; the prefix there
    # is poison and never read
    pO2, pL2 = pO.copy(), pL.copy()
    pO2[4:] = np.nan
    pL2[:, 4:] = np.nan
    o, l = O.merge_attn_states(pO2, pL2, sO, sL, 4)
    assert np.array_equal(o[4:], sO[4:]) and np.array_equal(l[:, 4:], sL[:, 4:])
    assert not np.isnan(o).any()


def test_merge_associative():
    rng = np.random.default_rng(12)
    T, H, D = 5, 2, 3
    parts = [(rng.standard_normal((T, H, D)), 3 * rng.standard_normal((H, T))) for _ in range(3)]
    (a, la), (b, lb), (c, lc) = parts
    x1, y1 = O.merge_attn_states(*O.merge_attn_states(a, la, b, lb, T), c, lc, T)
    x2, y2 = O.merge_attn_states(a, la, *O.merge_attn_states(b, lb, c, lc, T), T)
    np.testing.assert_allclose(x1, x2, atol=1e-12)
    np.testing.assert_allclose(y1, y2, atol=1e-12)


def check_split_keys_merge(attn, merge):
    """Attention over a key set equals the merge of attention over two
    disjoint parts of it (the identity the chunked scheme relies on), with
    the whole-set result taken from torch's SDPA."""
    rng = np.random.default_rng(13)
    q, kn, kp, v = _rand_attn(rng, m=4, n=12, H=3)
    o1, l1 = attn(q, kn[:5], kp[:5], v[:5], 0.6)
    o2, l2 = attn(q, kn[5:], kp[5:], v[5:], 0.6)
    o, l = merge(o1, l1, o2, l2, 4)
    np.testing.assert_allclose(o, sdpa_reference(q, kn, kp, v, 0.6), atol=1e-12)
    _, lall = attn(q, kn, kp, v, 0.6)
    np.testing.assert_allclose(l, lall, atol=1e-12)


def test_merge_of_split_keys_equals_whole():
    check_split_keys_merge(O.attention_with_lse, O.merge_attn_states)


def test_mask_empty_context_page_test(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "mask_empty_context.json")))
    H, T, D = g["num_heads"], g["num_tokens"], g["head_dim"]
    lo, hi = g["masked_rows"]
    rng = np.random.default_rng(14)
    lse = rng.standard_normal((H, T))
    out = rng.standard_normal((T, H, D))
    out[lo:hi] = np.nan
    qsl = P.query_start_loc(g["query_lens"])
    csl = P.query_start_loc(g["context_lens"])
    l2, o2 = O.mask_empty_context(lse, out, qsl, csl)
    exp_l, exp_o = lse.copy(), out.copy()
    exp_l[:, lo:hi] = -np.inf
    exp_o[lo:hi] = 0.0
    assert np.array_equal(l2, exp_l) and np.array_equal(o2, exp_o)
    # the partial initialisation gives the same rows
    pO, pL = O.init_context_partial(T, H, D, P.empty_token_slices(g["context_lens"], g["query_lens"]))
    assert np.all(np.isneginf(pL[:, lo:hi])) and np.all(pO[lo:hi] == 0)
    assert np.isnan(pL[:, :lo]).all() and np.isnan(pO[hi:]).all()


# ---------------------------------------------------------- whole path ----
def _np_inputs(w):
    x = W.make_inputs(w)
    return {k: (v.double().numpy() if v.is_floating_point() else v.numpy()) for k, v in x.items()}


def _dims(w):
    return O.MlaDims(w.num_heads, w.kv_lora_rank, w.qk_rope_dim, w.qk_nope_dim, w.v_dim,
                     w.block_size, w.softmax_scale)


def sdpa_full_prefill(x, w):
    """Unchunked result for every (token, head) by torch SDPA over
    [whole context ; new tokens] with the causal mask on the new part."""
    d = _dims(w)
    qsl = P.query_start_loc(w.query_lens)
    T = qsl[-1]
    out = np.zeros((T, w.num_heads, w.v_dim))
    for r, (c, ql) in enumerate(zip(w.context_lens, w.query_lens)):
        if ql == 0:
            continue
        a = qsl[r]
        rows = np.array([O.context_row(x["kv_cache"], x["block_table"], r, j, w.block_size)
                         for j in range(c)]).reshape(c, w.latent_dim)
        lat = np.concatenate([rows, x["new_latent"][a:a + ql]], axis=0)
        kn, v = O.up_project(lat, x["w_kv_b"], d)
        vis = np.ones((ql, c + ql), dtype=bool)
        vis[:, c:] = np.tril(np.ones((ql, ql), dtype=bool))
        out[a:a + ql] = sdpa_reference(x["q"][a:a + ql], kn, lat[:, w.kv_lora_rank:], v,
                                       w.softmax_scale, vis)
    return out


@pytest.mark.parametrize("budget,align", [(128, 16), (48, 16), (1000, 1), (37, 1)])
def test_chunked_equals_unchunked_tiny(budget, align):
    w = W.scaled(W.workload("tiny"), row_budget=budget, split_alignment=align,
                 max_context_chunk=budget)
    x = _np_inputs(w)
    d = _dims(w)
    o, l, plans = O.chunked_prefill(x["q"], x["new_latent"], x["kv_cache"], x["block_table"],
                                    x["w_kv_b"], w.context_lens, w.query_lens, d,
                                    w.row_budget, w.max_context_chunk, w.split_alignment)
    assert not np.isnan(o).any() and not np.isnan(l).any()
    ou, lu = O.unchunked_prefill(x["q"], x["new_latent"], x["kv_cache"], x["block_table"],
                                 x["w_kv_b"], w.context_lens, w.query_lens, d)
    np.testing.assert_allclose(o, ou, atol=1e-11)
    np.testing.assert_allclose(l, lu, atol=1e-11)
    np.testing.assert_allclose(o, sdpa_full_prefill(x, w), atol=1e-11)


def test_chunked_random_shapes_match_sdpa():
    rng = np.random.default_rng(15)
    for trial in range(4):
        R = int(rng.integers(1, 5))
        ctx = [int(c) if rng.random() > 0.3 else 0 for c in rng.integers(1, 90, size=R)]
        ql = [int(x) for x in rng.integers(1, 7, size=R)]
        w = W.MlaWorkload("rand", ctx, ql, num_heads=2, kv_lora_rank=8, qk_rope_dim=4,
                          qk_nope_dim=4, v_dim=3, block_size=8, row_budget=int(rng.integers(8, 64)),
                          split_alignment=8, dtype="f32", seed=50 + trial, w_std=0.3)
        x = _np_inputs(w)
        o, l, _ = O.chunked_prefill(x["q"], x["new_latent"], x["kv_cache"], x["block_table"],
                                    x["w_kv_b"], w.context_lens, w.query_lens, _dims(w),
                                    w.row_budget, w.max_context_chunk, w.split_alignment)
        np.testing.assert_allclose(o, sdpa_full_prefill(x, w), atol=1e-11)


# ------------------------------------------------------ planted mistakes --
def test_pins_catch_planted_mistakes():
    """Each copy below carries one plausible mistake; some pin must fail."""
    def attn_no_rope(q, kn, kp, v, scale, visible=None):
        return O.attention_with_lse(q, kn, np.zeros_like(kp), v, scale, visible)

    def attn_wrong_sign(q, kn, kp, v, scale, visible=None):
        return O.attention_with_lse(q, kn, kp, v, -scale, visible)

    def attn_lse_no_max(q, kn, kp, v, scale, visible=None):
        o, l = O.attention_with_lse(q, kn, kp, v, scale, visible)
        s = scale * (np.einsum("mhd,nhd->hmn", q[:, :, :kn.shape[2]], kn)
                     + np.einsum("mhp,np->hmn", q[:, :, kn.shape[2]:], kp))
        return o, l - s.max(axis=2)          # dropped the running-max term

    def merge_swapped(pO, pL, sO, sL, n):
        return O.merge_attn_states(sO, pL, pO, sL, n)   # O paired with wrong LSE

    for bad in (attn_no_rope, attn_wrong_sign):
        with pytest.raises(AssertionError):
            check_attention_vs_sdpa(bad)
    with pytest.raises(AssertionError):
        check_split_keys_merge(attn_lse_no_max, O.merge_attn_states)
    with pytest.raises(AssertionError):
        check_split_keys_merge(O.attention_with_lse, merge_swapped)
    # a planner that appends an overflowing request whole breaks the budget
    def literal_reading(ctx, budget, mcc, a):
        plans = P.plan_mla_context_chunks(ctx, budget, mcc, a)
        if len(plans) >= 2 and plans[1].starts[0] == 0:
            plans[0].seq_lens.append(ctx[plans[1].request_start])
            plans[0].starts.append(0)
            plans[0].request_end += 1
            plans.pop(1)
        return plans
    with pytest.raises(AssertionError):
        check_plan_invariants([1020, 10], literal_reading([1020, 10], 1024, 1024, 16), 1024)


# ------------------------------------------- the old equal-window scheme --
def test_equal_window_plan_invariants():
    rng = np.random.default_rng(16)
    for _ in range(500):
        n = int(rng.integers(1, 10))
        ctx = [int(x) if rng.random() > 0.3 else 0 for x in rng.integers(1, 3000, size=n)]
        if not any(ctx):
            continue
        align = int(rng.choice([1, 16, 64]))
        budget = int(rng.integers(align * n, 8000))
        win, starts, lens, empty = P.plan_equal_window_chunks(ctx, budget, align)
        with_ctx = sum(1 for c in ctx if c > 0)
        assert win % align == 0 and win * with_ctx <= budget and win > 0
        assert len(starts) == -(-max(ctx) // win)
        for c in range(len(starts)):
            assert sum(lens[c]) <= budget
            assert empty[c] == any(x == 0 for x in lens[c])
        for r in range(n):          # every row exactly once, in window order
            covered = [(starts[c][r], lens[c][r]) for c in range(len(starts)) if lens[c][r]]
            pos = 0
            for s, l in covered:
                assert s == pos
                pos += l
            assert pos == ctx[r]
    w = W.workload("hetero")
    win, starts, _, _ = P.plan_equal_window_chunks(w.context_lens, w.row_budget,
                                                   w.split_alignment)
    assert win == 1280 and len(starts) == 103     # vs 11 chunks of per-request packing


def test_equal_window_prefill_equals_chunked():
    for budget in (128, 64):
        w = W.scaled(W.workload("tiny"), row_budget=budget, max_context_chunk=budget)
        x = _np_inputs(w)
        d = _dims(w)
        o1, l1, n1 = O.equal_window_prefill(x["q"], x["new_latent"], x["kv_cache"],
                                            x["block_table"], x["w_kv_b"], w.context_lens,
                                            w.query_lens, d, w.row_budget, w.split_alignment)
        o2, l2, _ = O.chunked_prefill(x["q"], x["new_latent"], x["kv_cache"], x["block_table"],
                                      x["w_kv_b"], w.context_lens, w.query_lens, d, w.row_budget,
                                      w.max_context_chunk, w.split_alignment)
        assert n1 > 1
        np.testing.assert_allclose(o1, o2, atol=1e-11)
        np.testing.assert_allclose(l1, l2, atol=1e-11)
        np.testing.assert_allclose(o1, sdpa_full_prefill(x, w), atol=1e-11)
