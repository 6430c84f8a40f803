"""Oracle for the MLA chunked-context prefill arithmetic, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources
-------
* Gather: PR #50613 report, item 2 -- every context row of a chunk is gathered
  exactly once into the workspace, at the row offsets ``cu_seq_lens``.
* Partial lifecycle: PR #50613 report, item 3 -- ``init_mla_context_partial``
  gives rows of context-free requests (O=0, LSE=-inf);
  ``accumulate_mla_context_chunk`` merges each chunk into the partial.
* Empty-context rows: PR #49294 report ("Ignore empty MLA context chunks
  during merge"), motivation and the snippet ``test_mask_empty_context``:
  such rows read LSE=-inf and O=0.
* Merge with ``prefix_num_tokens``: PR #36540 report ("Remove trtllm ragged
  mla prefills"), "implementation breakdown", CUDA kernel layer: tokens at or
  past the threshold copy the suffix, the others merge prefix and suffix.
* The MLA arithmetic itself (latent cache, W_kv_b up-projection into K_nope
  and V, attention over concat(K_nope, k_pe), causal new-token attention) is
  not written on the pages; the plainest reading is used:
  cache row = [c_kv (kv_lora_rank) | k_pe (qk_rope_dim)], W_kv_b is
  [H*(Dn+Dv), kv_lora_rank] with head h's rows [h*(Dn+Dv), h*(Dn+Dv)+Dn)
  giving K_nope and the next Dv rows giving V; q = [q_nope | q_pe]; natural
  log LSE.

Layouts follow the pages' merge test: O is [tokens, heads, dim] and LSE is
head-major [heads, tokens].
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Sequence

import numpy as np

from . import planner as _planner

NEG_INF = -np.inf


@dataclass
class MlaDims:
    num_heads: int
    kv_lora_rank: int
    qk_rope_dim: int
    qk_nope_dim: int
    v_dim: int
    block_size: int
    softmax_scale: float


# --------------------------------------------------------------------------
# gather
# --------------------------------------------------------------------------
def context_row(cache, block_table, request: int, j: int, block_size: int):
    """Row ``j`` of request ``request``'s cached context: slot ``j % bs`` of
    the physical block ``block_table[request][j // bs]``."""
    return cache[int(block_table[request][j // block_size]), j % block_size]


def gather_chunk(cache, block_table, plan, block_size: int):
    """Copy every context row a chunk covers into a dense workspace, request
    after request, at the offsets ``cu_seq_lens`` (PR #50613 report, item 2).
    Returns float64 [rows, L+P]."""
    total = sum(plan.seq_lens)
    ws = np.empty((total, cache.shape[2]), dtype=np.float64)
    row = 0
    for i, req in enumerate(range(plan.request_start, plan.request_end)):
        for j in range(plan.starts[i], plan.starts[i] + plan.seq_lens[i]):
            ws[row] = context_row(cache, block_table, req, j, block_size)
            row += 1
    return ws


# --------------------------------------------------------------------------
# up-projection
# --------------------------------------------------------------------------
def up_project(latent, w_kv_b, dims: MlaDims):
    """K_nope, V = split(latent[:, :L] @ W_kv_b^T) per head.

    latent [n, >=L]; w_kv_b [H*(Dn+Dv), L].  Returns K_nope [n, H, Dn] and
    V [n, H, Dv] in float64.
    """
    L, H = dims.kv_lora_rank, dims.num_heads
    Dn, Dv = dims.qk_nope_dim, dims.v_dim
    c = np.asarray(latent, dtype=np.float64)[:, :L]
    w = np.asarray(w_kv_b, dtype=np.float64)
    kv = (c @ w.T).reshape(c.shape[0], H, Dn + Dv)
    return kv[:, :, :Dn], kv[:, :, Dn:]


# --------------------------------------------------------------------------
# attention with LSE
# --------------------------------------------------------------------------
def attention_with_lse(q, k_nope, k_pe, v, scale: float, visible=None):
    """Softmax attention of every query row and head over a key set.

    q [m, H, Dn+P]; k_nope [n, H, Dn]; k_pe [n, P] (shared by all heads);
    v [n, H, Dv]; ``visible`` optional bool [m, n] (True = key visible).
    score s = scale * (q_nope . k_nope + q_pe . k_pe); LSE = ln sum exp(s);
    O = sum exp(s - LSE) v.  A row that sees no key gets O = 0 and
    LSE = -inf.  Returns O [m, H, Dv], LSE [H, m].
    """
    q = np.asarray(q, dtype=np.float64)
    k_nope = np.asarray(k_nope, dtype=np.float64)
    k_pe = np.asarray(k_pe, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m, H, _ = q.shape
    n, Dn, Dv = k_nope.shape[0], k_nope.shape[2], v.shape[2]
    if n == 0:
        return np.zeros((m, H, Dv)), np.full((H, m), NEG_INF)
    # (einsum with optimize=True contracts through BLAS: the same float64
    # sums as numpy's own loops, in another order)
    s = np.einsum("mhd,nhd->hmn", q[:, :, :Dn], k_nope, optimize=True)
    s = s + np.einsum("mhp,np->hmn", q[:, :, Dn:], k_pe, optimize=True)
    s = s * scale
    if visible is not None:
        s = np.where(np.asarray(visible, dtype=bool)[None, :, :], s, NEG_INF)
    mx = s.max(axis=2)                                   # [H, m]
    seen = np.isfinite(mx)
    safe_mx = np.where(seen, mx, 0.0)
    e = np.exp(s - safe_mx[:, :, None])                  # exp(-inf) = 0
    tot = e.sum(axis=2)
    lse = np.where(seen, safe_mx + np.log(np.where(seen, tot, 1.0)), NEG_INF)
    p = np.where(seen[:, :, None], e / np.where(seen, tot, 1.0)[:, :, None], 0.0)
    o = np.einsum("hmn,nhd->mhd", p, v, optimize=True)
    return o, lse


# --------------------------------------------------------------------------
# merge
# --------------------------------------------------------------------------
def merge_attn_states(prefix_o, prefix_lse, suffix_o, suffix_lse,
                      prefix_num_tokens: int):
    """LSE-weighted merge of two partial attention results.

    O [T, H, D], LSE [H, T].  Per (token t, head h):
      t >= prefix_num_tokens  -> the suffix (O, LSE) as is;
      both LSE = -inf         -> O = 0, LSE = -inf;
      one LSE = -inf          -> the other side as is;
      both finite             -> m = max; a = e^(pL-m), b = e^(sL-m);
                                 O = (a pO + b sO)/(a+b); LSE = m + ln(a+b).
    A side that is not needed is never read into arithmetic (it may hold
    garbage or NaN): the cases are selected, not weighted by zero.
    """
    pO = np.asarray(prefix_o, dtype=np.float64)
    sO = np.asarray(suffix_o, dtype=np.float64)
    pL = np.asarray(prefix_lse, dtype=np.float64)
    sL = np.asarray(suffix_lse, dtype=np.float64)
    T, H, D = sO.shape
    out = np.zeros((T, H, D))
    out_lse = np.full((H, T), NEG_INF)
    tok = np.arange(T)[None, :].repeat(H, axis=0)          # [H, T]
    passthru = tok >= prefix_num_tokens
    below = ~passthru
    p_empty = np.zeros((H, T), dtype=bool)
    s_empty = np.isneginf(sL)
    p_empty[below] = np.isneginf(pL[below])
    take_s = passthru | (below & p_empty & ~s_empty)
    take_p = below & ~p_empty & s_empty
    both = below & ~p_empty & ~s_empty
    # (both empty below the threshold keeps the zero / -inf initialisation)
    hs, ts = np.nonzero(take_s)
    out[ts, hs] = sO[ts, hs]
    out_lse[hs, ts] = sL[hs, ts]
    hp, tp = np.nonzero(take_p)
    out[tp, hp] = pO[tp, hp]
    out_lse[hp, tp] = pL[hp, tp]
    hb, tb = np.nonzero(both)
    if hb.size:
        a_l, b_l = pL[hb, tb], sL[hb, tb]
        mx = np.maximum(a_l, b_l)
        a = np.exp(a_l - mx)
        b = np.exp(b_l - mx)
        out[tb, hb] = (a[:, None] * pO[tb, hb] + b[:, None] * sO[tb, hb]) \
            / (a + b)[:, None]
        out_lse[hb, tb] = mx + np.log(a + b)
    return out, out_lse


# --------------------------------------------------------------------------
# empty-context rows
# --------------------------------------------------------------------------
def mask_empty_context(lse, out, query_start_loc, context_start_loc):
    """Old-scheme fix-up (PR #49294 report, snippet of
    ``test_mask_empty_context``): rows of every request whose context length
    in this chunk (difference of ``context_start_loc``) is 0 get LSE = -inf
    and O = 0; other rows are left as they are.  Works in place on copies and
    returns (lse, out)."""
    lse = np.array(lse, dtype=np.float64, copy=True)
    out = np.array(out, dtype=np.float64, copy=True)
    R = len(query_start_loc) - 1
    for r in range(R):
        if context_start_loc[r + 1] - context_start_loc[r] == 0:
            lo, hi = int(query_start_loc[r]), int(query_start_loc[r + 1])
            lse[:, lo:hi] = NEG_INF
            out[lo:hi] = 0.0
    return lse, out


def init_context_partial(num_tokens: int, num_heads: int, v_dim: int,
                         empty_slices):
    """Fresh context partial (PR #50613 report, item 3,
    ``init_mla_context_partial``): rows of context-free requests (the given
    token slices) read O = 0, LSE = -inf; every other row is undefined (NaN
    here, so that any read of it shows)."""
    O = np.full((num_tokens, num_heads, v_dim), np.nan)
    L = np.full((num_heads, num_tokens), np.nan)
    for lo, hi in empty_slices:
        O[lo:hi] = 0.0
        L[:, lo:hi] = NEG_INF
    return O, L


# --------------------------------------------------------------------------
# the whole path
# --------------------------------------------------------------------------
def _causal(m: int):
    return np.tril(np.ones((m, m), dtype=bool))


def suffix_attention(q, new_latent, w_kv_b, query_lens, dims: MlaDims):
    """New-token attention: token i of a request sees the request's new
    tokens 0..i.  Keys and values come from up-projecting the new tokens'
    latent rows with the same W_kv_b; their k_pe is the latent tail."""
    L = dims.kv_lora_rank
    lat = np.asarray(new_latent, dtype=np.float64)
    k_nope, v = up_project(lat, w_kv_b, dims)
    k_pe = lat[:, L:]
    qsl = _planner.query_start_loc(query_lens)
    T = qsl[-1]
    O = np.zeros((T, dims.num_heads, dims.v_dim))
    LSE = np.full((dims.num_heads, T), NEG_INF)
    for r in range(len(query_lens)):
        a, b = qsl[r], qsl[r + 1]
        if a == b:
            continue
        O[a:b], LSE[:, a:b] = attention_with_lse(
            q[a:b], k_nope[a:b], k_pe[a:b], v[a:b], dims.softmax_scale,
            visible=_causal(b - a))
    return O, LSE


def chunked_prefill(q, new_latent, cache, block_table, w_kv_b,
                    context_lens: Sequence[int], query_lens: Sequence[int],
                    dims: MlaDims, row_budget: int, max_context_chunk: int,
                    split_alignment: int):
    """MLA chunked-context prefill, step by step as the pages order it.

    1. plan the chunks (PR #50613 report, item 2);
    2. init the context partial (item 3);
    3. per chunk: gather the rows, up-project them, attend each request's
       queries to its rows in the chunk, accumulate into the partial
       (a merge only where the chunk continues a request);
    4. causal new-token (suffix) attention;
    5. final merge with ``prefix_num_tokens`` (PR #36540 report).

    Returns (O [T, H, Dv], LSE [H, T], plans).
    """
    L = dims.kv_lora_rank
    plans = _planner.plan_mla_context_chunks(
        context_lens, row_budget, max_context_chunk, split_alignment)
    qsl = _planner.query_start_loc(query_lens)
    T = qsl[-1]
    pnt = _planner.prefix_num_tokens(context_lens, query_lens)
    pO, pL = init_context_partial(
        T, dims.num_heads, dims.v_dim,
        _planner.empty_token_slices(context_lens, query_lens))
    q = np.asarray(q, dtype=np.float64)
    for plan in plans:
        meta = _planner.chunk_metadata(plan, query_lens)
        ws = gather_chunk(cache, block_table, plan, dims.block_size)
        k_nope, v = up_project(ws, w_kv_b, dims)
        k_pe = ws[:, L:]
        for i, req in enumerate(range(plan.request_start, plan.request_end)):
            a, b = qsl[req], qsl[req + 1]
            if a == b:
                continue
            r0, r1 = meta.cu_seq_lens[i], meta.cu_seq_lens[i + 1]
            o, lse = attention_with_lse(q[a:b], k_nope[r0:r1], k_pe[r0:r1],
                                        v[r0:r1], dims.softmax_scale)
            if plan.starts[i] > 0:      # an earlier chunk began this request
                o, lse = merge_attn_states(pO[a:b], pL[:, a:b], o, lse, b - a)
            pO[a:b], pL[:, a:b] = o, lse
    sO, sL = suffix_attention(q, new_latent, w_kv_b, query_lens, dims)
    out, out_lse = merge_attn_states(pO, pL, sO, sL, pnt)
    return out, out_lse, plans


def unchunked_rows(q, new_latent, cache, block_table, w_kv_b,
                   context_lens: Sequence[int], query_lens: Sequence[int],
                   dims: MlaDims, tokens: Sequence[int], heads: Sequence[int]):
    """Reference without chunks, for chosen (token, head) pairs: one softmax
    over the request's whole cached context followed by its new tokens up to
    and including the token itself.  Returns O [k, Dv], LSE [k]."""
    L, H = dims.kv_lora_rank, dims.num_heads
    Dn, Dv = dims.qk_nope_dim, dims.v_dim
    qsl = _planner.query_start_loc(query_lens)
    q = np.asarray(q)
    lat_new = np.asarray(new_latent, dtype=np.float64)
    w = np.asarray(w_kv_b, dtype=np.float64)
    req_of = np.searchsorted(np.asarray(qsl), np.asarray(tokens), side="right") - 1
    out_o = np.zeros((len(tokens), Dv))
    out_l = np.zeros(len(tokens))
    groups = {}
    for k, (t, h) in enumerate(zip(tokens, heads)):
        groups.setdefault((int(req_of[k]), int(h)), []).append(k)
    for (r, h), ks in groups.items():
        c = int(context_lens[r])
        a = qsl[r]
        rows = np.empty((c, cache.shape[2]), dtype=np.float64)
        for j in range(c):
            rows[j] = context_row(cache, block_table, r, j, dims.block_size)
        last = max(int(tokens[k]) for k in ks)
        keys_lat = np.concatenate([rows, lat_new[a:last + 1]], axis=0)
        wh = w[h * (Dn + Dv):(h + 1) * (Dn + Dv)]
        kv = keys_lat[:, :L] @ wh.T
        kn, vv, kp = kv[:, :Dn], kv[:, Dn:], keys_lat[:, L:]
        for k in ks:
            t = int(tokens[k])
            n = c + (t - a) + 1
            qv = np.asarray(q[t, h], dtype=np.float64)
            s = dims.softmax_scale * (kn[:n] @ qv[:Dn] + kp[:n] @ qv[Dn:])
            mx = s.max()
            e = np.exp(s - mx)
            out_l[k] = mx + math.log(e.sum())
            out_o[k] = (e / e.sum()) @ vv[:n]
    return out_o, out_l


def unchunked_prefill(q, new_latent, cache, block_table, w_kv_b,
                      context_lens, query_lens, dims: MlaDims):
    """Unchunked reference for every (token, head)."""
    T = int(sum(query_lens))
    H = dims.num_heads
    toks = np.repeat(np.arange(T), H)
    hs = np.tile(np.arange(H), T)
    o, l = unchunked_rows(q, new_latent, cache, block_table, w_kv_b,
                          context_lens, query_lens, dims, toks, hs)
    return o.reshape(T, H, dims.v_dim), l.reshape(T, H).T.copy()


def equal_window_prefill(q, new_latent, cache, block_table, w_kv_b,
                         context_lens: Sequence[int], query_lens: Sequence[int],
                         dims: MlaDims, row_budget: int, split_alignment: int):
    """The old scheme end to end (PR #49294 report: per chunk, attention over
    the whole prefill batch's windows, then mask_empty_context on requests
    whose window is empty, then a merge into the running result; PR #36540
    report: the final merge with the new-token attention).  Same result as
    chunked_prefill up to rounding.  Returns (O, LSE, number of chunks)."""
    L = dims.kv_lora_rank
    window, starts, seq_lens, _ = _planner.plan_equal_window_chunks(
        context_lens, row_budget, split_alignment)
    qsl = _planner.query_start_loc(query_lens)
    T = qsl[-1]
    R = len(context_lens)
    q = np.asarray(q, dtype=np.float64)
    pO = np.zeros((T, dims.num_heads, dims.v_dim))
    pL = np.full((dims.num_heads, T), NEG_INF)
    for c in range(len(starts)):
        cO = np.full((T, dims.num_heads, dims.v_dim), np.nan)   # rows a backend leaves
        cL = np.full((dims.num_heads, T), np.nan)
        for r in range(R):
            a, b = qsl[r], qsl[r + 1]
            n = seq_lens[c][r]
            if a == b or n == 0:
                continue
            rows = np.array([context_row(cache, block_table, r, j, dims.block_size)
                             for j in range(starts[c][r], starts[c][r] + n)],
                            dtype=np.float64).reshape(n, -1)
            k_nope, v = up_project(rows, w_kv_b, dims)
            cO[a:b], cL[:, a:b] = attention_with_lse(q[a:b], k_nope, rows[:, L:], v,
                                                     dims.softmax_scale)
        csl = [0]
        for r in range(R):
            csl.append(csl[-1] + seq_lens[c][r])
        cL, cO = mask_empty_context(cL, cO, qsl, csl)
        pO, pL = merge_attn_states(pO, pL, cO, cL, T)
    sO, sL = suffix_attention(q, new_latent, w_kv_b, query_lens, dims)
    pnt = _planner.prefix_num_tokens(context_lens, query_lens)
    out, out_lse = merge_attn_states(pO, pL, sO, sL, pnt)
    return out, out_lse, len(starts)
