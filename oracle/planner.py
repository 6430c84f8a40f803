"""Oracle for the context-chunk planner and the per-chunk metadata.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: the PR #50613 report ("MLA prefill schedules chunks per request"),
section "implementation breakdown" item 2 and the key source snippet of
``mla_attention.py`` (``_ContextChunkPlan``, ``plan_mla_context_chunks``,
``aligned_split_len``), and the worked example in the test snippet
``test_tail_splitting_minimizes_chunks``.

What the planner does: walk the requests in order; requests without cached
context are skipped; every other request's context rows are packed into the
current chunk until the chunk's workspace row budget would overflow.  The
request that overflows is cut at the largest aligned length that still fits
(the rest of it opens the next chunk, which is then a "continuation"), and the
chunk is closed.

Readings taken where the page is silent or garbled:

* An overflowing request whose aligned split is empty (no aligned length fits
  in the rows left) closes the chunk without being appended; it opens the next
  chunk.  Appending it whole would break the page's invariant "a chunk does not
  exceed the workspace".  The worked example is the same under both readings.
* ``padded_rows`` defaults to the identity.
* The split search is written here as its plain definition (largest aligned
  length that fits, found by scanning); the page searches the same monotone
  predicate by bisection.  The two agree whenever ``padded_rows`` is
  non-decreasing, which every padding function is.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, Optional, Sequence


class PlannerStuck(ValueError):
    """A request cannot be placed: no aligned split fits an empty chunk."""


@dataclass
class ChunkPlan:
    """One chunk: a contiguous range of requests with context.

    ``starts[i]``/``seq_lens[i]`` are the offset into, and the number of rows
    of, the context of request ``request_start + i`` that this chunk covers.
    ``is_continuation`` is true when the chunk resumes a request that an
    earlier chunk began (PR #50613 report, key source snippet,
    ``_ContextChunkPlan``).
    """

    request_start: int
    request_end: int
    starts: list = field(default_factory=list)
    seq_lens: list = field(default_factory=list)
    is_continuation: bool = False


def _identity(x: int) -> int:
    return x


def aligned_split_len(start: int, remaining: int, available: int,
                      max_context_chunk: int, split_alignment: int,
                      padded_rows: Callable[[int], int] = _identity) -> int:
    """Largest multiple of ``split_alignment`` that may end a split here.

    The length is at most ``max_context_chunk``, strictly below
    ``remaining`` rounded down to the alignment (a split never takes the
    whole rest of the request; ``remaining - 1`` is rounded down), and the
    padded rows it adds, ``padded_rows(start + len) - padded_rows(start)``,
    must not exceed ``available``.  Returns 0 when no positive length fits.

    (PR #50613 report, key source snippet: ``aligned_split_len``.)
    """
    a = split_alignment
    cap = min(max_context_chunk, ((remaining - 1) // a) * a)
    best = 0
    k = 1
    while k * a <= cap:
        length = k * a
        if padded_rows(start + length) - padded_rows(start) <= available:
            best = length
        k += 1
    return best


def plan_mla_context_chunks(context_lens: Sequence[int], row_budget: int,
                            max_context_chunk: int, split_alignment: int,
                            padded_rows: Optional[Callable[[int], int]] = None
                            ) -> list:
    """Pack every request's context into chunks of at most ``row_budget`` rows.

    (PR #50613 report, "implementation breakdown" item 2 and the key source
    snippet ``plan_mla_context_chunks``.)
    """
    rows_of = padded_rows if padded_rows is not None else _identity
    lens = [int(x) for x in context_lens]
    plans = []
    n = len(lens)
    req = 0
    offset = 0          # rows of lens[req] already placed in earlier chunks
    while req < n:
        if lens[req] == 0:
            # Requests without context never enter a chunk.
            if offset != 0:
                raise PlannerStuck("zero-length request while mid-split")
            req += 1
            continue
        plan = ChunkPlan(request_start=req, request_end=req)
        used = 0
        while req < n and lens[req] > 0:
            left = lens[req] - offset
            need = rows_of(offset + left) - rows_of(offset)
            if used + need <= row_budget:
                plan.starts.append(offset)
                plan.seq_lens.append(left)
                used += need
                req += 1
                offset = 0
                continue
            cut = aligned_split_len(offset, left, row_budget - used,
                                    max_context_chunk, split_alignment, rows_of)
            if cut > 0:
                plan.starts.append(offset)
                plan.seq_lens.append(cut)
                used += rows_of(offset + cut) - rows_of(offset)
                offset += cut
            break  # the overflowing request always closes the chunk
        if not plan.seq_lens:
            raise PlannerStuck(
                f"request {req}: no aligned split of {lens[req] - offset} rows "
                f"fits a budget of {row_budget}")
        plan.request_end = plan.request_start + len(plan.seq_lens)
        plan.is_continuation = plan.starts[0] > 0
        plans.append(plan)
    return plans


@dataclass
class ChunkMeta:
    """Per-chunk arrays (PR #50613 report, item 2: cu_seq_lens, seq_lens,
    token_to_seq; the ContextChunk's request and token slices)."""

    plan: ChunkPlan
    cu_seq_lens: list        # workspace row offset of each request, plus total
    token_to_seq: list       # workspace row -> local request index
    token_slice: tuple       # [first, last) new-token index of the chunk
    max_seq_len: int


def query_start_loc(query_lens: Sequence[int]) -> list:
    out = [0]
    for x in query_lens:
        out.append(out[-1] + int(x))
    return out


def chunk_metadata(plan: ChunkPlan, query_lens: Sequence[int]) -> ChunkMeta:
    qsl = query_start_loc(query_lens)
    cu = [0]
    t2s = []
    for i, ln in enumerate(plan.seq_lens):
        cu.append(cu[-1] + ln)
        t2s.extend([i] * ln)
    return ChunkMeta(plan=plan, cu_seq_lens=cu, token_to_seq=t2s,
                     token_slice=(qsl[plan.request_start], qsl[plan.request_end]),
                     max_seq_len=max(plan.seq_lens))


def prefix_num_tokens(context_lens: Sequence[int],
                      query_lens: Sequence[int]) -> int:
    """Number of leading new tokens whose context partial must be merged.

    Reading of the PR #36540 report ("implementation breakdown", CUDA kernel
    layer and the business-logic layer): tokens of requests with context come
    first; tokens at or past this count copy the suffix output.  Here: the
    end of the last request that has context, 0 when none has.
    """
    qsl = query_start_loc(query_lens)
    last = -1
    for r, c in enumerate(context_lens):
        if c > 0:
            last = r
    return qsl[last + 1] if last >= 0 else 0


def empty_token_slices(context_lens: Sequence[int],
                       query_lens: Sequence[int]) -> list:
    """Token ranges below ``prefix_num_tokens`` owned by requests without
    context (PR #50613 report, item 1: ``empty_token_slices``)."""
    qsl = query_start_loc(query_lens)
    limit = prefix_num_tokens(context_lens, query_lens)
    out = []
    for r, c in enumerate(context_lens):
        lo, hi = qsl[r], min(qsl[r + 1], limit)
        if c == 0 and lo < hi:
            out.append((lo, hi))
    return out


# --------------------------------------------------------------------------
# the old scheme: equal context windows
# --------------------------------------------------------------------------
def plan_equal_window_chunks(context_lens: Sequence[int], row_budget: int,
                             split_alignment: int):
    """The scheme the per-request packing replaced (PR #50613 report,
    "motivation": the workspace was divided evenly among the requests with
    context and every iteration processed the same context window of every
    request; PR #49294 report, snippet of build_mla_chunked_context_metadata:
    per chunk a row of starts/ends over the requests, seq_lens =
    clamp(ends - starts, 0), has_empty_context = any(seq_lens == 0)).

    Reading: window = budget // (requests with context), rounded down to the
    split alignment; chunk c covers context rows [c*window, (c+1)*window) of
    every request, clipped to its length.  Returns (window, starts, seq_lens,
    has_empty_context) with starts / seq_lens as lists of per-request lists.
    """
    lens = [int(x) for x in context_lens]
    with_ctx = sum(1 for c in lens if c > 0)
    if with_ctx == 0:
        return 0, [], [], []
    window = (row_budget // with_ctx) // split_alignment * split_alignment
    if window <= 0:
        raise PlannerStuck("budget below one aligned window per request")
    n_chunks = -(-max(lens) // window)
    starts, seq_lens, empty = [], [], []
    for c in range(n_chunks):
        st = [min(c * window, x) for x in lens]
        en = [min((c + 1) * window, x) for x in lens]
        sl = [max(e - s, 0) for s, e in zip(st, en)]
        starts.append(st)
        seq_lens.append(sl)
        empty.append(any(x == 0 for x in sl))
    return window, starts, seq_lens, empty
