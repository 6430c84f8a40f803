#!/usr/bin/env python
"""Benchmark of MLA chunked-context prefill on one or more GB300s.

One step = one call of mla_chunked_prefill (plan, metadata upload, empty-row
fill, per chunk gather + W_kv_b up-projection + attention + accumulate,
new-token up-projection + causal attention, final merge_attn_states) over the
heterogeneous batch: 32 requests, one context of 131072 rows, 24 log-uniform
on [1, 2048], 7 empty; queries uniform on [1, 256]; DeepSeek-V3 MLA shapes
(128 heads, latent 512 + rope 64, nope 128, v 128, bf16, block 64);
workspace 32768 rows, split alignment 64.  All inputs are seeded synthetic.

Printed JSON line (rank 0):
  value      tokens/s of the whole job, inputs resident in HBM
  e2e        tokens/s with host buffers: pinned host->device copies of the
             step's inputs and a device->host read of the output inside the
             timed region
  breakdown  every launch of the timed steps timed in place (the library's
             per-launch CUDA events on the launching streams), summed per step
             of the method; the tensor-target bar = (up-projection + context
             attention FLOPs) / (span of the gather .. context attention)
  rooflines  per kernel: algorithmic work / its in-step CUDA-event time vs the
             measured peak, from a third timed region with the pipeline's
             overlap off (each kernel alone inside real steps); roofline =
             the one with the largest share of that region's kernel time;
             rooflines_overlapped: the same from the overlapped region
  configs    the other workloads (tiny, uniform, long) through the same call
  merge      merge_attn_states alone on 8192 tokens x 128 heads x 128 (bf16,
             15% empty prefix rows, prefix_num_tokens 6144): GB/s of the bytes
             that must move and the fraction of the measured HBM copy peak
  cpu_baseline  the float64 oracle on the host cores, on a bounded sample
             (every token, a few heads; throughput scaled to all heads)

--impl reference times the oracle alone (the slow reference arm).
Multi-GPU (torchrun): every rank runs its own replica of the batch (the path
has no exchange step); value = all ranks' tokens / max over ranks of time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "chunked-context MLA prefill tok/s; merge_attn_states GB/s (% HBM peak)"
L2_FLUSH_BYTES = 256 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.idx)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l for ts, l in self.lines if self.t0 is None or (self.t0 - 0.15 <= ts <= self.t1 + 0.15)]
        if not rows:
            rows = [l for _, l in self.lines]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- workloads --
def flops_of(w, plans):
    """Algorithmic FLOPs of one prefill (each multiply-add = 2): the
    up-projection of every context row and new token, the context attention
    over every (query, context row) pair and the causal new-token attention."""
    H, L, Dn, Dv, P = w.num_heads, w.kv_lora_rank, w.qk_nope_dim, w.v_dim, w.qk_rope_dim
    ctx_rows = sum(sum(p.seq_lens) for p in plans)
    T = w.num_tokens
    up = 2.0 * L * H * (Dn + Dv) * (ctx_rows + T)
    attn_ctx = 2.0 * H * (Dn + P + Dv) * sum(q * c for q, c in zip(w.query_lens, w.context_lens))
    attn_suf = 2.0 * H * (Dn + P + Dv) * sum(q * (q + 1) / 2 for q in w.query_lens)
    return dict(up_proj_ctx=2.0 * L * H * (Dn + Dv) * ctx_rows,
                up_proj_new=2.0 * L * H * (Dn + Dv) * T, attn_ctx=attn_ctx, attn_new=attn_suf,
                total=up + attn_ctx + attn_suf, context_rows=ctx_rows,
                attn_ctx_bytes=attn_ctx_bytes(w, plans), attn_new_bytes=attn_new_bytes(w))


def attn_new_bytes(w):
    """Bytes the new-token attention (with the final merge in its epilogue)
    must move per prefill: every new token's queries and its fp16 K_nope / V
    (every head) and bf16 k_pe, the float32 context partial of the tokens
    whose request has context (O and LSE), and the output (O in the storage
    type, LSE)."""
    H, Dn, Dv, P = w.num_heads, w.qk_nope_dim, w.v_dim, w.qk_rope_dim
    es = 2 if w.dtype == "bf16" else 4
    T = w.num_tokens
    with_ctx = sum(q for q, c in zip(w.query_lens, w.context_lens) if c > 0)
    return (T * H * (Dn + P) * 2 + T * (H * (Dn + Dv) * 2 + P * 2)
            + with_ctx * H * (Dv + 1) * 4 + T * H * (Dv * es + 4))


def attn_ctx_bytes(w, plans):
    """Bytes the context attention kernel must move per prefill: every
    context row's fp16 K_nope and V for every head and its bf16 k_pe (once),
    each chunk's queries of its requests (q_nope fp16 + q_pe bf16), and the
    float32 partial (O and LSE) written -- and read back where the request
    continues from an earlier chunk."""
    H, Dn, Dv, P = w.num_heads, w.qk_nope_dim, w.v_dim, w.qk_rope_dim
    b = 0.0
    for p in plans:
        rows = sum(p.seq_lens)
        b += rows * (H * (Dn + Dv) * 2 + P * 2)
        for i, r in enumerate(range(p.request_start, p.request_end)):
            q = w.query_lens[r]
            part = q * H * (Dv + 1) * 4
            b += q * H * (Dn + P) * 2 + part * (2 if p.starts[i] > 0 else 1)
    return b


def execution_groups(plans, budget):
    """The chunks as mla_chunked_prefill runs them: consecutive chunks with
    no continuation after the first and rows within the budget together."""
    rows_of = lambda c: sum(c.seq_lens)  # noqa: E731  (no padding here)
    groups, c0 = [], 0
    while c0 < len(plans):
        c1, rows = c0 + 1, rows_of(plans[c0])
        while (c1 < len(plans) and not plans[c1].is_continuation
               and rows + rows_of(plans[c1]) <= budget):
            rows += rows_of(plans[c1])
            c1 += 1
        groups.append(plans[c0:c1])
        c0 = c1
    return groups


def last_group_work(w, plans):
    """FLOPs and bytes of the final launch that attends the last execution
    group's context rows and the new tokens at once (when the prefill runs
    it that way): the new-token attention's work plus the last group's
    context attention, with queries read once, no partial written for the
    last group and the partial read only for tokens whose request has
    context in an earlier group; and the context attention of the other
    groups (FLOPs, bytes)."""
    H, Dn, Dv, P = w.num_heads, w.qk_nope_dim, w.v_dim, w.qk_rope_dim
    es = 2 if w.dtype == "bf16" else 4
    groups = execution_groups(plans, w.row_budget)
    last = groups[-1] if groups else []
    rest = [c for g in groups[:-1] for c in g]
    per_pair = 2.0 * H * (Dn + P + Dv)
    ctx_flops = lambda cs: per_pair * sum(  # noqa: E731
        w.query_lens[r] * c.seq_lens[i] for c in cs
        for i, r in enumerate(range(c.request_start, c.request_end)))
    last_rows = sum(sum(c.seq_lens) for c in last)
    earlier = set(r for c in rest for r, n in zip(range(c.request_start, c.request_end),
                                                   c.seq_lens) if n > 0)
    for c in last:  # a request continued into the last group has an earlier partial
        if c.is_continuation:
            earlier.add(c.request_start)
    T = w.num_tokens
    merge_tokens = sum(w.query_lens[r] for r in earlier)
    fl_last = per_pair * sum(q * (q + 1) / 2 for q in w.query_lens) + ctx_flops(last)
    by_last = (T * H * (Dn + P) * 2 + (T + last_rows) * (H * (Dn + Dv) * 2 + P * 2)
               + merge_tokens * H * (Dv + 1) * 4 + T * H * (Dv * es + 4))
    return fl_last, by_last, ctx_flops(rest), attn_ctx_bytes(w, rest)


def config_of(w, plans, world):
    """The workload description both arms print."""
    return {"workload": f"{w.name}: {w.num_requests} requests, context rows "
                        f"{sum(w.context_lens)} (max {max(w.context_lens)}), "
                        f"{w.num_tokens} new tokens, {len(plans)} chunks",
            "heads": w.num_heads, "kv_lora_rank": w.kv_lora_rank, "rope": w.qk_rope_dim,
            "nope": w.qk_nope_dim, "v": w.v_dim, "block_size": w.block_size,
            "row_budget": w.row_budget, "split_alignment": w.split_alignment,
            "chunks": len(plans), "storage": w.dtype, "parallelism": f"replicas x{world}",
            "l2": "flushed between timed steps (256 MB write outside the events)"}


def merge_bytes(x, T, H, D, es=2):
    """Bytes the merge must move: both LSEs of every row below the threshold,
    each finite side's O, the output O and LSE; above it the suffix only."""
    pnt = x["prefix_num_tokens"]
    pl = x["prefix_lse"][:, :pnt]
    sl = x["suffix_lse"][:, :pnt]
    pf = torch.isfinite(pl).sum().item()
    sf = torch.isfinite(sl).sum().item()
    below = H * pnt
    above = H * (T - pnt)
    b = below * 8 + (pf + sf) * D * es + below * (D * es + 4)
    b += above * (4 + D * es + D * es + 4)
    full = T * H * (3 * D * es + 12)
    return b, full


# ------------------------------------------------------- multi-rank glue ---
def job_time_ms(local_ms: float, world: int, device) -> float:
    """The job's time: the maximum over ranks of each rank's timed region
    (every rank runs its own replica of the batch; no data-path exchange)."""
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.item()


def whole_job_rate(units_per_rank_step: float, world: int, steps: int, job_ms: float) -> float:
    """Units all ranks processed per second of job time (weak scaling)."""
    return world * steps * units_per_rank_step / (job_ms / 1e3)


# ------------------------------------------------- in-step launch profile --
ROLE_GATHER, ROLE_UP, ROLE_ATTN = "a4 gather", "a5 up-projection", "a6-a7 context attention"
ROLE_UP_NEW, ROLE_ATTN_NEW = "a8 new-token up-projection", "a9-a10 new-token attention + merge"
# the last group's context attention and the new-token attention as one launch
ROLE_LAST = "a6-a10 last context group + new tokens"


def split_steps(records, steps):
    """The per-launch records of `steps` identical steps, one list per step
    (every step enqueues the same launches in the same order)."""
    n = len(records)
    if steps < 1 or n % steps:
        raise RuntimeError(f"{n} launch records do not split into {steps} steps")
    k = n // steps
    return [records[i * k:(i + 1) * k] for i in range(steps)]


def attributed_ms(rs):
    """Wall time of one step's launches with overlap shared out: every
    instant is split equally among the launches running then, so the shares
    add up to the time the GPU ran any of them (per role)."""
    pts = sorted({p for r in rs for p in (r[2], r[2] + r[3])})
    out = {}
    for a, b in zip(pts, pts[1:]):
        live = [r for r in rs if r[2] <= a and r[2] + r[3] >= b]
        for r in live:
            out[r[4]] = out.get(r[4], 0.0) + (b - a) / len(live)
    return out


def breakdown_of(records, steps, w, plans, peaks):
    """Per step of the method: launches, summed in-place CUDA-event time and
    overlap-attributed time per prefill step; per kernel: its rooflines; the
    tensor-target bar: (a5 + a6 FLOPs) / (span from the first gather's start to
    the end of the last context-attention launch)."""
    per_step = split_steps(records, steps)
    fl = flops_of(w, plans)
    roles, kernels = {}, {}
    spans = []
    attributed = {}
    for rs in per_step:
        for role, ms in attributed_ms(rs).items():
            attributed[role or "(other)"] = attributed.get(role or "(other)", 0.0) + ms / steps
        # the span ends with the last context attention (in the final launch
        # when the last group's attention runs there: the span then also
        # holds the new-token attention, which only lowers the bar)
        ctx = [r for r in rs if r[4] in (ROLE_GATHER, ROLE_UP, ROLE_ATTN, ROLE_LAST)]
        if ctx:
            t0 = min(r[2] for r in ctx)
            ends = [r[2] + r[3] for r in ctx if r[4] in (ROLE_ATTN, ROLE_LAST)]
            t1 = max(ends) if ends else max(r[2] + r[3] for r in ctx)
            spans.append(t1 - t0)
        for name, stream, start, ms, role in rs:
            e = roles.setdefault(role or "(other)", {"launches": 0, "ms": 0.0, "kernels": set()})
            e["launches"] += 1
            e["ms"] += ms
            e["kernels"].add(name)
            k = kernels.setdefault(name, {"launches": 0, "ms": 0.0})
            k["launches"] += 1
            k["ms"] += ms
    for name, e in roles.items():
        e["launches"] /= steps
        e["ms"] /= steps
        e["kernels"] = sorted(e["kernels"])
        e["attributed_ms"] = attributed.get(name, 0.0)
    for k in kernels.values():
        k["launches"] /= steps
        k["ms"] /= steps
    span_ms = statistics.median(spans) if spans else None
    es = 2 if w.dtype == "bf16" else 4
    row_bytes = (w.kv_lora_rank + w.qk_rope_dim) * es

    def rl(ms, work, launches, unit, peak, peak_src, bound, share):
        if not ms or not launches:
            return None
        sc = 1e12 if unit == "TFLOP/s" else 1e9
        ach = work / (ms / 1e3) / sc
        return {"bound": bound, "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak,
                "peak_source": peak_src, "launches_per_step": launches,
                "ms_per_step": ms, "attributed_ms_per_step": share, "work_per_step": work}
    def attn_rl(ms, launches, share, flops, nbytes):
        # tensor- or HBM-bound by which lower bound on the time is larger:
        # FLOPs at the bf16 peak, or the bytes the kernel must move at the
        # copy bandwidth (a chunk of few queries over many context rows is
        # bound by its K/V reads; so is attention over short causal windows)
        t_tc = flops / (bf * 1e12)
        t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
        if t_hbm > t_tc:
            r = rl(ms, nbytes, launches, "GB/s", peaks["hbm_gbs"], src + " copy", "hbm", share)
        else:
            r = rl(ms, flops, launches, "TFLOP/s", bf, src + " bf16 burst", "tensor", share)
        if r is not None:
            r["flops_per_step"] = flops
            r["bytes_per_step"] = nbytes
            r["bound_basis"] = ("max(FLOPs / bf16 peak, q + K/V + k_pe + partial + output bytes "
                                "/ copy bandwidth): t_tensor %.3f ms, t_hbm %.3f ms" %
                                (t_tc * 1e3, t_hbm * 1e3))
        return r
    g = roles.get(ROLE_UP, {"ms": 0, "launches": 0})
    gn = roles.get(ROLE_UP_NEW, {"ms": 0, "launches": 0})
    a = roles.get(ROLE_ATTN, {"ms": 0, "launches": 0})
    an = roles.get(ROLE_ATTN_NEW, {"ms": 0, "launches": 0})
    al = roles.get(ROLE_LAST, {"ms": 0, "launches": 0})
    ga = roles.get(ROLE_GATHER, {"ms": 0, "launches": 0})
    ctx_fl, ctx_by = fl["attn_ctx"], fl["attn_ctx_bytes"]
    if al["launches"]:
        last_fl, last_by, ctx_fl, ctx_by = last_group_work(w, plans)
    bf = peaks["bf16_tflops"]
    src = peaks["source"]
    at = lambda *rs: sum(attributed.get(r, 0.0) for r in rs)  # noqa: E731
    rooflines = {
        "up_proj": rl(g["ms"] + gn["ms"], fl["up_proj_ctx"] + fl["up_proj_new"],
                      g["launches"] + gn["launches"], "TFLOP/s", bf, src + " bf16 burst",
                      "tensor", at(ROLE_UP, ROLE_UP_NEW)),
        "context_attention": attn_rl(a["ms"], a["launches"], at(ROLE_ATTN), ctx_fl, ctx_by),
        "new_token_attention_merge": attn_rl(an["ms"], an["launches"], at(ROLE_ATTN_NEW),
                                             fl["attn_new"], fl["attn_new_bytes"]),
        "last_group_and_new_token_attention": (
            attn_rl(al["ms"], al["launches"], at(ROLE_LAST), last_fl, last_by)
            if al["launches"] else None),
        "gather": rl(ga["ms"], 2.0 * fl["context_rows"] * row_bytes, ga["launches"], "GB/s",
                     peaks["hbm_gbs"], src + " copy", "hbm", at(ROLE_GATHER)),
    }
    rooflines = {k: v for k, v in rooflines.items() if v is not None}
    for k, v in rooflines.items():
        # DRAM bytes per launch of the role on this workload (ncu), null when
        # not captured or the kernel's sources changed since
        v["traffic"] = committed_traffic(TRAFFIC_KEY.get(k, k), w.name)
    bar = None
    if span_ms:
        ach = (fl["up_proj_ctx"] + fl["attn_ctx"]) / (span_ms / 1e3) / 1e12
        bar = {"what": "(a5 up-projection + a6 context attention FLOPs) / (a4..a7 span)",
               "a4_a7_span_ms": span_ms, "tflops": ach, "frac_burst": ach / bf,
               "frac_sustained": (ach / peaks["bf16_tflops_sustained"]
                                  if peaks.get("bf16_tflops_sustained") else None)}
    timeline = [{"kernel": r[0], "role": r[4], "stream": r[1], "start_ms": round(r[2] - per_step[0][0][2], 4),
                 "ms": round(r[3], 4)} for r in per_step[0]] if per_step and per_step[0] else []
    return {"roles": roles, "kernels": kernels, "target_bar": bar, "rooflines": rooflines,
            "timeline_first_step": timeline}


# roofline role -> key of profiles/traffic.json
TRAFFIC_KEY = {"up_proj": "kv_up_proj", "context_attention": "attn_ctx"}


def committed_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, if the kernel's source files have not changed since it was
    taken (else null)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = (d.get(kernel) or {}).get(workload)
    if not e or e.get("sources_sha1") != sources_hash(e.get("sources", [])):
        return None
    return e.get("bytes_per_launch")


def sources_hash(files):
    """sha1 over the named files under the package's csrc/, in order."""
    h = hashlib.sha1()
    c = os.path.join(ROOT, "mla_chunked_context_gb300", "csrc")
    for f in files:
        h.update(open(os.path.join(c, f), "rb").read())
    return h.hexdigest()


def timed_steps(M, step, steps, warmup, flush, stream, profile=True, world=1, sampler=None):
    """W untimed steps, then K steps each bracketed by CUDA events on the
    launching stream, an L2 flush (a 256 MB write) between them outside the
    events; the library's per-launch profile covers the K timed steps.
    Returns (per-step ms, launch records, launches counted)."""
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.mark("t0")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    launched0 = M.mla_kernel_launches()
    if profile:
        M.mla_profile_begin()
    for i in range(steps):
        flush.fill_(i & 0xff)                   # L2 flush outside the timed events
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    launched = M.mla_kernel_launches() - launched0  # this library's kernels only
    torch.cuda.synchronize()
    records = M.mla_profile_end() if profile else []
    if sampler is not None:
        sampler.mark("t1")
    if world > 1:
        torch.distributed.barrier()
    return [a.elapsed_time(b) for a, b in evs], records, launched


def prefill_runner(M, W, w, dev):
    x = W.make_inputs(w)
    g = {k: v.to(dev) for k, v in x.items()}
    plans = M.mla_plan_context_chunks(w.context_lens, w.row_budget, w.max_context_chunk,
                                      w.split_alignment)
    pf = M.ChunkedPrefill(M.Dims.of(w), w.context_lens, w.query_lens, w.row_budget,
                          w.max_context_chunk, w.split_alignment, device=dev)
    out = torch.empty(w.num_tokens, w.num_heads, w.v_dim, dtype=w.torch_dtype, device=dev)
    out_lse = torch.empty(w.num_heads, w.num_tokens, device=dev)

    def step():
        pf(g["q"], g["new_latent"], g["kv_cache"], g["block_table"], g["w_kv_b"], out, out_lse)
    return x, g, plans, pf, out, step


def serial_region(M, step, steps, flush, stream):
    """K steps with the pipeline's overlap off and the per-launch profile on:
    every kernel of a step alone, one after another, on the caller's
    stream."""
    prev = M.mla_set_pipeline_overlap(False)
    try:
        ms, records, _ = timed_steps(M, step, steps, 1, flush, stream, profile=True)
    finally:
        M.mla_set_pipeline_overlap(prev)
    return ms, records


def bench_config(M, W, name, dev, peaks, flush, steps, warmup):
    """One more workload through mla_chunked_prefill: step time, algorithmic
    throughput and the in-step breakdown (same method as the main line)."""
    w = W.workload(name)
    x, g, plans, pf, out, step = prefill_runner(M, W, w, dev)
    stream = torch.cuda.current_stream()
    ms, _, launched = timed_steps(M, step, steps, warmup, flush, stream, profile=False)
    _, records, _ = timed_steps(M, step, steps, 1, flush, stream, profile=True)
    ser_ms, ser_records = serial_region(M, step, steps, flush, stream)
    step_ms = statistics.median(ms)
    fl = flops_of(w, plans)
    br = breakdown_of(records, steps, w, plans, peaks)
    br_ser = breakdown_of(ser_records, steps, w, plans, peaks)
    tf = fl["total"] / (step_ms / 1e3) / 1e12
    res = {"config": config_of(w, plans, 1), "steps": steps, "ms_per_step": step_ms,
           "ms_per_step_all": ms, "tok_per_s": w.num_tokens / (step_ms / 1e3),
           "tflops": tf, "flops_per_step": fl, "gpu_launches_per_step": launched / steps,
           "frac_burst": tf / peaks["bf16_tflops"],
           "frac_sustained": (tf / peaks["bf16_tflops_sustained"]
                              if peaks.get("bf16_tflops_sustained") else None),
           "ms_per_step_serial": statistics.median(ser_ms),
           "target_bar": br["target_bar"], "rooflines": br_ser["rooflines"],
           "rooflines_overlapped": br["rooflines"], "roles": br["roles"]}
    if w.dtype != "bf16":
        res["note"] = ("float32 storage: the CUDA-core kernels (the tensor-core kernels serve "
                       "bf16); fractions are of the bf16 tensor peak for reference only")
    del x, g, pf, out
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------ our arm -----
def run_ours(args, rank, world, dev):
    import mla_chunked_context_gb300 as M
    from mla_chunked_context_gb300 import workloads as W

    w = W.workload(args.workload)
    peaks = load_peaks()
    x, g, plans, pf, out, step = prefill_runner(M, W, w, dev)
    T, H = w.num_tokens, w.num_heads
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    step_ms, _, launched = timed_steps(M, step, args.steps, args.warmup, flush, stream,
                                       profile=False, world=world, sampler=sampler)
    clocks = sampler.stop()
    max_ms = job_time_ms(sum(step_ms), world, dev)
    value = whole_job_rate(T, world, args.steps, max_ms)
    # a second timed region of the same steps with the library's per-launch
    # events on (the in-step breakdown and timeline, kernels side by side)
    prof_ms, records, _ = timed_steps(M, step, args.steps, 1, flush, stream, profile=True)
    # a third with the pipeline's overlap off: the same kernels one after
    # another, so each launch's time is its own (the kernels' rooflines and
    # the dominant kernel, whose shares then match a serialised ncu launch
    # list)
    ser_ms, ser_records = serial_region(M, step, args.steps, flush, stream)

    # ---- e2e: host buffers, copies inside the timed region.  Inputs are
    # double-buffered on the device: step i+1's host->device copy (on a copy
    # stream) overlaps step i's compute; each step's output is read back to
    # pinned host memory on a second copy stream, so the two directions of
    # the host link run side by side.  The region runs from the first copy
    # to the last read-back.
    host = {k: v.pin_memory() for k, v in x.items()}
    sets = [g, {k: torch.empty_like(v) for k, v in g.items()}]
    outs = [out, torch.empty_like(out)]
    host_out = [torch.empty(T, H, w.v_dim, dtype=w.torch_dtype).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = host_out[0].numel() * host_out[0].element_size()
    copy_stream = torch.cuda.Stream(device=dev)
    back_stream = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    back_stream.wait_event(e0)
    in_ready, done, read_back = [None, None], [None, None], [None, None]

    def h2d_into(k):
        with torch.cuda.stream(copy_stream):
            if done[k] is not None:
                copy_stream.wait_event(done[k])      # the step that used this set is done
            for name in sets[k]:
                sets[k][name].copy_(host[name], non_blocking=True)
            in_ready[k] = ev()
            in_ready[k].record(copy_stream)

    h2d_into(0)
    for i in range(args.steps):
        k = i & 1
        if i + 1 < args.steps:
            h2d_into(1 - k)
        stream.wait_event(in_ready[k])
        if read_back[k] is not None:
            stream.wait_event(read_back[k])          # output buffer k was read back
        sk = sets[k]
        pf(sk["q"], sk["new_latent"], sk["kv_cache"], sk["block_table"], sk["w_kv_b"], outs[k],
           None)
        done[k] = ev()
        done[k].record(stream)
        with torch.cuda.stream(back_stream):
            back_stream.wait_event(done[k])
            host_out[k].copy_(outs[k], non_blocking=True)
            read_back[k] = ev()
            read_back[k].record(back_stream)
    for k in range(2):
        if read_back[k] is not None:
            stream.wait_event(read_back[k])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_value = whole_job_rate(T, world, args.steps, job_time_ms(e0.elapsed_time(e1), world, dev))
    del sets[1], outs[1]

    result = None
    if rank == 0:
        fl = flops_of(w, plans)
        br = breakdown_of(records, args.steps, w, plans, peaks)
        br_ser = breakdown_of(ser_records, args.steps, w, plans, peaks)
        # the dominant kernel: the largest share of the step's kernel time
        # with the kernels run one after another
        dom = max(br_ser["rooflines"].items(), key=lambda kv: kv[1]["ms_per_step"])
        roofline = dict(dom[1])
        roofline["kernel"] = dom[0]
        roofline["traffic"] = committed_traffic(TRAFFIC_KEY.get(dom[0], dom[0]), w.name)
        launches = roofline["launches_per_step"]
        roofline["achieved_per_launch_basis"] = (
            "algorithmic work per step / launches = per launch; / mean launch time in steps "
            "run with the pipeline's overlap off (each kernel alone, warm, in a real step)")
        roofline["traffic_basis"] = "DRAM bytes per launch (ncu), null if not captured"
        step_ms_mean = max_ms / args.steps
        merge = bench_merge(M, W, dev, peaks, flush)
        comparator = bench_equal_window(M, w, g, M.Dims.of(w), dev, flush, step_ms_mean)
        configs = {}
        if not args.no_configs:
            del host, host_out
            for name in ("tiny", "uniform", "long"):
                configs[name] = bench_config(M, W, name, dev, peaks, flush, args.config_steps,
                                             3)
        result = {
            "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms_mean,
            "ms_per_step_with_launch_events": statistics.mean(prof_ms),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded host draws; random-init W_kv_b)",
            "config": config_of(w, plans, world),
            "tflops": fl["total"] / (step_ms_mean / 1e3) / 1e12,
            "tensor_frac_step": fl["total"] / (step_ms_mean / 1e3) / 1e12 / peaks["bf16_tflops"],
            "tensor_frac_step_sustained": (
                fl["total"] / (step_ms_mean / 1e3) / 1e12 / peaks["bf16_tflops_sustained"]
                if peaks.get("bf16_tflops_sustained") else None),
            "clocks": clocks,
            "e2e": {"value": e2e_value, "unit": "tok/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launched,
            "roofline": roofline,
            "rooflines": br_ser["rooflines"],
            "rooflines_overlapped": br["rooflines"],
            "ms_per_step_serial": statistics.mean(ser_ms),
            "target_bar": br["target_bar"],
            "breakdown": {"roles": br["roles"], "kernels": br["kernels"],
                          "timeline_first_step": br["timeline_first_step"],
                          "how": "CUDA events recorded by the library on the launching "
                                 "stream around every launch of a second timed region of "
                                 "the same steps (mla_profile_begin/_end); launches on the "
                                 "side streams overlap the caller's, so ms adds up to more "
                                 "than the step and attributed_ms shares overlap out; "
                                 "rooflines come from a third region with the overlap off "
                                 "(mla_set_pipeline_overlap(False))",
                          "kernels_serial": br_ser["kernels"]},
            "merge": merge,
            "comparator": comparator,
            "configs": configs,
            "flops_per_step": fl,
        }
        if world == 1 and not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(w, x, heads=args.cpu_heads)
    return result


def bench_equal_window(M, w, g, dims, dev, flush, new_ms, steps=3):
    """The old equal-window scheme on the same batch (comparator for the
    pages' claim that per-request packing cuts chunks and latency)."""
    window, n_chunks = M.mla_plan_equal_window_chunks(w.context_lens, w.row_budget,
                                                      w.split_alignment)
    ws = torch.empty(M.mla_prefill_equal_window_workspace_bytes(
        dims, w.context_lens, w.query_lens, w.row_budget, w.split_alignment),
        dtype=torch.uint8, device=dev)
    out = torch.empty(w.num_tokens, w.num_heads, w.v_dim, dtype=w.torch_dtype, device=dev)
    stream = torch.cuda.current_stream()

    def go():
        M.mla_chunked_prefill_equal_window(dims, w.context_lens, w.query_lens, w.row_budget,
                                           w.split_alignment, g["q"], g["new_latent"],
                                           g["kv_cache"], g["block_table"], g["w_kv_b"], ws, out)
    go()
    torch.cuda.synchronize()
    ms = []
    for _ in range(steps):
        flush.fill_(4)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        go()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    med = statistics.median(ms)
    plans = M.mla_plan_context_chunks(w.context_lens, w.row_budget, w.max_context_chunk,
                                      w.split_alignment)
    return {"scheme": "equal context windows (the scheme per-request packing replaced)",
            "window_rows": window, "chunks": n_chunks, "ms_per_step": med,
            "packed_chunks": len(plans), "packed_ms_per_step": new_ms,
            "latency_ratio": med / new_ms}


def bench_merge(M, W, dev, peaks, flush, reps=20):
    m = W.MergeWorkload()
    x = W.make_merge_inputs(m, poison=True)
    g = {k: v.to(dev) for k, v in x.items() if torch.is_tensor(v)}
    T, H, D = m.num_tokens, m.num_heads, m.head_dim
    out = torch.empty(T, H, D, dtype=torch.bfloat16, device=dev)
    out_lse = torch.empty(H, T, device=dev)
    stream = torch.cuda.current_stream()

    def go():
        M.merge_attn_states(out, out_lse, g["prefix_o"], g["prefix_lse"], g["suffix_o"],
                            g["suffix_lse"], m.prefix_num_tokens)
    for _ in range(3):
        go()
    ms = []
    for _ in range(reps):
        flush.fill_(2)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        go()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    med = statistics.median(ms)
    need, full = merge_bytes(x, T, H, D)
    gbs = need / (med / 1e3) / 1e9
    return {"workload": "8192 tokens x 128 heads x 128, bf16, 15% empty prefix, "
                        "prefix_num_tokens 6144", "us": med * 1e3, "bytes": need,
            "gbs": gbs, "frac": gbs / peaks["hbm_gbs"], "peak_gbs": peaks["hbm_gbs"],
            "peak_source": peaks["source"] + " copy", "frac_of_8000": gbs / 8000.0,
            "gbs_if_every_byte_read": full / (med / 1e3) / 1e9}


# --------------------------------------------------------- oracle (CPU) ----
def cpu_baseline(w, x, heads=2, start_head=0):
    """The float64 oracle as it stands on a bounded sample: every token of
    the batch for `heads` heads (the oracle run with those heads' W_kv_b rows
    and query columns); tokens/s scaled to all heads."""
    from oracle import mla as O
    H = w.num_heads
    Dn, Dv = w.qk_nope_dim, w.v_dim
    q = x["q"].float().numpy()
    lat = x["new_latent"].float().numpy()
    cache = x["kv_cache"].float().numpy()
    bt = x["block_table"].numpy()
    wk = x["w_kv_b"].float().numpy()
    t0 = time.perf_counter()
    for h in range(start_head, start_head + heads):
        hh = h % H
        d = O.MlaDims(1, w.kv_lora_rank, w.qk_rope_dim, Dn, Dv, w.block_size, w.softmax_scale)
        O.chunked_prefill(q[:, hh:hh + 1], lat, cache, bt, wk[hh * (Dn + Dv):(hh + 1) * (Dn + Dv)],
                          w.context_lens, w.query_lens, d, w.row_budget, w.max_context_chunk,
                          w.split_alignment)
    dt = time.perf_counter() - t0
    threads = None
    try:
        from threadpoolctl import threadpool_info
        threads = max((i.get("num_threads", 0) for i in threadpool_info()), default=None)
    except Exception:
        threads = None
    return {"value": w.num_tokens * heads / H / dt, "unit": "tok/s",
            "cores": threads or os.cpu_count(), "host_cpus": os.cpu_count(), "kind": "oracle",
            "sample": f"all {w.num_tokens} tokens x {heads} of {H} heads of the {w.name} batch "
                      f"(oracle.mla.chunked_prefill, float64, {dt:.1f} s); tok/s scaled by "
                      f"{heads}/{H}"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from mla_chunked_context_gb300 import workloads as W
    from oracle import planner as OP
    w = W.workload(args.workload)
    x = W.make_inputs(w)
    plans = OP.plan_mla_context_chunks(w.context_lens, w.row_budget, w.max_context_chunk,
                                       w.split_alignment)
    cpu_baseline(W.scaled(w, context_lens=[64], query_lens=[4]), W.make_inputs(
        W.scaled(w, context_lens=[64], query_lens=[4])), heads=1)   # warm-up: imports, BLAS
    vals = []
    t0 = time.perf_counter()
    for i in range(args.steps):
        cb = cpu_baseline(w, x, heads=1, start_head=i)
        vals.append(cb)
    dt = time.perf_counter() - t0
    value = w.num_tokens * args.steps / w.num_heads / dt
    cb = dict(vals[-1])
    cb["value"] = value
    cb["sample"] = (f"per step: all {w.num_tokens} tokens x 1 of {w.num_heads} heads "
                    f"(float64 oracle); tok/s scaled by 1/{w.num_heads}")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, plans, world),
            "execution": "float64 oracle on the host cores, rank 0 only",
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_kernel_case(args, dev):
    """One kernel alone on a small DeepSeek-shaped case (for ncu captures and
    quick timing): up_proj, attn (context or causal), fused (context attention
    with the up-projection fused in), merge or gather."""
    import mla_chunked_context_gb300 as M
    from mla_chunked_context_gb300 import workloads as W
    peaks = load_peaks()
    w = W.scaled(W.workload("uniform"), num_heads=args.heads)
    dims = M.Dims.of(w)
    H = args.heads
    kvd = M.mla_chunk_kv_dtype(dims)
    torch.manual_seed(5)
    bf = torch.bfloat16
    info = {}
    if args.kernel == "up_proj":
        rows = args.rows
        lat = torch.randn(rows, 576, device=dev).to(bf)
        wkv = (torch.randn(H * 256, 512, device=dev) * 0.02).to(bf)
        kv = torch.empty(rows, H * 256, dtype=kvd, device=dev)
        fn = lambda: M.mla_kv_up_proj(dims, lat, rows, wkv, kv)  # noqa: E731
        work, unit, peak = 2.0 * rows * 512 * H * 256, "TFLOP/s", peaks["bf16_tflops"]
        info = {"rows": rows, "N": H * 256, "K": 512,
                "bytes": rows * 576 * 2 + H * 256 * 512 * 2 + rows * H * 256 * kv.element_size()}
    elif args.kernel == "attn":
        n, ql, kl = args.seqs, args.qlen, (args.qlen if args.causal else args.klen)
        q = torch.randn(n * ql, H, 192, device=dev).to(bf)
        kv = (0.45 * torch.randn(n * kl, H * 256, device=dev)).to(kvd)
        lat = torch.randn(n * kl, 576, device=dev).to(bf)
        o = torch.empty(n * ql, H, 128, device=dev)
        lse = torch.empty(H, n * ql, device=dev)
        q_loc = [i * ql for i in range(n + 1)]
        k_loc = [i * kl for i in range(n + 1)]
        qd = torch.tensor(q_loc, dtype=torch.int32, device=dev)
        kd = torch.tensor(k_loc, dtype=torch.int32, device=dev)
        fn = lambda: M.mla_varlen_attn(dims, args.causal, q_loc, k_loc, q, kv, lat, o, lse,  # noqa
                                       q_loc_dev=qd, k_loc_dev=kd)
        if args.profile_launches:
            M.mla_profile_begin()
            fn()
            info["launches"] = M.mla_profile_end()
        pairs = n * (ql * (ql + 1) / 2 if args.causal else ql * kl)
        work, unit, peak = 2.0 * H * (192 + 128) * pairs, "TFLOP/s", peaks["bf16_tflops"]
        info = {"seqs": n, "q": ql, "k": kl, "causal": bool(args.causal)}
    elif args.kernel == "step":
        # whole prefills of --workload (the launches of one step, for a
        # traffic capture); work = the step's algorithmic FLOPs
        w = W.workload(args.workload)
        if args.requests or args.first_request:
            # N requests from the K-th on only (a smaller capture)
            r0 = args.first_request
            r1 = r0 + args.requests if args.requests else w.num_requests
            w = W.scaled(w, context_lens=list(w.context_lens[r0:r1]),
                         query_lens=list(w.query_lens[r0:r1]))
        x, g, plans, pf, out, step = prefill_runner(M, W, w, dev)
        fn = step
        work, unit, peak = flops_of(w, plans)["total"], "TFLOP/s", peaks["bf16_tflops"]
        info = {"workload": args.workload, "requests": w.num_requests}
    elif args.kernel == "fused":
        # context attention with the up-projection fused in (one query tile
        # per sequence); work = the up-projection plus the attention
        n, ql, kl = args.seqs, args.qlen, args.klen
        q = torch.randn(n * ql, H, 192, device=dev).to(bf)
        lat = torch.randn(n * kl, 576, device=dev).to(bf)
        wkv = (torch.randn(H * 256, 512, device=dev) * 0.02).to(bf)
        o = torch.empty(n * ql, H, 128, device=dev)
        lse = torch.empty(H, n * ql, device=dev)
        q_loc = [i * ql for i in range(n + 1)]
        k_loc = [i * kl for i in range(n + 1)]
        qd = torch.tensor(q_loc, dtype=torch.int32, device=dev)
        kd = torch.tensor(k_loc, dtype=torch.int32, device=dev)
        ws = torch.empty(M.mla_fused_attn_workspace_bytes(dims, n * ql), dtype=torch.uint8,
                         device=dev)
        fn = lambda: M.mla_fused_context_attn(dims, q_loc, k_loc, q, lat, wkv, o, lse,  # noqa
                                              workspace=ws, q_loc_dev=qd, k_loc_dev=kd)
        work = 2.0 * n * kl * 512 * H * 256 + 2.0 * H * (192 + 128) * n * ql * kl
        unit, peak = "TFLOP/s", peaks["bf16_tflops"]
        info = {"seqs": n, "q": ql, "k": kl}
    elif args.kernel == "merge":
        m = W.MergeWorkload()
        x = W.make_merge_inputs(m, poison=True)
        g = {k: v.to(dev) for k, v in x.items() if torch.is_tensor(v)}
        out = torch.empty_like(g["suffix_o"])
        out_lse = torch.empty_like(g["suffix_lse"])
        fn = lambda: M.merge_attn_states(out, out_lse, g["prefix_o"], g["prefix_lse"],  # noqa
                                         g["suffix_o"], g["suffix_lse"], m.prefix_num_tokens)
        need, _ = merge_bytes(x, m.num_tokens, m.num_heads, m.head_dim)
        work, unit, peak = float(need), "GB/s", peaks["hbm_gbs"]
    elif args.kernel == "gather":
        wl = W.workload("hetero")
        x = W.make_inputs(wl)
        cache, bt = x["kv_cache"].to(dev), x["block_table"].to(dev)
        rows = 32768
        req = torch.tensor([int(np.argmax(wl.context_lens))], dtype=torch.int32, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        cu = torch.tensor([0, rows], dtype=torch.int32, device=dev)
        ws = torch.empty(rows, 576, dtype=bf, device=dev)
        fn = lambda: M.mla_gather_context_rows(M.Dims.of(wl), cache, bt, req, st, cu, rows, ws)  # noqa
        work, unit, peak = 2.0 * rows * 576 * 2, "GB/s", peaks["hbm_gbs"]
    else:
        raise SystemExit(f"unknown kernel {args.kernel}")
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ms = []
    for _ in range(args.launches):
        flush.fill_(3)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    med = statistics.median(ms)
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    ach = work / (med / 1e3) / scale
    print(json.dumps({"kernel": args.kernel, "us": med * 1e3, "achieved": ach, "unit": unit,
                      "peak": peak, "frac": ach / peak, "heads": H, **info,
                      "errors": M.mla_device_error_flags()}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="hetero", choices=["hetero", "uniform", "long"])
    ap.add_argument("--cpu-heads", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the tiny / uniform / long sub-records")
    ap.add_argument("--config-steps", type=int, default=5)
    ap.add_argument("--profile-launches", action="store_true",
                    help="--kernel attn: list the launches of one call")
    ap.add_argument("--kernel", default=None,
                    choices=["up_proj", "attn", "fused", "merge", "gather", "step"],
                    help="time one kernel alone on a small case instead of the full step")
    ap.add_argument("--heads", type=int, default=128)
    ap.add_argument("--rows", type=int, default=8192)
    ap.add_argument("--seqs", type=int, default=4)
    ap.add_argument("--qlen", type=int, default=256)
    ap.add_argument("--klen", type=int, default=4096)
    ap.add_argument("--causal", type=int, default=0)
    ap.add_argument("--launches", type=int, default=10)
    ap.add_argument("--requests", type=int, default=0,
                    help="--kernel step: N requests of the workload only")
    ap.add_argument("--first-request", type=int, default=0,
                    help="--kernel step: start at the workload's K-th request")
    args = ap.parse_args()
    if args.kernel:
        torch.cuda.set_device(0)
        run_kernel_case(args, torch.device("cuda", 0))
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    res = run_ours(args, rank, world, dev)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
