"""Seeded synthetic inputs for MLA chunked-context prefill.

This module only draws inputs: request lengths, the paged latent cache and its
block table, queries, new-token latents, the W_kv_b weight, and the merge
inputs.  It holds none of the method's arithmetic, so both the CUDA path and
the float64 oracle may consume what it returns.

Every array is drawn on the host with ``numpy.random.default_rng(seed)`` in a
fixed order; bf16 tensors are the float32 draw rounded to bf16 (round to
nearest even, by torch's conversion).

Workloads (all synthetic; sizes are those of the DeepSeek-V3 MLA layer shape
unless stated):

* ``tiny``      4 requests, context [0,64,200,37], queries [3,1,16,5]; 16
                heads; latent 64 + rope 16, block 16; W N(0,0.02) up to nope 32
                and v 32; float32 everything; budget 128, alignment 16.
* ``merge``     standalone merge: 8192 tokens x 128 heads x 128; O bf16
                N(0,1); LSE fp32 N(5,2); 15% of tokens have an empty prefix
                (LSE=-inf, O=0); prefix_num_tokens 6144; 4 (token, head) rows
                with both sides empty.
* ``uniform``   16 requests x (context 4096, query 512); 128 heads; latent 512
                + rope 64, bf16 cache with block 64; nope 128, v 128; scale
                1/sqrt(192); budget 65536, alignment 64.
* ``hetero``    32 requests: one context of 131072, 24 drawn log-uniform on
                [1, 2048], 7 zero, in a seeded order; queries uniform on
                [1, 256]; budget 32768, alignment 64.
* ``long``      4 requests x (context 65536, query 2048); budget 65536.

Unused slots of each request's last cache block are NaN, so any read of a row
past a request's context shows up in the output.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np
import torch


@dataclass
class MlaWorkload:
    name: str
    context_lens: list
    query_lens: list
    num_heads: int
    kv_lora_rank: int
    qk_rope_dim: int
    qk_nope_dim: int
    v_dim: int
    block_size: int
    row_budget: int
    split_alignment: int
    dtype: str                      # "bf16" or "f32": storage of every input
    seed: int
    max_context_chunk: Optional[int] = None   # None: equal to row_budget
    softmax_scale: Optional[float] = None     # None: 1/sqrt(nope + rope)
    w_std: float = 0.02
    extra: dict = field(default_factory=dict)

    def __post_init__(self):
        if self.max_context_chunk is None:
            self.max_context_chunk = self.row_budget
        if self.softmax_scale is None:
            self.softmax_scale = 1.0 / math.sqrt(self.qk_nope_dim + self.qk_rope_dim)

    @property
    def num_requests(self) -> int:
        return len(self.context_lens)

    @property
    def num_tokens(self) -> int:
        return int(sum(self.query_lens))

    @property
    def latent_dim(self) -> int:
        return self.kv_lora_rank + self.qk_rope_dim

    @property
    def qk_dim(self) -> int:
        return self.qk_nope_dim + self.qk_rope_dim

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


DEEPSEEK = dict(num_heads=128, kv_lora_rank=512, qk_rope_dim=64,
                qk_nope_dim=128, v_dim=128, block_size=64, dtype="bf16")


def _hetero_lens(seed: int):
    rng = np.random.default_rng(seed)
    u = rng.uniform(0.0, math.log(2048.0), size=24)
    drawn = [int(round(math.exp(x))) for x in u]
    lens = [131072] + drawn + [0] * 7
    perm = rng.permutation(len(lens))
    ctx = [lens[i] for i in perm]
    qlens = [int(x) for x in rng.integers(1, 257, size=len(ctx))]
    return ctx, qlens


def workload(name: str) -> MlaWorkload:
    """The named synthetic workload (see module docstring)."""
    if name == "tiny":
        return MlaWorkload("tiny", [0, 64, 200, 37], [3, 1, 16, 5], num_heads=16,
                           kv_lora_rank=64, qk_rope_dim=16, qk_nope_dim=32,
                           v_dim=32, block_size=16, row_budget=128,
                           split_alignment=16, dtype="f32", seed=0)
    if name == "uniform":
        return MlaWorkload("uniform", [4096] * 16, [512] * 16, row_budget=65536,
                           split_alignment=64, seed=2, **DEEPSEEK)
    if name == "hetero":
        ctx, ql = _hetero_lens(3)
        return MlaWorkload("hetero", ctx, ql, row_budget=32768,
                           split_alignment=64, seed=3, **DEEPSEEK)
    if name == "long":
        return MlaWorkload("long", [65536] * 4, [2048] * 4, row_budget=65536,
                           split_alignment=64, seed=4, **DEEPSEEK)
    raise KeyError(name)


def scaled(w: MlaWorkload, **kw) -> MlaWorkload:
    """A copy with some fields replaced (smaller parity cases)."""
    out = replace(w, **kw)
    out.__post_init__()
    return out


def _to_storage(a: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def make_inputs(w: MlaWorkload) -> dict:
    """Draw every input of the prefill; CPU torch tensors in storage dtype.

    Keys: q [T, H, Dn+P]; new_latent [T, L+P]; kv_cache [blocks, bs, L+P];
    block_table [R, max_blocks] int32; w_kv_b [H*(Dn+Dv), L].
    """
    rng = np.random.default_rng(1000 + w.seed)
    H, L, P = w.num_heads, w.kv_lora_rank, w.qk_rope_dim
    Dn, Dv, bs = w.qk_nope_dim, w.v_dim, w.block_size
    T = w.num_tokens
    w_kv_b = rng.standard_normal((H * (Dn + Dv), L), dtype=np.float32) * np.float32(w.w_std)
    q = rng.standard_normal((T, H, Dn + P), dtype=np.float32)
    new_latent = rng.standard_normal((T, L + P), dtype=np.float32)
    nblk = [(c + bs - 1) // bs for c in w.context_lens]
    total = max(1, sum(nblk))
    cache = rng.standard_normal((total, bs, L + P), dtype=np.float32)
    phys = rng.permutation(total).astype(np.int32)
    maxb = max(1, max(nblk))
    bt = np.zeros((w.num_requests, maxb), dtype=np.int32)
    k = 0
    for r, nb in enumerate(nblk):
        bt[r, :nb] = phys[k:k + nb]
        k += nb
        tail = w.context_lens[r] % bs
        if nb and tail:
            cache[bt[r, nb - 1], tail:, :] = np.nan
    return dict(q=_to_storage(q, w.dtype), new_latent=_to_storage(new_latent, w.dtype),
                kv_cache=_to_storage(cache, w.dtype), block_table=torch.from_numpy(bt),
                w_kv_b=_to_storage(w_kv_b, w.dtype))


@dataclass
class MergeWorkload:
    num_tokens: int = 8192
    num_heads: int = 128
    head_dim: int = 128
    prefix_num_tokens: int = 6144
    empty_frac: float = 0.15
    both_empty: int = 4
    dtype: str = "bf16"
    seed: int = 1


def make_merge_inputs(m: MergeWorkload, poison: bool = True) -> dict:
    """Inputs of the standalone merge.  O [T, H, D] in storage dtype, LSE
    [H, T] float32.  With ``poison`` the prefix side of tokens at or past
    ``prefix_num_tokens`` is NaN (it must never be read)."""
    rng = np.random.default_rng(m.seed)
    T, H, D = m.num_tokens, m.num_heads, m.head_dim
    p_o = rng.standard_normal((T, H, D), dtype=np.float32)
    s_o = rng.standard_normal((T, H, D), dtype=np.float32)
    p_l = (5.0 + 2.0 * rng.standard_normal((H, T))).astype(np.float32)
    s_l = (5.0 + 2.0 * rng.standard_normal((H, T))).astype(np.float32)
    n_empty = int(round(m.empty_frac * T))
    empty_tok = np.sort(rng.choice(T, size=n_empty, replace=False))
    p_l[:, empty_tok] = -np.inf
    p_o[empty_tok] = 0.0
    below = empty_tok[empty_tok < m.prefix_num_tokens]
    both = []
    if m.both_empty and below.size:
        toks = rng.choice(below, size=min(m.both_empty, below.size), replace=False)
        heads = rng.integers(0, H, size=toks.size)
        for t, h in zip(toks, heads):
            s_l[h, t] = -np.inf
            s_o[t, h] = 0.0
            both.append((int(t), int(h)))
    if poison:
        p_o[m.prefix_num_tokens:] = np.nan
        p_l[:, m.prefix_num_tokens:] = np.nan
    return dict(prefix_o=_to_storage(p_o, m.dtype), prefix_lse=torch.from_numpy(p_l),
                suffix_o=_to_storage(s_o, m.dtype), suffix_lse=torch.from_numpy(s_l),
                prefix_num_tokens=m.prefix_num_tokens, empty_tokens=empty_tok,
                both_empty=both)
