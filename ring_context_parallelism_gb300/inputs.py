"""Seeded synthetic inputs for the attention workloads.

This module only draws numbers: it holds none of the attention arithmetic, so
both the CUDA path and the fp64 oracle can be fed from it.  Every tensor is
N(0, 1) drawn in float32 from a seeded ``torch.Generator`` and rounded to the
storage dtype (round-to-nearest-even for bf16).  Small workloads are drawn on
the CPU; the large ones can be drawn on the GPU with a seeded CUDA generator
and copied back in the slices the oracle needs.

Workload shapes follow the pages' long-context and fan-out examples:
  * a 1M-token, 32-head, d_k = 128 context ("RingAttention and Context
    Parallelism", section 1 and section 7 memory table),
  * Llama-3-70B-shaped GQA attention (64 query heads, 8 KV heads),
  * agentic fan-out: one shared prefix, several branches with a few new query
    rows and a private suffix each ("AHBM Agentic Runtime Architecture",
    sections 1.1 and 3.2).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class AttnWorkload:
    name: str
    B: int
    S: int
    Hq: int
    Hkv: int
    D: int
    dtype: str            # "f32" or "bf16"
    causal: bool
    n_shards: int
    block: int
    seed: int
    key_boost_frac: float = 0.0   # fraction of key positions scaled by key_boost
    key_boost: float = 8.0
    partials: bool = False        # per-shard partials + merge instead of one fused pass

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


@dataclass(frozen=True)
class FanoutWorkload:
    name: str
    S_prefix: int
    S_suffix: int
    n_branches: int
    rows_lo: int           # new query rows per branch ~ U{rows_lo .. rows_hi}
    rows_hi: int
    Hq: int
    Hkv: int
    D: int
    dtype: str
    seed: int

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = {
    "tiny_exact_f32": AttnWorkload("tiny_exact_f32", 1, 1024, 4, 4, 64, "f32", False, 4, 64, 1001),
    "gqa_causal_prefill_32k": AttnWorkload("gqa_causal_prefill_32k", 1, 32768, 32, 8, 128, "bf16",
                                           True, 8, 128, 1002),
    "llama70b_layer_128k_partials": AttnWorkload("llama70b_layer_128k_partials", 1, 131072, 64, 8, 128,
                                                 "bf16", True, 16, 128, 1003, partials=True),
    "million_token_stress": AttnWorkload("million_token_stress", 1, 1048576, 32, 8, 128, "bf16", True,
                                         64, 128, 1005, key_boost_frac=0.01),
    "fanout_decode": FanoutWorkload("fanout_decode", 65536, 512, 16, 1, 16, 64, 8, 128, "bf16", 1004),
    "fanout_decode1": FanoutWorkload("fanout_decode1", 65536, 512, 16, 1, 1, 64, 8, 128, "bf16", 1004),
    # fan-out prefill: 8 sub-agents x 20 new tokens (M = 160 stacked rows), each the tail of a
    # 512-token private suffix, against the 65536-token shared prefix
    "fanout_prefill_8x20": FanoutWorkload("fanout_prefill_8x20", 65536, 512, 8, 20, 20, 64, 8, 128, "bf16", 1006),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn(shape, gen: torch.Generator, dtype, device) -> torch.Tensor:
    """N(0,1) in float32, then rounded to ``dtype``."""
    x = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    return x if dtype == torch.float32 else x.to(dtype)


def attention_inputs(w: AttnWorkload, device="cpu"):
    """q [B,S,Hq,D], k/v [B,S,Hkv,D] for workload ``w`` (seeded)."""
    g = _gen(w.seed, device)
    q = randn((w.B, w.S, w.Hq, w.D), g, w.torch_dtype, device)
    k = randn((w.B, w.S, w.Hkv, w.D), g, w.torch_dtype, device)
    v = randn((w.B, w.S, w.Hkv, w.D), g, w.torch_dtype, device)
    if w.key_boost_frac > 0:
        pos = boosted_key_positions(w, device)
        k.index_copy_(1, pos, k.index_select(1, pos) * w.key_boost)
    return q, k, v


def boosted_key_positions(w: AttnWorkload, device="cpu") -> torch.Tensor:
    """round(frac * S) distinct key positions, drawn without replacement by seed.

    The whole key row (all KV heads, all d) at these positions is multiplied by
    ``key_boost`` (a power of two, so exact in bf16)."""
    n = int(round(w.key_boost_frac * w.S))
    g = _gen(w.seed + 7919, "cpu")
    return torch.randperm(w.S, generator=g)[:n].sort().values.to(device)


def branch_rows(w: FanoutWorkload) -> list[int]:
    """New query rows per branch ~ U{rows_lo..rows_hi}, seeded."""
    g = _gen(w.seed + 104729, "cpu")
    return torch.randint(w.rows_lo, w.rows_hi + 1, (w.n_branches,), generator=g).tolist()


def fanout_inputs(w: FanoutWorkload, device="cpu", rows=None):
    """Stacked branch rows and the shared / private KV for workload ``w``.

    Returns dict with q_rows [R,Hq,D], offsets int32 [nb+1] (CSR over stacked
    rows), k_prefix/v_prefix [S_prefix,Hkv,D], k_suffix/v_suffix
    [nb,S_suffix,Hkv,D]."""
    rows = branch_rows(w) if rows is None else list(rows)
    offsets = [0]
    for n in rows:
        offsets.append(offsets[-1] + n)
    R = offsets[-1]
    g = _gen(w.seed, device)
    dt = w.torch_dtype
    k_prefix = randn((w.S_prefix, w.Hkv, w.D), g, dt, device)
    v_prefix = randn((w.S_prefix, w.Hkv, w.D), g, dt, device)
    k_suffix = randn((w.n_branches, w.S_suffix, w.Hkv, w.D), g, dt, device)
    v_suffix = randn((w.n_branches, w.S_suffix, w.Hkv, w.D), g, dt, device)
    q_rows = randn((R, w.Hq, w.D), g, dt, device)
    return dict(q_rows=q_rows, offsets=torch.tensor(offsets, dtype=torch.int32, device=device),
                k_prefix=k_prefix, v_prefix=v_prefix, k_suffix=k_suffix, v_suffix=v_suffix,
                R=R, rows=rows)


def sample_queries(w: AttnWorkload, n: int, seed: int | None = None) -> torch.Tensor:
    """Stratified sample of query ids (b*S + i)*Hq + h.

    Always includes row 0, row S-1 and the first and last row of every shard
    (each with a random head and batch); the rest are uniform.  Ids are unique
    and sorted."""
    g = _gen(w.seed + 31337 if seed is None else seed, "cpu")
    L = w.S // w.n_shards
    fixed = [0, w.S - 1]
    for j in range(w.n_shards):
        fixed += [j * L, (j + 1) * L - 1]
    rows = torch.tensor(fixed, dtype=torch.int64)
    extra = max(n - rows.numel(), 0)
    rows = torch.cat([rows, torch.randint(0, w.S, (extra,), generator=g)])
    heads = torch.randint(0, w.Hq, (rows.numel(),), generator=g)
    batch = torch.randint(0, w.B, (rows.numel(),), generator=g)
    ids = (batch * w.S + rows) * w.Hq + heads
    return torch.unique(ids)


def small(w, **kw):
    """A copy of a workload with some fields replaced (for test-sized cases)."""
    return replace(w, **kw)
