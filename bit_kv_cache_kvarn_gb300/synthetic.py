"""Seeded synthetic inputs for the KVarN codec workloads.

This module only draws random numbers; it holds none of the codec's arithmetic, so both the
CUDA path and the fp64 oracle can be fed from it.  Every draw comes from one torch.Generator
seeded with the workload's seed, in a fixed order, so a (seed, shape, device type) triple always
gives the same tensor.  CPU generation is used for the small parity cases; the large benchmark
workloads are generated on the GPU (same recipe, CUDA Philox stream).

Recipe for a K or V cache with outliers (the pages' KV caches come from Qwen3-4B / Phi-4 on
real text, which is not available here; these draws stand in for them):
  base    ~ N(0, 1)                              [units, tokens, 128]
  chan    ~ lognormal(0, 1) per (unit, channel); 4 distinct random channels per unit x20
  tok     ~ lognormal(0, 0.5) per (unit, token); round(5% of tokens) distinct tokens x8
  x       = base * chan[:, None, :] * tok[:, :, None], rounded to bfloat16 (round-to-nearest-even)
A unit is one (sequence, kv head).  K is drawn first, then V, from the same generator.
"""
from __future__ import annotations

import torch

HEAD_DIM = 128


def _outlier_kv(gen: torch.Generator, units: int, tokens: int, device) -> torch.Tensor:
    base = torch.randn(units, tokens, HEAD_DIM, generator=gen, device=device)
    chan = torch.exp(torch.randn(units, HEAD_DIM, generator=gen, device=device))
    pick_c = torch.rand(units, HEAD_DIM, generator=gen, device=device).argsort(dim=1)[:, :4]
    chan.scatter_(1, pick_c, chan.gather(1, pick_c) * 20.0)
    tok = torch.exp(0.5 * torch.randn(units, tokens, generator=gen, device=device))
    n_out = int(round(0.05 * tokens))
    if n_out > 0:
        pick_t = torch.rand(units, tokens, generator=gen, device=device).argsort(dim=1)[:, :n_out]
        tok.scatter_(1, pick_t, tok.gather(1, pick_t) * 8.0)
    x = base.mul_(chan[:, None, :]).mul_(tok[:, :, None])
    return x.to(torch.bfloat16)


def outlier_kv(seed: int, units: int, tokens: int, device="cpu"):
    """(K, V) bfloat16 tensors of shape [units, tokens, 128] drawn with the recipe above."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    k = _outlier_kv(gen, units, tokens, device)
    v = _outlier_kv(gen, units, tokens, device)
    return k, v


def queries(seed: int, batch: int, heads: int, device="cpu", scale: float = 1.0) -> torch.Tensor:
    """bfloat16 queries [batch, heads, 128] ~ N(0, 1) * scale (drawn from seed + 1_000_003)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 1_000_003)
    q = torch.randn(batch, heads, HEAD_DIM, generator=gen, device=device) * scale
    return q.to(torch.bfloat16)


def ragged_lengths(seed: int, batch: int, lo: int, hi: int) -> list[int]:
    """Context lengths drawn uniformly from the integers [lo, hi] (inclusive), one per sequence."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed + 2_000_003)
    return [int(v) for v in torch.randint(lo, hi + 1, (batch,), generator=gen)]


def tile_permutation(seed: int, n: int, device="cpu") -> torch.Tensor:
    """A random permutation of tile ids (emulates a paged pool whose blocks are scattered)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed + 3_000_003)
    return torch.randperm(n, generator=gen).to(device)
