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


# ---- the block pseudo-decode stack (an attention-only model with random weights) --------------
def pseudo_decode_weights(seed: int, layers: int, hidden: int, hq: int, hkv: int, device="cpu",
                          kv_outliers: bool = False):
    """Per layer {wq [hq*128, D], wk, wv [hkv*128, D], wo [D, hq*128]}, N(0, 0.02), bf16.

    kv_outliers: give the K and V projections the outlier channels of the cache recipe above --
    each output row (one channel of one kv head) of W_K, and separately of W_V, is multiplied by
    lognormal(0, 1), and 4 distinct channels per kv head by a further x20 -- drawn from a second
    generator, so the base weights are the same with and without."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    out = []
    for _ in range(layers):
        w = {}
        for name, shape in (("wq", (hq * HEAD_DIM, hidden)), ("wk", (hkv * HEAD_DIM, hidden)),
                            ("wv", (hkv * HEAD_DIM, hidden)), ("wo", (hidden, hq * HEAD_DIM))):
            w[name] = torch.randn(shape, generator=g) * 0.02
        out.append(w)
    if kv_outliers:
        g2 = torch.Generator(device="cpu").manual_seed(seed + 104_729)
        for w in out:
            for name in ("wk", "wv"):
                chan = torch.exp(torch.randn(hkv, HEAD_DIM, generator=g2))
                pick = torch.rand(hkv, HEAD_DIM, generator=g2).argsort(dim=1)[:, :4]
                chan.scatter_(1, pick, chan.gather(1, pick) * 20.0)
                w[name] = w[name] * chan.reshape(-1, 1)
    return [{k: v.to(torch.bfloat16).to(device) for k, v in w.items()} for w in out]


def pseudo_decode_input(seed: int, tokens: int, hidden: int, device="cpu") -> torch.Tensor:
    """Layer-0 inputs [tokens, hidden], N(0, 1), bf16."""
    g = torch.Generator(device="cpu").manual_seed(seed + 7919)
    return torch.randn(tokens, hidden, generator=g).to(torch.bfloat16).to(device)


def pseudo_decode_token_scales(seed: int, tokens: int) -> torch.Tensor:
    """Per-position multipliers of the K and V projections for the outlier variant of the stack:
    lognormal(0, 0.5), with round(5% of positions) distinct positions x8 -- the token part of the
    cache recipe above.  (A pre-norm model removes any scale of its input tokens, so the variant
    applies them to the projections' outputs.)  float32 [tokens] on the CPU."""
    g = torch.Generator(device="cpu").manual_seed(seed + 130_363)
    tok = torch.exp(0.5 * torch.randn(tokens, generator=g))
    n_out = int(round(0.05 * tokens))
    if n_out > 0:
        pick = torch.rand(tokens, generator=g).argsort()[:n_out]
        tok[pick] *= 8.0
    return tok
