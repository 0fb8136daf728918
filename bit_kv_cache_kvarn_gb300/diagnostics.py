"""Error diagnostics of the codec: magnitude vs direction error and token-scale statistics.

For each token row of a K (or V) tile the squared reconstruction error splits exactly into a
magnitude part E_M = (|x| - |x_hat|)^2 and a direction part E_D = 2 |x| |x_hat| (1 - cos theta)
([pheeree] "핵심 세 가지" §2; the paper reads that the largest errors are mostly magnitude errors,
i.e. wrong token scales).  The token-scale ratio |x_hat| / |x| per token shows how well each
token's scale survives, including the tails of the token-norm distribution ([paperlayer] "B Full
Token-Scale Distribution Error": rotation alone helps the bulk, variance normalisation the very
large and very small tokens).

Encode and dequantisation run through libkvarn; the statistics are plain PyTorch (fp64) on the
dequantised tiles.  Compared presets: KVarN (K2V2, K4V2), rotation only, and plain RTN (KIVI's
grouping).
"""
from __future__ import annotations

import torch

FRACTIONS = (0.5, 0.1, 0.05, 0.01, 0.001)
PRESETS = ("kivi_k2v2_g128", "hadamard_k2v2_g128", "kvarn_k2v2_g128", "kvarn_k4v2_g128")


def roundtrip(kv, cfg, kind: int, x):
    """x: [n, 128, 128] bf16 tiles -> dequantised float32 tiles in the original basis."""
    n = x.shape[0]
    bits = cfg.k_bits if kind == kv.KVARN_KIND_K else cfg.v_bits
    codes = torch.empty(n, 2048 * bits, dtype=torch.uint8, device=x.device)
    params = torch.empty(n, 512, dtype=torch.uint8, device=x.device)
    scale = torch.empty(n, dtype=torch.float32, device=x.device)
    kv.kvarn_encode_blocks(cfg, kind, x, codes, params, scale)
    out = torch.empty(n, 128, 128, dtype=torch.float32, device=x.device)
    kv.kvarn_dequant(cfg, kind, codes, params, scale, out, original_basis=1)
    return out


def stats(x, x_hat):
    """Token rows of x, x_hat ([..., 128]) -> dict of the diagnostics (plain floats)."""
    x = x.reshape(-1, x.shape[-1]).double()
    xh = x_hat.reshape(-1, x_hat.shape[-1]).double()
    n = torch.linalg.vector_norm(x, dim=1)
    nh = torch.linalg.vector_norm(xh, dim=1)
    e_m = (n - nh) ** 2
    e_d = 2.0 * (n * nh - (x * xh).sum(dim=1))
    tot = e_m + e_d
    order = torch.argsort(tot, descending=True, stable=True)
    share = {}
    for f in FRACTIONS:
        top = order[:max(1, int(round(f * tot.numel())))]
        share[str(f)] = float(e_m[top].sum() / tot[top].sum())
    ratio = torch.where(n > 0, nh / torch.where(n > 0, n, torch.ones_like(n)), torch.ones_like(n))
    lr = torch.log2(ratio).abs()
    by_norm = torch.argsort(n, stable=True)
    k = max(1, n.numel() // 100)
    return {
        "mse_per_element": float(tot.sum() / x.numel()),
        "magnitude_share_of_all_error": float(e_m.sum() / tot.sum()),
        "magnitude_share_of_top_errors": share,
        "token_scale_abs_log2_ratio": {
            "mean": float(lr.mean()),
            "p99": float(torch.quantile(lr.float(), 0.99)),
            "smallest_1pct_tokens": float(lr[by_norm[:k]].mean()),
            "largest_1pct_tokens": float(lr[by_norm[-k:]].mean()),
        },
    }


def run(kv, k, v, presets=PRESETS):
    """k, v: [n, 128, 128] bf16 tiles on the GPU -> {preset: {"K": stats, "V": stats}}."""
    res = {}
    for name in presets:
        cfg = kv.kvarn_config_from_preset(name)
        res[name] = {"K": stats(k.float(), roundtrip(kv, cfg, kv.KVARN_KIND_K, k)),
                     "V": stats(v.float(), roundtrip(kv, cfg, kv.KVARN_KIND_V, v))}
    return res
