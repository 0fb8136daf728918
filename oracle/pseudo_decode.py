"""fp64 reference of the block pseudo-decode through the KVarN cache.

TEST INFRASTRUCTURE ONLY (same rules as ``kvarn_oracle``: only the tests may import it; it shares no
code with the CUDA path or with the GPU harness in ``bit_kv_cache_kvarn_gb300.pseudo_decode``).

The evaluation is described in [agihunt] (pipeline paragraph: the sequence is cut into blocks of
usually 128 tokens, each block's K/V is quantised once the block is done, and the growth of the
attention-output reconstruction error over blocks is tracked) and [pheeree] "핵심 세 가지" §1
(the next block reads the quantised cache and makes its own K/V from it; tokens inside a block
still see each other's unquantised K/V).  The pages give no model, so these readings are taken:

* attention-only layers with a residual: h <- h + W_O attn(h); pre-norm RMSNorm (eps 1e-6, unit
  weight); q = W_Q n, k = W_K n, v = W_V n with grouped-query heads (kv head of query head h is
  h // (Hq / Hkv)); rotate-half RoPE with base 1e6 on q and k at absolute positions; softmax scale
  1/sqrt(128); causal inside the block;
* K and V enter the cache as bfloat16 values (the codec's input precision) and the query is
  rounded to bfloat16 too (the decode kernel's input); the block's own unquantised K/V are those
  bfloat16 values;
* the quantised cache of a finished block = dequantise(encode(block)) per kv head, K with
  cfg k_bits, V with v_bits ([paperlayer] "2 Preliminaries": one 128 x 128 tile per head and block);
* the reported error of block j, layer l = mean |attn_quantised - attn_reference| over the block's
  tokens, heads and channels, attn taken before W_O, both runs free-running (each feeds its own
  outputs forward).
"""
from __future__ import annotations

import numpy as np

from oracle import kvarn_oracle as o

HEAD = 128
ROPE_BASE = 1e6
RMS_EPS = 1e-6


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 (ties to even), via float32 bit patterns.

    fp64 -> fp32 is itself a rounding; double rounding only matters for values within 2^-29
    relative of a bf16 half-way point, which the fp32 inputs used here never are (pinned)."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def rmsnorm(x: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) over the last axis (unit weight)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def rope(x: np.ndarray, pos: np.ndarray, base: float = ROPE_BASE) -> np.ndarray:
    """Rotate-half RoPE: channel i < 64 pairs with i + 64, angle pos * base^(-i/64).
    x: [T, H, 128], pos: [T]."""
    half = HEAD // 2
    freq = base ** (-np.arange(half, dtype=np.float64) / half)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * freq[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def causal_block_attention(q, k_prev, v_prev, k_blk, v_blk, scale):
    """Attention of the block's queries q [T, Hq, 128] over the previous tokens (k_prev, v_prev:
    [P, Hkv, 128]) and, causally, the block's own tokens (k_blk, v_blk: [T, Hkv, 128])."""
    t_blk, hq = q.shape[0], q.shape[1]
    hkv = k_blk.shape[1]
    group = hq // hkv
    out = np.zeros((t_blk, hq, HEAD))
    for h in range(hq):
        kv = h // group
        keys = np.concatenate([k_prev[:, kv], k_blk[:, kv]], axis=0)
        vals = np.concatenate([v_prev[:, kv], v_blk[:, kv]], axis=0)
        s = scale * (q[:, h] @ keys.T)  # [T, P + T]
        p_len = k_prev.shape[0]
        mask = np.arange(p_len + t_blk)[None, :] > (p_len + np.arange(t_blk))[:, None]
        s = np.where(mask, -np.inf, s)
        s = s - s.max(axis=1, keepdims=True)
        w = np.exp(s)
        out[:, h] = (w / w.sum(axis=1, keepdims=True)) @ vals
    return out


def quantise_block(kv_blk: np.ndarray, kind: str, bits: int, iters: int, rotate: bool,
                   normalize: bool) -> np.ndarray:
    """Dequantised cache entries of one finished block: [T=128, Hkv, 128] -> same shape."""
    out = np.zeros_like(kv_blk)
    for h in range(kv_blk.shape[1]):
        e = o.encode_tile(kv_blk[:, h], kind, bits, iters, rotate, normalize)
        out[:, h] = o.dequant_tile(e["codes"], e["S1"], e["s2"], e["Z"], e["g"], kind,
                                   original_basis=True, rotate=rotate)
    return out


def run(weights, x, hq: int, hkv: int, quantised: bool, k_bits: int = 2, v_bits: int = 2,
        iters: int = o.DEFAULT_ITERS, rotate: bool = True, normalize: bool = True,
        block: int = o.TILE, kv_token_scale=None):
    """Free-running pseudo-decode.  weights: list of dicts with wq [Hq*128, D], wk, wv
    [Hkv*128, D], wo [D, Hq*128]; x: [T, D] layer-0 inputs.  Returns attn[j][l]: [block, Hq, 128].

    kv_token_scale: optional [T] multipliers of each position's K and V projections, for a stack
    whose K/V carry token-scale outliers (the pages' caches have them; a pre-norm stack would
    remove any scale of its input tokens, so it is applied to the projections' outputs)."""
    x = np.asarray(x, dtype=np.float64)
    n_blocks = x.shape[0] // block
    scale = 1.0 / np.sqrt(HEAD)
    caches = [([], []) for _ in weights]  # per layer: lists of [block, Hkv, 128] entries
    attn = []
    for j in range(n_blocks):
        h = x[j * block:(j + 1) * block].copy()
        pos = np.arange(j * block, (j + 1) * block)
        per_layer = []
        for l, w in enumerate(weights):
            n = rmsnorm(h)
            q = rope((n @ w["wq"].T).reshape(block, hq, HEAD), pos)
            kp, vp = n @ w["wk"].T, n @ w["wv"].T
            if kv_token_scale is not None:
                ts = np.asarray(kv_token_scale, dtype=np.float64)[j * block:(j + 1) * block, None]
                kp, vp = kp * ts, vp * ts
            k = rope(kp.reshape(block, hkv, HEAD), pos)
            v = vp.reshape(block, hkv, HEAD)
            q, k, v = bf16_round(q), bf16_round(k), bf16_round(v)
            kc, vc = caches[l]
            k_prev = np.concatenate(kc, axis=0) if kc else np.zeros((0, hkv, HEAD))
            v_prev = np.concatenate(vc, axis=0) if vc else np.zeros((0, hkv, HEAD))
            a = causal_block_attention(q, k_prev, v_prev, k, v, scale)
            per_layer.append(a)
            h = h + a.reshape(block, hq * HEAD) @ w["wo"].T
            if quantised:
                kc.append(quantise_block(k, "K", k_bits, iters, rotate, normalize))
                vc.append(quantise_block(v, "V", v_bits, iters, rotate, normalize))
            else:
                kc.append(k)
                vc.append(v)
        attn.append(per_layer)
    return attn


def mae_curves(attn_q, attn_ref):
    """mae[j][l] = mean |attn_q - attn_ref| of block j, layer l."""
    return np.array([[float(np.mean(np.abs(a - b))) for a, b in zip(rq, rr)]
                     for rq, rr in zip(attn_q, attn_ref)])
