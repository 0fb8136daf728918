"""Block pseudo-decode through the packed KVarN cache, on the GPU.

The evaluation the pages use to show error accumulation ([agihunt], pipeline paragraph; [pheeree]
"핵심 세 가지" §1): the sequence is processed in 128-token blocks; once a block is done its K/V are
encoded into the cache, and every later block attends to the cache through the codec, while the
tokens of the current block see each other unquantised.  The reported quantity is the mean
absolute difference of each block's attention outputs (before W_O) from a run with an
unquantised cache, layer by layer.

The model is a synthetic attention-only stack (the pages name none): per layer pre-norm RMSNorm
(eps 1e-6, unit weight), grouped-query projections, rotate-half RoPE (base 1e6) on q and k,
softmax scale 1/sqrt(128), residual h += W_O attn.  Weights and inputs are seeded synthetic
tensors.  The projections, norm and RoPE are plain PyTorch (fp32, TF32 off); every step of the
codec -- the encode of each finished block and the attention over the packed cache -- runs in
libkvarn's kernels: a block's 128 queries are 128 one-query "sequences" sharing the block table of
the previous blocks, with lengths 128 j + t + 1 and the current block as their bf16 tail.
"""
from __future__ import annotations

import math
import time

import torch

from . import synthetic

HEAD = 128
BLOCK = 128
ROPE_BASE = 1e6
RMS_EPS = 1e-6


def make_weights(seed: int, layers: int, hidden: int, hq: int, hkv: int, device="cuda", kv_outliers=False):
    """The stack's weights (synthetic.pseudo_decode_weights) on `device`."""
    return synthetic.pseudo_decode_weights(seed, layers, hidden, hq, hkv, device, kv_outliers)


def make_input(seed: int, tokens: int, hidden: int, device="cuda"):
    """Layer-0 inputs [tokens, hidden] (synthetic.pseudo_decode_input) on `device`."""
    return synthetic.pseudo_decode_input(seed, tokens, hidden, device)


def _rmsnorm(x):
    return x * torch.rsqrt(torch.mean(x * x, dim=-1, keepdim=True) + RMS_EPS)


def _rope(x, pos):
    half = HEAD // 2
    freq = ROPE_BASE ** (-torch.arange(half, dtype=torch.float64, device=x.device) / half)
    ang = pos.to(torch.float64)[:, None] * freq[None, :]
    c = torch.cos(ang).to(torch.float32)[:, None, :]
    s = torch.sin(ang).to(torch.float32)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1)


def _exact_attention(q, k_all, v_all, n_prev, scale):
    """Reference attention on an unquantised cache: q [T, Hq, 128] over k_all, v_all
    [n_prev + T, Hkv, 128] (fp32), causal inside the block."""
    t, hq = q.shape[0], q.shape[1]
    group = hq // k_all.shape[1]
    kk = k_all.repeat_interleave(group, dim=1).permute(1, 2, 0)  # [Hq, 128, L]
    vv = v_all.repeat_interleave(group, dim=1).permute(1, 0, 2)  # [Hq, L, 128]
    s = torch.bmm(q.permute(1, 0, 2), kk) * scale  # [Hq, T, L]
    length = k_all.shape[0]
    mask = torch.arange(length, device=q.device)[None, :] > (n_prev + torch.arange(t, device=q.device))[:, None]
    s = s.masked_fill(mask[None], float("-inf"))
    return torch.bmm(torch.softmax(s, dim=-1), vv).permute(1, 0, 2)  # [T, Hq, 128]


def run(kv, cfg, weights, x, hq: int, hkv: int, quantised: bool = True, capture=None, kv_token_scale=None):
    """Free-running pseudo-decode over all blocks of x.  Returns (attn, seconds) with attn[j][l]
    the fp32 attention output [128, hq, 128] of block j, layer l.

    kv_token_scale: optional [tokens] multipliers of each position's K and V projections (the
    outlier variant, synthetic.pseudo_decode_token_scales).

    capture: optional dict keyed by (block, layer); for each key present the codec's inputs and
    output at that point are stored as its value -- dict(q, k_blk, v_blk, attn, pools,
    n_prev_blocks), pools = the packed tiles of the previous blocks (tile id = block * hkv + kv
    head) -- for a teacher-forced check."""
    dev = x.device
    n_blocks = x.shape[0] // BLOCK
    layers = len(weights)
    scale = 1.0 / math.sqrt(HEAD)
    if quantised:
        kb, vb = cfg.k_bits, cfg.v_bits
        # attention keeps the current block in the bf16 tail: the full FP16 window
        cfg_dec = kv.make_config(cfg.k_bits, cfg.v_bits, cfg.sinkhorn_iters, cfg.flags | kv.KVARN_FLAG_FULL_TAIL)
    old_tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    # per layer: packed pools (tile id of block j, kv head h = j * hkv + h) or exact caches
    n_tiles = n_blocks * hkv
    pools = []
    exact = []
    for _ in range(layers):
        if quantised:
            pools.append((torch.empty(n_tiles, HEAD * 16 * kb, dtype=torch.uint8, device=dev),
                          torch.empty(n_tiles, 512, dtype=torch.uint8, device=dev),
                          torch.empty(n_tiles, dtype=torch.float32, device=dev),
                          torch.empty(n_tiles, HEAD * 16 * vb, dtype=torch.uint8, device=dev),
                          torch.empty(n_tiles, 512, dtype=torch.uint8, device=dev),
                          torch.empty(n_tiles, dtype=torch.float32, device=dev)))
        else:
            exact.append((torch.empty(n_blocks * BLOCK, hkv, HEAD, device=dev),
                          torch.empty(n_blocks * BLOCK, hkv, HEAD, device=dev)))
    max_tiles = max(n_blocks, 1)
    table = (torch.arange(max_tiles, device=dev, dtype=torch.int32)[None, :] * hkv
             + torch.arange(hkv, device=dev, dtype=torch.int32)[:, None])  # [hkv, max_tiles]
    table = table[None].expand(BLOCK, hkv, max_tiles).contiguous()
    if quantised:
        ws = torch.empty(kv.kvarn_decode_workspace_size(cfg_dec, BLOCK, hq, hkv, max_tiles) // 4 + 4, device=dev)
    out = torch.empty(BLOCK, hq, HEAD, device=dev)
    tok_scale = None if kv_token_scale is None else kv_token_scale.to(device=dev, dtype=torch.float32)
    attn = []
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for j in range(n_blocks):
        h = x[j * BLOCK:(j + 1) * BLOCK].float()
        pos = torch.arange(j * BLOCK, (j + 1) * BLOCK, device=dev)
        per_layer = []
        for l, w in enumerate(weights):
            n = _rmsnorm(h)
            q = _rope((n @ w["wq"].float().T).reshape(BLOCK, hq, HEAD), pos).to(torch.bfloat16)
            k_proj = n @ w["wk"].float().T
            v_proj = n @ w["wv"].float().T
            if tok_scale is not None:
                ts = tok_scale[j * BLOCK:(j + 1) * BLOCK, None]
                k_proj, v_proj = k_proj * ts, v_proj * ts
            k = _rope(k_proj.reshape(BLOCK, hkv, HEAD), pos).to(torch.bfloat16)
            v = v_proj.reshape(BLOCK, hkv, HEAD).to(torch.bfloat16)
            if quantised:
                kc, kp, ks, vc, vp, vs = pools[l]
                lens = (j * BLOCK + 1 + torch.arange(BLOCK, device=dev, dtype=torch.int32)).contiguous()
                # the current block is every pseudo-sequence's tail: [128 seq][hkv][128 tok][128]
                k_tail = k.permute(1, 0, 2)[None].expand(BLOCK, hkv, BLOCK, HEAD).contiguous()
                v_tail = v.permute(1, 0, 2)[None].expand(BLOCK, hkv, BLOCK, HEAD).contiguous()
                kv.kvarn_decode_attention(cfg_dec, q.contiguous(), hkv, kc, kp, ks, vc, vp, vs, table, lens,
                                          k_tail, v_tail, scale, ws, out)
                a = out.clone()
                if capture is not None and (j, l) in capture:
                    capture[(j, l)] = dict(q=q.clone(), k_blk=k.clone(), v_blk=v.clone(), attn=a.clone(),
                                           pools=tuple(t[:j * hkv].clone() for t in pools[l]),
                                           n_prev_blocks=j)
                # the finished block enters the cache: one tile per kv head
                sl = slice(j * hkv, (j + 1) * hkv)
                kv.kvarn_encode_kv_blocks(cfg, k.permute(1, 0, 2).contiguous(), v.permute(1, 0, 2).contiguous(),
                                          kc[sl], kp[sl], ks[sl], vc[sl], vp[sl], vs[sl])
            else:
                ke, ve = exact[l]
                ke[j * BLOCK:(j + 1) * BLOCK] = k.float()
                ve[j * BLOCK:(j + 1) * BLOCK] = v.float()
                a = _exact_attention(q.float(), ke[:(j + 1) * BLOCK], ve[:(j + 1) * BLOCK], j * BLOCK, scale)
            per_layer.append(a)
            h = h + a.reshape(BLOCK, hq * HEAD) @ w["wo"].float().T
        attn.append(per_layer)
    torch.cuda.synchronize()
    seconds = time.perf_counter() - t0
    torch.backends.cuda.matmul.allow_tf32 = old_tf32
    return attn, seconds


def mae_curves(attn_q, attn_ref, relative: bool = False):
    """mae[j][l] = mean |attn_q - attn_ref| of block j, layer l (a nested list of floats); with
    relative=True divided by mean |attn_ref| of the same block and layer."""
    return [[float((a - b).abs().mean() / (b.abs().mean() if relative else 1.0)) for a, b in zip(rq, rr)]
            for rq, rr in zip(attn_q, attn_ref)]


def presets(kv):
    """The codecs the MAE curves compare: KVarN (2-bit and 4-bit K), rotation only, plain RTN."""
    return (("kvarn_k2v2", kv.kvarn_config_from_preset("kvarn_k2v2_g128")),
            ("kvarn_k4v2", kv.kvarn_config_from_preset("kvarn_k4v2_g128")),
            ("hadamard_k2v2 (rotation, no normalisation)", kv.kvarn_config_from_preset("hadamard_k2v2_g128")),
            ("rtn_k2v2 (no rotation, no normalisation)", kv.kvarn_config_from_preset("kivi_k2v2_g128")))


def main():
    """Config 4 (4 layers, 32q/8kv, hidden 4096, 64 blocks of 128 tokens, seed 4): MAE per block
    and layer of each codec's cache against the unquantised run.  --kv-outliers runs the variant
    whose K/V carry the outlier structure of the cache recipe (synthetic.pseudo_decode_weights,
    synthetic.pseudo_decode_token_scales)."""
    import argparse
    import json

    import bit_kv_cache_kvarn_gb300 as kv

    ap = argparse.ArgumentParser()
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--hidden", type=int, default=4096)
    ap.add_argument("--hq", type=int, default=32)
    ap.add_argument("--hkv", type=int, default=8)
    ap.add_argument("--blocks", type=int, default=64)
    ap.add_argument("--seed", type=int, default=4)
    ap.add_argument("--kv-outliers", action="store_true")
    args = ap.parse_args()
    kv.load()
    w = make_weights(args.seed, args.layers, args.hidden, args.hq, args.hkv, kv_outliers=args.kv_outliers)
    x = make_input(args.seed, args.blocks * BLOCK, args.hidden)
    ts = synthetic.pseudo_decode_token_scales(args.seed, args.blocks * BLOCK) if args.kv_outliers else None
    ref, t_ref = run(kv, None, w, x, args.hq, args.hkv, quantised=False, kv_token_scale=ts)
    res = {"config": vars(args), "reference_s": round(t_ref, 3)}
    for name, c in presets(kv):
        a, t = run(kv, c, w, x, args.hq, args.hkv, quantised=True, kv_token_scale=ts)
        res[name] = {"seconds": round(t, 3), "mae": mae_curves(a, ref),
                     "relative_mae": mae_curves(a, ref, relative=True)}
    assert kv.kvarn_device_error() == 0
    print(json.dumps(res))


if __name__ == "__main__":
    main()
