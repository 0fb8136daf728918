"""fp64 CPU oracle for the KVarN KV-cache codec.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this module.  The CUDA product path never
calls it and shares no code, table or constant generator with it.

Plain, slow and meant to be checked by eye against the pages describing KVarN
(arXiv:2606.03458).  Sources are cited by page and section:

  [paperlayer]   paperlayer.ai source-linked summary of arXiv v1 ("KVarN: Variance-Normalized
                 KV-Cache Quantization Mitigates Error Accumulation in Reasoning Tasks").
  [dimensionstp] dimensionstp.github.io review of the paper and its README.
  [agihunt]      agihunt.info summary of arXiv:2606.03458.
  [pheeree]      pheeree.github.io blog post (quotes the paper's sections in its footnotes).

Everything is fp64 except where the format itself fixes the precision (FP8 E4M3 scales, FP16
zero-points, integer codes).  Where the pages leave a step open the reading taken is stated in
the function's docstring.  Parity pins for each function live in tests/test_oracle_*.py.
"""
from __future__ import annotations

import numpy as np

TILE = 128  # tokens per tile and channels per head ([paperlayer] "2 Preliminaries": 128 x 128)
DEFAULT_ITERS = 8  # [paperlayer] "4 Experiments", Efficiency: eight normalisation iterations
DEGENERATE_REL = 1e-5  # a row/column whose variance <= 1e-5 * mean square is treated as constant
E4M3_MAX = 448.0
E4M3_MIN_SUBNORMAL = 2.0 ** -9


# ----------------------------------------------------------------------------------------------
# Hadamard rotation
# ----------------------------------------------------------------------------------------------
def fwht(x: np.ndarray) -> np.ndarray:
    """Orthonormal Walsh-Hadamard transform along the last axis: returns x @ H.

    H[i, j] = (-1)^popcount(i & j) / sqrt(n) (Sylvester natural order).  The pages ask for a
    channel-wise orthonormal Hadamard rotation with O(N log N) cost ([paperlayer] "2 Preliminaries",
    "A Hadamard Transform Arrangement"; [dimensionstp] "3-2 (2) Hadamard rotation"); they fix
    neither the row order nor the scaling, so the reading is the Sylvester order, scaled to be
    orthonormal.  Computed with butterflies: stage s pairs indices that differ only in bit s.
    """
    y = np.array(x, dtype=np.float64, copy=True)
    n = y.shape[-1]
    assert n > 0 and (n & (n - 1)) == 0, "length must be a power of two"
    lead = y.shape[:-1]
    h = 1
    while h < n:
        y = y.reshape(*lead, n // (2 * h), 2, h)
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(*lead, n)
        h *= 2
    return y / np.sqrt(n)


# ----------------------------------------------------------------------------------------------
# Number formats (written from the format definitions)
# ----------------------------------------------------------------------------------------------
def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest FP8 E4M3 value (OCP 'e4m3fn': bias 7, 3 mantissa bits, largest
    finite 448, subnormal step 2^-9), ties to even, saturating to +-448 ("satfinite").

    The pages say the scales are FP8 ([paperlayer] "D Experimental details"; [agihunt]); the FP8
    variant is not named, so the reading is E4M3, the variant with the finer mantissa.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)  # a = m * 2^e with m in [0.5, 1): floor(log2 a) = e - 1 for a > 0
    expo = np.maximum(e - 1, -6)  # below 2^-6 the quantum stays that of the subnormal range
    quantum = np.ldexp(1.0, expo - 3)
    r = np.rint(a / quantum) * quantum  # np.rint rounds half to even
    r = np.where(a == 0, 0.0, r)
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)


def e4m3_round_up(x: np.ndarray) -> np.ndarray:
    """Smallest E4M3 value >= x, for 0 <= x <= 448 (the group scale's rounding; see encode_tile)."""
    a = np.asarray(x, dtype=np.float64)
    assert np.all(a >= 0) and np.all(a <= E4M3_MAX)
    _, e = np.frexp(a)
    quantum = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
    return np.where(a == 0, 0.0, np.ceil(a / quantum) * quantum)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Bytes of non-negative values that already lie on the E4M3 grid (see e4m3_round)."""
    v = np.asarray(v, dtype=np.float64)
    assert np.all(v >= 0) and np.all(v <= E4M3_MAX)
    out = np.zeros(v.shape, dtype=np.uint8)
    _, e = np.frexp(v)
    normal = v >= 2.0 ** -6
    expo_field = np.where(normal, (e - 1) + 7, 0)
    mant = np.where(normal, (v / np.ldexp(1.0, e - 1) - 1.0) * 8.0, v / E4M3_MIN_SUBNORMAL)
    assert np.all(mant == np.rint(mant)), "value not on the E4M3 grid"
    out[...] = (expo_field.astype(np.int64) << 3) | mant.astype(np.int64)
    return out


def e4m3_decode(b: np.ndarray) -> np.ndarray:
    """Values of E4M3 bytes (sign bit honoured; the NaN pattern 0x7F/0xFF gives NaN)."""
    b = np.asarray(b, dtype=np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    ef = (b >> 3) & 0xF
    mf = b & 0x7
    val = np.where(ef == 0, mf * E4M3_MIN_SUBNORMAL, np.ldexp(1.0 + mf / 8.0, ef - 7))
    val = np.where((b & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def fp16_round(x: np.ndarray) -> np.ndarray:
    """Round to IEEE binary16, ties to even (numpy's cast), returned as fp64."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


# ----------------------------------------------------------------------------------------------
# Dual-axis variance normalisation
# ----------------------------------------------------------------------------------------------
def dual_axis_normalize(y: np.ndarray, iters: int = DEFAULT_ITERS, trace: list | None = None):
    """Sinkhorn-Knopp style alternating standard-deviation normalisation in the log domain.

    Returns (log_r, log_c): log token factors (one per row) and log channel factors (one per
    column) such that y / (r c^T) has balanced row and column standard deviations.

    Pages: the normalisation alternates row-wise and column-wise standard-deviation
    normalisation in log space ([dimensionstp] "3-2 (3) Dual-axis variance normalization";
    [pheeree] "핵심 세 가지" §3: column and row variances are matched alternately, Sinkhorn
    style, adapted to a log-domain iteration); it runs eight iterations ([paperlayer]
    "4 Experiments", Efficiency); it acts on signed matrices, so magnitude-based normalisation
    is unsuitable ([paperlayer] "3 Methods").  Readings where the pages are silent:
      * one iteration = a token (row) step followed by a channel (column) step;
      * "standard deviation" is the centred population std (ddof = 0);
      * factors start at 1 and each step adds log(sigma) of the currently normalised matrix;
      * a row/column whose variance is <= DEGENERATE_REL times its mean square (including an
        all-zero one) is treated as constant: its factor is left unchanged.
    trace: optional list; each step appends ("token" | "channel", iteration, var / ms) so a test can
    see how far each row's or column's degeneracy decision is from the threshold.
    """
    y = np.asarray(y, dtype=np.float64)
    log_r = np.zeros(y.shape[0])
    log_c = np.zeros(y.shape[1])
    for it in range(iters):
        # token step: each row's std over channels
        z = y / np.exp(log_r)[:, None] / np.exp(log_c)[None, :]
        var = z.var(axis=1)
        ms = (z * z).mean(axis=1)
        ok = var > DEGENERATE_REL * ms
        if trace is not None:
            with np.errstate(divide="ignore", invalid="ignore"):
                trace.append(("token", it, var / ms))
        log_r[ok] += 0.5 * np.log(var[ok])
        # channel step: each column's std over tokens
        z = y / np.exp(log_r)[:, None] / np.exp(log_c)[None, :]
        var = z.var(axis=0)
        ms = (z * z).mean(axis=0)
        ok = var > DEGENERATE_REL * ms
        if trace is not None:
            with np.errstate(divide="ignore", invalid="ignore"):
                trace.append(("channel", it, var / ms))
        log_c[ok] += 0.5 * np.log(var[ok])
    return log_r, log_c


# ----------------------------------------------------------------------------------------------
# Tile encode / decode
# ----------------------------------------------------------------------------------------------
def _ceil_log2(v: float) -> int:
    frac, e = np.frexp(v)  # v = frac * 2^e, frac in [0.5, 1)
    return int(e - 1) if frac == 0.5 else int(e)


def tile_factor(s_max: float, m_max: float) -> float:
    """The per-tile power of two g (see encode_tile step 5)."""
    expo = []
    if s_max > 0:
        expo.append(_ceil_log2(s_max) - 8)
    if m_max > 0:
        expo.append(_ceil_log2(m_max) - 15)
    return float(np.ldexp(1.0, max(expo))) if expo else 1.0


def encode_tile(x: np.ndarray, kind: str, bits: int, iters: int = DEFAULT_ITERS,
                rotate: bool = True, normalize: bool = True, forced: dict | None = None) -> dict:
    """Encode one 128 x 128 tile (rows = tokens, columns = channels) of K (kind 'K') or V ('V').

    Steps, in the order the pages give them ([agihunt] pipeline paragraph; [paperlayer]
    "3 Methods"; [dimensionstp] "2-2 Design intuition": X -> HX -> D_r HX D_c -> Q_b):
      1. Y = X H (channel-wise rotation), unless rotate is False.
      2. (log_r, log_c) = dual_axis_normalize(Y, iters), unless normalize is False.
      3. Scale split.  Groups follow KIVI: K per channel, V per token ([paperlayer]
         "2 Preliminaries").  The group-axis factor is absorbed into each group's scale and
         zero-point ([agihunt]: the normalisation factors are absorbed into a high-precision
         per-group scale); it cancels exactly in the group's min/max, so it is not stored.
         The other-axis factor becomes the second FP8 scale s2 ([paperlayer] "I KVarN
         Dequantization Overhead": a per-row second scale s2).  Reading: s2 is normalised to
         geometric mean 1 over the tile, rounded to E4M3 and clamped to [2^-9, 448].
      4. W = Y / s2 (broadcast over the other axis).  Asymmetric min/max round-to-nearest per
         group ([dimensionstp] "3-2 (4) Low-bit quantization"): m = min W, M = max W,
         S = (M - m) / (2^b - 1); no clipping.
      5. Tile factor g = 2^max(ceil(log2 S_max) - 8, ceil(log2 m_max) - 15), where S_max is the
         largest group scale and m_max the largest |m| (a zero quantity drops out; g = 1 if both
         are zero).  This factor is the library's own (the pages leave the range of the FP8
         scale and FP16 zero open): it puts the largest S/g in (128, 256], inside E4M3's normal
         range and below its 448 limit, unless that would push |m|/g above 32768, next to
         FP16's 65504 limit.  Z = FP16(m / g) (round to nearest).  S1 = S / g rounded UP to the
         E4M3 grid.  The pages do not say how the FP8 scale is rounded; rounding up keeps
         (M/g - Z)/S1 <= 2^b - 1, so a group's extreme value is never clipped (round-to-nearest
         can shrink the step by up to 1/16 and clip the top value by up to a full code step at
         4 bits), and those extreme values are the outliers the paper finds matter most
         ([paperlayer] "C Outlier Contributions to MSE").
      6. u = (W / g - Z) / S1; code = clamp(round_half_even(u), 0, 2^b - 1); code = 0 where
         S1 = 0.
    Returns the codes [token, channel] (uint8), the stored parameters (as the values the format
    holds) and the unrounded quantities the parity tests use to recognise rounding ties.

    forced: optional {"s2", "S1", "Z", "g"} values that replace the computed ones from that step
    on (teacher forcing, so a parity test can compare each later step on identical inputs).
    """
    forced = forced or {}
    assert kind in ("K", "V") and bits in (2, 4, 8, 16)
    x = np.asarray(x, dtype=np.float64)
    assert x.shape == (TILE, TILE)
    y = fwht(x) if rotate else x.copy()
    if normalize:
        log_r, log_c = dual_axis_normalize(y, iters)
    else:
        log_r, log_c = np.zeros(TILE), np.zeros(TILE)
    log_other = log_r if kind == "K" else log_c
    s2_raw = np.exp(log_other - log_other.mean())  # geometric mean 1
    s2 = np.clip(e4m3_round(s2_raw), E4M3_MIN_SUBNORMAL, E4M3_MAX)
    if "s2" in forced:
        s2 = np.asarray(forced["s2"], dtype=np.float64)
    if kind == "K":
        w = y / s2[:, None]  # token factor divides each row; groups are columns
        wg = w.T  # [group, element]
    else:
        w = y / s2[None, :]  # channel factor divides each column; groups are rows
        wg = w
    levels = 2 ** bits - 1
    m = wg.min(axis=1)
    mx = wg.max(axis=1)
    scale = (mx - m) / levels
    g = tile_factor(scale.max(), np.abs(m).max())
    if "g" in forced:
        g = float(forced["g"])
    s1_raw = scale / g
    z_raw = m / g
    s1 = e4m3_round_up(s1_raw) if "S1" not in forced else np.asarray(forced["S1"], np.float64)
    z = fp16_round(z_raw) if "Z" not in forced else np.asarray(forced["Z"], np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        u = (wg / g - z[:, None]) / s1[:, None]
    u = np.where(s1[:, None] > 0, u, 0.0)
    codes_g = np.clip(np.rint(u), 0, levels).astype(np.int64)
    codes = codes_g.T if kind == "K" else codes_g
    u_tc = u.T if kind == "K" else u
    return {
        "codes": codes.astype(np.uint16 if bits > 8 else np.uint8),
        "S1": s1, "s2": s2, "Z": z, "g": g,
        "u": u_tc, "s2_raw": s2_raw, "S1_raw": s1_raw, "Z_raw": z_raw,
        "log_r": log_r, "log_c": log_c, "Y": y,
    }


def dequant_tile(codes: np.ndarray, s1, s2, z, g: float, kind: str,
                 original_basis: bool = False, rotate: bool = True) -> np.ndarray:
    """Yhat[t, j] = g * s2[other] * (S1[group] * code[t, j] + Z[group]); optionally Yhat H.

    Both scales are applied in the same dequantisation ([paperlayer] "I KVarN Dequantization
    Overhead": s2 is fused into the dequantisation kernel).  Since H is symmetric and
    orthonormal, X = Y H^T = Y H, so the original basis is one more forward transform.
    """
    c = np.asarray(codes, dtype=np.float64)
    s1 = np.asarray(s1, dtype=np.float64)
    s2 = np.asarray(s2, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    if kind == "K":
        yhat = g * s2[:, None] * (s1[None, :] * c + z[None, :])
    else:
        yhat = g * s2[None, :] * (s1[:, None] * c + z[:, None])
    if original_basis and rotate:
        yhat = fwht(yhat)
    return yhat


# ----------------------------------------------------------------------------------------------
# Byte layout of a packed tile (the library's format; the pages fix only the accounting)
# ----------------------------------------------------------------------------------------------
def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """[128 rows, 128 columns] codes -> [128 * 16 * bits] bytes.

    Each row is 16 little-endian lanes of `bits` bytes; the code of column j = 16 i + h goes to
    lane h at bit offset bits * i.  (K tiles are packed with rows = tokens, V tiles with rows =
    channels; see pack_tile.)
    """
    assert bits in (2, 4)
    codes = np.asarray(codes, dtype=np.uint64)
    lanes = np.zeros((TILE, 16), dtype=np.uint64)
    for j in range(TILE):
        h, i = j % 16, j // 16
        lanes[:, h] |= codes[:, j] << np.uint64(bits * i)
    dtype = np.dtype("<u2") if bits == 2 else np.dtype("<u4")
    return lanes.astype(dtype).view(np.uint8).reshape(-1)


def unpack_codes(packed: np.ndarray, bits: int) -> np.ndarray:
    """Inverse of pack_codes."""
    assert bits in (2, 4)
    dtype = np.dtype("<u2") if bits == 2 else np.dtype("<u4")
    lanes = np.asarray(packed, dtype=np.uint8).reshape(-1).view(dtype).reshape(TILE, 16)
    lanes = lanes.astype(np.uint64)
    codes = np.zeros((TILE, TILE), dtype=np.uint8)
    mask = np.uint64((1 << bits) - 1)
    for j in range(TILE):
        h, i = j % 16, j // 16
        codes[:, j] = (lanes[:, h] >> np.uint64(bits * i)) & mask
    return codes


def pack_params(s1, s2, z) -> np.ndarray:
    """S1 (E4M3 bytes) || s2 (E4M3 bytes) || Z (little-endian FP16) -> 512 bytes."""
    out = np.zeros(512, dtype=np.uint8)
    out[0:128] = e4m3_encode(np.asarray(s1))
    out[128:256] = e4m3_encode(np.asarray(s2))
    out[256:512] = np.asarray(z, dtype=np.float64).astype("<f2").view(np.uint8)
    return out


def unpack_params(p: np.ndarray):
    p = np.asarray(p, dtype=np.uint8).reshape(512)
    s1 = e4m3_decode(p[0:128])
    s2 = e4m3_decode(p[128:256])
    z = p[256:512].copy().view("<f2").astype(np.float64)
    return s1, s2, z


def bits_per_element(bits: int) -> float:
    """Storage per element: codes + S1 (8 bits) + s2 (8 bits) + Z (16 bits) per 128-element
    group + the 32-bit tile factor per 16384 elements.  The paper counts 2 + (8+8+16)/128 = 2.25
    for 2-bit codes ([paperlayer] "D Experimental details")."""
    return bits + (8 + 8 + 16) / 128 + 32 / (TILE * TILE)


def pack_tile(codes: np.ndarray, bits: int, kind: str) -> np.ndarray:
    """Packed bytes of one tile's codes [token, channel]: K rows are tokens; V rows are channels
    (the V tile is stored transposed, so a row holds one channel's 128 tokens)."""
    return pack_codes(codes if kind == "K" else np.asarray(codes).T, bits)


def unpack_tile(packed: np.ndarray, bits: int, kind: str) -> np.ndarray:
    """Inverse of pack_tile: codes [token, channel]."""
    c = unpack_codes(packed, bits)
    return c if kind == "K" else c.T.copy()


def encode_blocks(x_tiles: np.ndarray, kind: str, bits: int, iters: int = DEFAULT_ITERS,
                  rotate: bool = True, normalize: bool = True):
    """Encode [n, 128, 128] tiles; returns (codes [n, 16*bits*128] bytes, params [n, 512],
    tile_scale [n] float32, per-tile encode dicts)."""
    x_tiles = np.asarray(x_tiles, dtype=np.float64)
    n = x_tiles.shape[0]
    code_bytes = TILE * 16 * bits  # 128 rows x 16 lanes x `bits` bytes
    codes = np.zeros((n, code_bytes), dtype=np.uint8)
    params = np.zeros((n, 512), dtype=np.uint8)
    scale = np.zeros(n, dtype=np.float32)
    infos = []
    for k in range(n):
        e = encode_tile(x_tiles[k], kind, bits, iters, rotate, normalize)
        codes[k] = pack_tile(e["codes"], bits, kind)
        params[k] = pack_params(e["S1"], e["s2"], e["Z"])
        scale[k] = e["g"]
        infos.append(e)
    return codes, params, scale, infos


def dequant_blocks(codes: np.ndarray, params: np.ndarray, tile_scale: np.ndarray, kind: str,
                   bits: int, original_basis: bool = False, rotate: bool = True) -> np.ndarray:
    """[n] packed tiles -> [n, 128, 128] fp64."""
    n = codes.shape[0]
    out = np.zeros((n, TILE, TILE))
    for k in range(n):
        c = unpack_tile(codes[k], bits, kind)
        s1, s2, z = unpack_params(params[k])
        out[k] = dequant_tile(c, s1, s2, z, float(tile_scale[k]), kind, original_basis, rotate)
    return out


# ----------------------------------------------------------------------------------------------
# Decode attention over the packed cache
# ----------------------------------------------------------------------------------------------
def attention_single_query(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """softmax(scale * q k^T) v for one query q [d] over keys k [L, d], values v [L, d].
    Length 0 gives zeros (the library's convention for an empty context)."""
    q = np.asarray(q, dtype=np.float64)
    if k.shape[0] == 0:
        return np.zeros(q.shape[-1])
    s = scale * (np.asarray(k, dtype=np.float64) @ q)
    p = np.exp(s - s.max())
    return (p / p.sum()) @ np.asarray(v, dtype=np.float64)


def gather_cache(k_codes, k_params, k_scale, v_codes, v_params, v_scale, tile_ids, length,
                 k_tail, v_tail, k_bits, v_bits, rotate=True, full_tail=False):
    """Rebuild one (sequence, kv head)'s keys and values in the original basis, fp64:
    dequantised full tiles (in block-table order) followed by the unquantised tail rows.

    The tail holds the tokens after the last full tile (L mod 128 of them), or with full_tail a
    whole FP16 recent window of the last ((L - 1) mod 128) + 1 tokens ([paperlayer] "D
    Experimental details": the most recent tokens stay in FP16, R = 128)."""
    n_full = ((length - 1) // TILE if length > 0 else 0) if full_tail else length // TILE
    tail = length - n_full * TILE
    ks, vs = [], []
    for i in range(n_full):
        t = int(tile_ids[i])
        ks.append(dequant_blocks(k_codes[t:t + 1], k_params[t:t + 1], k_scale[t:t + 1], "K",
                                 k_bits, original_basis=True, rotate=rotate)[0])
        vs.append(dequant_blocks(v_codes[t:t + 1], v_params[t:t + 1], v_scale[t:t + 1], "V",
                                 v_bits, original_basis=True, rotate=rotate)[0])
    ks.append(np.asarray(k_tail, dtype=np.float64)[:tail])
    vs.append(np.asarray(v_tail, dtype=np.float64)[:tail])
    return np.concatenate(ks, axis=0), np.concatenate(vs, axis=0)


def decode_attention(q, hq: int, hkv: int, k_codes, k_params, k_scale, v_codes, v_params,
                     v_scale, block_table, seq_lens, k_tail, v_tail, softmax_scale: float,
                     k_bits: int, v_bits: int, rotate: bool = True, pairs=None,
                     full_tail: bool = False, k_sink=None, v_sink=None, sink_len: int = 0):
    """Decode attention over the packed cache, plain definition in the original basis.

    For query head h of sequence b, kv head = h // (hq // hkv) (grouped-query attention); keys
    and values are the dequantised tiles followed by the unquantised tail
    ([paperlayer] "D Experimental details": the most recent tokens stay in FP16).  Rotating the
    query instead of the keys gives the same scores because H is orthonormal
    ([paperlayer] "A Hadamard Transform Arrangement").
    q: [B, hq, 128]; block_table: [B, hkv, max_tiles]; tails: [B, hkv, 128, 128].
    pairs: optional list of (b, h) to compute (others stay NaN), for sampled checks.
    With sink_len > 0 the first min(sink_len, L) tokens are FP16 sink rows (k_sink, v_sink:
    [B, hkv, 128, 128]) and the block table and tail describe the remaining body ([paperlayer] "D
    Experimental details": FP16 sink tokens before the quantised body).
    """
    q = np.asarray(q, dtype=np.float64)
    bsz = q.shape[0]
    group = hq // hkv
    out = np.full((bsz, hq, TILE), np.nan)
    want = set(pairs) if pairs is not None else None
    for b in range(bsz):
        for kv in range(hkv):
            heads = [kv * group + g for g in range(group)]
            if want is not None and not any((b, h) in want for h in heads):
                continue
            n_sink = min(sink_len, int(seq_lens[b]))
            kk, vv = gather_cache(k_codes, k_params, k_scale, v_codes, v_params, v_scale,
                                  block_table[b, kv], int(seq_lens[b]) - n_sink, k_tail[b, kv],
                                  v_tail[b, kv], k_bits, v_bits, rotate, full_tail)
            if n_sink:
                kk = np.concatenate([np.asarray(k_sink[b, kv], dtype=np.float64)[:n_sink], kk], axis=0)
                vv = np.concatenate([np.asarray(v_sink[b, kv], dtype=np.float64)[:n_sink], vv], axis=0)
            for h in heads:
                if want is None or (b, h) in want:
                    out[b, h] = attention_single_query(q[b, h], kk, vv, softmax_scale)
    return out


# ----------------------------------------------------------------------------------------------
# Error diagnostics
# ----------------------------------------------------------------------------------------------
def error_decomposition(x: np.ndarray, x_hat: np.ndarray):
    """Per-row split of the squared reconstruction error into a magnitude and a direction part,
    ||x - x_hat||^2 = (||x|| - ||x_hat||)^2 + 2 ||x|| ||x_hat|| (1 - cos theta)  -- an identity
    ([pheeree] "핵심 세 가지" §2, E_M and E_D).  x, x_hat: [T, d]; returns (E_M, E_D), each [T]."""
    x = np.asarray(x, dtype=np.float64)
    x_hat = np.asarray(x_hat, dtype=np.float64)
    n = np.linalg.norm(x, axis=1)
    nh = np.linalg.norm(x_hat, axis=1)
    e_m = (n - nh) ** 2
    e_d = 2.0 * (n * nh - np.sum(x * x_hat, axis=1))  # 2 |x| |x_hat| (1 - cos theta)
    return e_m, e_d


def magnitude_share_of_top_errors(e_m, e_d, fractions=(0.5, 0.1, 0.05, 0.01, 0.001)):
    """For the rows with the largest total error (top fraction f of rows, at least one): the share
    of their summed error that is magnitude error, sum E_M / sum (E_M + E_D) ([pheeree] "핵심 세
    가지" §2: the share grows toward the largest errors)."""
    e_m = np.asarray(e_m, dtype=np.float64)
    tot = e_m + np.asarray(e_d, dtype=np.float64)
    order = np.argsort(-tot, kind="stable")
    out = {}
    for f in fractions:
        top = order[:max(1, int(round(f * tot.size)))]
        s = tot[top].sum()
        out[f] = float(e_m[top].sum() / s) if s > 0 else 0.0
    return out


def token_scale_ratio(x: np.ndarray, x_hat: np.ndarray) -> np.ndarray:
    """||x_hat_t|| / ||x_t|| per row t: how well the token's scale survives quantisation
    ([paperlayer] "B Full Token-Scale Distribution Error")."""
    n = np.linalg.norm(np.asarray(x, dtype=np.float64), axis=1)
    nh = np.linalg.norm(np.asarray(x_hat, dtype=np.float64), axis=1)
    return np.where(n > 0, nh / np.where(n > 0, n, 1.0), 1.0)


# ----------------------------------------------------------------------------------------------
# Appending tokens to the cache
# ----------------------------------------------------------------------------------------------
def append_tokens(k_new, v_new, n_accept, seq_lens, k_tail, v_tail, block_table, full_tail=False):
    """Commit the first n_accept[b] of the offered tokens of each sequence to its cache.

    The newest tokens stay unquantised in the tail; a 128-token block is quantised once it is
    complete ([paperlayer] "D Experimental details": quantised body, FP16 trailing tokens;
    [agihunt] pipeline paragraph: a block is quantised once it is done).  With the default
    convention a block is complete when it holds 128 tokens; with full_tail it stays in the tail
    until a newer token arrives (the full FP16 window of 1..128 tokens).  Only accepted tokens are
    committed (speculative decoding keeps the rest out of the cache).
    k_new, v_new: [B, hkv, n_new, 128]; tails: [B, hkv, 128, 128] (updated copies returned).
    Returns (seq_lens', k_tail', v_tail', blocks) with blocks a list of (b, kv head, pool tile id,
    k_block [128, 128], v_block [128, 128]) -- the blocks to encode into the pools."""
    k_tail, v_tail = np.array(k_tail, copy=True), np.array(v_tail, copy=True)
    lens = np.array(seq_lens, dtype=np.int64, copy=True)
    blocks = []
    bsz, hkv, n_new = k_new.shape[0], k_new.shape[1], k_new.shape[2]
    for b in range(bsz):
        a = int(min(max(int(n_accept[b]), 0), n_new))
        length = int(lens[b])
        if full_tail:
            t0 = ((length - 1) % TILE) + 1 if length > 0 else 0
            blk = (length - 1) // TILE if length > 0 else 0
            complete = t0 + a > TILE
        else:
            t0, blk = length % TILE, length // TILE
            complete = t0 + a >= TILE
        need = TILE - t0 if complete else a
        for h in range(hkv):
            if complete:
                kb = np.concatenate([k_tail[b, h, :t0], k_new[b, h, :need]], axis=0)
                vb = np.concatenate([v_tail[b, h, :t0], v_new[b, h, :need]], axis=0)
                blocks.append((b, h, int(block_table[b, h, blk]), kb, vb))
                k_tail[b, h, :a - need] = k_new[b, h, need:a]
                v_tail[b, h, :a - need] = v_new[b, h, need:a]
            else:
                k_tail[b, h, t0:t0 + a] = k_new[b, h, :a]
                v_tail[b, h, t0:t0 + a] = v_new[b, h, :a]
        lens[b] = length + a
    return lens, k_tail, v_tail, blocks
