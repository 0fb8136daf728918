"""Pins for the fp64 oracle: each check is independent of the oracle's own code (a library
routine, a closed form, an invariant, brute force, or a figure the pages print), chosen so that a
dropped term, a wrong sign/index or a transposed operand in the oracle fails at least one."""
import os

import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import kvarn_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("--")[0].strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


def _outlier_tile(seed, t=128):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((t, 128))
    chan = np.exp(rng.standard_normal(128))
    chan[rng.choice(128, 4, replace=False)] *= 20
    tok = np.exp(0.5 * rng.standard_normal(t))
    tok[rng.choice(t, max(1, round(0.05 * t)), replace=False)] *= 8
    return x * chan[None, :] * tok[:, None]


# --- Hadamard ---------------------------------------------------------------------------------
@pytest.mark.parametrize("n", [2, 4, 16, 128])
def test_fwht_equals_sylvester_matrix_product(n):
    x = np.random.default_rng(n).standard_normal((5, n))
    h = scipy.linalg.hadamard(n) / np.sqrt(n)  # scipy builds the Sylvester matrix
    assert np.abs(o.fwht(x) - x @ h).max() <= 1e-13


def test_fwht_orthonormal_round_trip():
    x = _outlier_tile(1)
    assert np.abs(o.fwht(o.fwht(x)) - x).max() <= 1e-12 * np.abs(x).max()
    eye = o.fwht(np.eye(128))
    assert np.abs(eye @ eye.T - np.eye(128)).max() <= 1e-13
    assert np.abs(eye - eye.T).max() == 0.0  # symmetric


# --- number formats ---------------------------------------------------------------------------
def test_e4m3_round_matches_torch_cast():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.uniform(-460, 460, 400_000),
        np.exp(rng.uniform(np.log(2.0 ** -12), np.log(460.0), 600_000)) * rng.choice([-1, 1], 600_000),
        np.arange(-1024, 1025) * 2.0 ** -10,  # includes exact ties in the subnormal range
    ])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(o.e4m3_round(x), ref)


def test_e4m3_round_up_is_smallest_grid_value_above():
    grid = np.sort(torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn)
                   .to(torch.float64).numpy())
    x = np.concatenate([np.random.default_rng(30).uniform(0, 448, 50_000), grid])
    got = o.e4m3_round_up(x)
    assert np.array_equal(got, grid[np.searchsorted(grid, x, side="left")])


def test_e4m3_saturates_and_all_bytes_round_trip():
    assert o.e4m3_round(np.array([470.0, 1e6, -1e6]))[0] == 448.0
    assert o.e4m3_round(np.array([-1e6]))[0] == -448.0
    for b in range(256):
        if b & 0x7F == 0x7F:
            assert np.isnan(o.e4m3_decode(np.array([b]))[0])
            continue
        v = o.e4m3_decode(np.array([b]))[0]
        assert o.e4m3_round(np.array([v]))[0] == v
        if b < 0x80:
            assert int(o.e4m3_encode(np.array([v]))[0]) == b
    # a few values by hand: 1.0 = 0 0111 000, 448 = 0 1111 110, 2^-9 = 0 0000 001
    assert list(o.e4m3_encode(np.array([1.0, 448.0, 2.0 ** -9, 0.0]))) == [0x38, 0x7E, 0x01, 0x00]


def test_fp16_round_matches_torch_cast_and_brute_force():
    # torch casts float64 -> float16 through float32 (two roundings), so compare it on inputs
    # that are exactly float32; for float64 inputs compare with a brute-force nearest search.
    x32 = (np.random.default_rng(4).standard_normal(100_000) * 300).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.float16).to(torch.float64).numpy()
    assert np.array_equal(o.fp16_round(x32.astype(np.float64)), ref)
    grid = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)  # +finite
    x = np.abs(np.random.default_rng(5).standard_normal(20_000) * 300)
    x = np.concatenate([x, (grid[1:200] + grid[:199]) / 2])  # exact midpoints -> ties to even
    idx = np.clip(np.searchsorted(grid, x), 1, len(grid) - 1)
    lo, hi = grid[idx - 1], grid[idx]
    pick_hi = (hi - x < x - lo) | ((hi - x == x - lo) & (idx % 2 == 0))
    assert np.array_equal(o.fp16_round(x), np.where(pick_hi, hi, lo))


# --- normalisation ----------------------------------------------------------------------------
def test_normalization_fixed_point_balances_rows_and_columns():
    y = o.fwht(_outlier_tile(5))
    log_r, log_c = o.dual_axis_normalize(y, iters=200)
    z = y / np.exp(log_r)[:, None] / np.exp(log_c)[None, :]
    rs, cs = z.std(axis=1), z.std(axis=0)
    # Each axis is balanced.  With centred stds the common row level and the common column level
    # differ by a constant set by the row/column means (here ~0.3%), a gauge the quantiser
    # absorbs; the scaling r c^T itself is stationary.
    assert rs.max() / rs.min() - 1 <= 1e-3 and cs.max() / cs.min() - 1 <= 1e-3
    log_r2, log_c2 = o.dual_axis_normalize(y, iters=201)
    assert np.abs((log_r2[:, None] + log_c2[None, :]) - (log_r[:, None] + log_c[None, :])).max() < 1e-6
    # at 8 iterations (the pages' count) the residual imbalance is already small
    log_r8, log_c8 = o.dual_axis_normalize(y, iters=8)
    z8 = y / np.exp(log_r8)[:, None] / np.exp(log_c8)[None, :]
    assert z8.std(axis=1).max() / z8.std(axis=1).min() < 1.1


def test_normalization_recovers_separable_scales_closed_form():
    # Y = diag(a) S diag(b), S = +-1 block pattern whose rows and columns have mean 0 and std 1.
    # One token step gives r = a * k, then one channel step gives c = b / k, so r c^T = a b^T.
    rng = np.random.default_rng(6)
    a = np.exp(rng.standard_normal(128))
    b = np.exp(rng.standard_normal(128))
    s = np.kron(np.array([[1.0, -1.0], [-1.0, 1.0]]), np.ones((64, 64)))
    y = a[:, None] * s * b[None, :]
    for iters in (1, 8):
        log_r, log_c = o.dual_axis_normalize(y, iters)
        rc = np.exp(log_r)[:, None] * np.exp(log_c)[None, :]
        assert np.abs(rc / np.outer(a, b) - 1).max() <= 1e-12


def test_normalization_degenerate_rows_and_columns_keep_factor():
    y = np.zeros((128, 128))
    log_r, log_c = o.dual_axis_normalize(y, 8)
    assert not log_r.any() and not log_c.any()
    y = _outlier_tile(7)
    y[:, 3] = 0.0  # zero column
    y[10, :] = 0.0  # zero row
    log_r, log_c = o.dual_axis_normalize(y, 8)
    assert log_c[3] == 0.0 and log_r[10] == 0.0
    assert np.all(np.isfinite(log_r)) and np.all(np.isfinite(log_c))


def test_normalization_threshold_of_near_constant_rows_closed_form():
    # A row of two levels c and c + 1 with k of 128 entries at c + 1 has, in closed form,
    # variance f (1 - f) and mean square (c + f)^2 + f (1 - f), f = k / 128.  In the first token
    # step (all channel factors 1) the row's factor is its std when var / ms > 1e-5, else it stays 1
    # -- rows at 0.56x, 0.985x, 1.012x and 2.07x of the threshold land on the predicted sides.
    from tests import _tiles

    x, rows = _tiles.threshold_row_tile(1)
    y = x.float().double().numpy()
    log_r, _ = o.dual_axis_normalize(y, 1)
    for label, t in rows.items():
        c, k = _tiles.THRESHOLD_LEVELS[label]
        f = k / 128
        var, ms = f * (1 - f), (c + f) ** 2 + f * (1 - f)
        want = 0.5 * np.log(var) if var > 1e-5 * ms else 0.0
        assert (var > 1e-5 * ms) == (label in ("1.012x", "2.07x"))
        assert abs(log_r[t] - want) <= 1e-12, label


# --- encode -----------------------------------------------------------------------------------
@pytest.mark.parametrize("kind", ["K", "V"])
@pytest.mark.parametrize("bits", [2, 4])
def test_codes_equal_brute_force_nearest_level(kind, bits):
    e = o.encode_tile(_outlier_tile(8), kind, bits)
    y, s2, s1, z, g = e["Y"], e["s2"], e["S1"], e["Z"], e["g"]
    w = y / (s2[:, None] if kind == "K" else s2[None, :])
    grp_s1 = s1[None, :] if kind == "K" else s1[:, None]
    grp_z = z[None, :] if kind == "K" else z[:, None]
    levels = np.arange(2 ** bits)
    grid = grp_z[..., None] + grp_s1[..., None] * levels  # [t, j, level]
    dist = np.abs(w[..., None] / g - grid)
    best = dist.min(axis=-1, keepdims=True)
    # nearest level, ties to the even level
    cand = np.where(np.isclose(dist, best, rtol=0, atol=1e-12 * (1 + np.abs(grid))), levels, 10 ** 6)
    even_first = np.where(cand % 2 == 0, cand, cand + 10 ** 5)
    brute = np.min(even_first, axis=-1) % 10 ** 5
    assert np.array_equal(e["codes"].astype(np.int64), brute)


@pytest.mark.parametrize("kind", ["K", "V"])
def test_no_rotate_no_normalize_is_textbook_minmax_rtn(kind):
    # KIVI grouping: K per channel, V per token; asymmetric min/max RTN with scale/zero rounded
    # to the storage formats.
    x = _outlier_tile(9)
    e = o.encode_tile(x, kind, 2, rotate=False, normalize=False)
    grp = x.T if kind == "K" else x
    lo, hi = grp.min(axis=1), grp.max(axis=1)
    assert np.all(e["s2"] == 1.0)
    g = e["g"]
    # S1 = the smallest E4M3 value >= scale / g, found on the enumerated E4M3 grid
    grid = np.sort(torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn)
                   .to(torch.float64).numpy())
    want = grid[np.searchsorted(grid, (hi - lo) / 3 / g, side="left")]
    assert np.array_equal(e["S1"], want)
    assert np.array_equal(e["Z"], np.float16(lo / g).astype(np.float64))
    # g is the power of two that puts the largest scale in (128, 256] (|min|/g stays far below
    # FP16's limit here)
    assert 128 < ((hi - lo) / 3).max() / g <= 256 and np.abs(lo).max() / g <= 32768
    assert np.log2(g) == np.round(np.log2(g))


def test_token_permutation_equivariance():
    x = _outlier_tile(10)
    perm = np.random.default_rng(11).permutation(128)
    for kind in ("K", "V"):
        e1 = o.encode_tile(x, kind, 2)
        e2 = o.encode_tile(x[perm], kind, 2)
        assert np.array_equal(e2["codes"], e1["codes"][perm])
        if kind == "K":  # s2 per token follows the tokens; group params are unchanged
            assert np.array_equal(e2["s2"], e1["s2"][perm])
            assert np.allclose(e2["S1"], e1["S1"]) and np.allclose(e2["Z"], e1["Z"])
        else:  # groups are tokens
            assert np.array_equal(e2["S1"], e1["S1"][perm])


def test_power_of_two_scaling_is_exact():
    x = _outlier_tile(12)
    for kind in ("K", "V"):
        e1 = o.encode_tile(x, kind, 4)
        for k in (-40, 17):
            e2 = o.encode_tile(x * 2.0 ** k, kind, 4)
            assert np.array_equal(e1["codes"], e2["codes"])
            assert e2["g"] == e1["g"] * 2.0 ** k
            assert np.array_equal(e1["S1"], e2["S1"]) and np.array_equal(e1["Z"], e2["Z"])


def test_zero_and_constant_tiles():
    for kind in ("K", "V"):
        e = o.encode_tile(np.zeros((128, 128)), kind, 2)
        assert not e["codes"].any() and not e["S1"].any() and e["g"] == 1.0
        yh = o.dequant_tile(e["codes"], e["S1"], e["s2"], e["Z"], e["g"], kind, True)
        assert not yh.any()
        # constant tile without rotation reconstructs exactly (3.0 is an FP16 value)
        c = np.full((128, 128), 3.0)
        e = o.encode_tile(c, kind, 2, rotate=False)
        yh = o.dequant_tile(e["codes"], e["S1"], e["s2"], e["Z"], e["g"], kind)
        assert np.array_equal(yh, c)
        # with rotation, Y has one non-zero column; for K (groups = channels) it is a constant
        # group, stored in the FP16 zero-point alone: error <= half an FP16 ulp (relative 2^-11).
        # For V (groups = tokens) the E4M3 group scale carries it: error <= 1/16 relative.
        e = o.encode_tile(c, kind, 2)
        xh = o.dequant_tile(e["codes"], e["S1"], e["s2"], e["Z"], e["g"], kind, True)
        bound = 3.0 * 2.0 ** -11 if kind == "K" else 3.0 / 16
        assert np.abs(xh - c).max() <= bound


@pytest.mark.parametrize("kind", ["K", "V"])
def test_dequant_error_shrinks_with_bits(kind):
    x = _outlier_tile(13)
    errs = []
    for bits in (2, 4, 8, 16):
        e = o.encode_tile(x, kind, bits)
        xh = o.dequant_tile(e["codes"], e["S1"], e["s2"], e["Z"], e["g"], kind, True)
        errs.append(np.sqrt(np.mean((xh - x) ** 2)) / np.sqrt(np.mean(x ** 2)))
    # RTN error ~ range / 2^b: going from b to 2b bits divides it by ~2^b
    assert errs[1] < errs[0] / 3 and errs[2] < errs[1] / 10 and errs[3] < errs[2] / 100
    assert errs[3] < 1e-4
    # no element is clipped: every code reconstructs within half a step of W / g
    for bits in (2, 4, 8):
        e = o.encode_tile(x, kind, bits)
        u = e["u"]
        assert u.min() > -0.5 - 1e-9 and u.max() < 2 ** bits - 0.5


def test_pack_layout_by_hand():
    codes = np.zeros((128, 128), dtype=np.uint8)
    codes[0, 17] = 3  # channel 17 = 16*1 + 1 -> lane 1, bit offset 2*1 (2-bit) / 4*1 (4-bit)
    codes[1, 0] = 1   # row 1, lane 0, offset 0
    p2 = o.pack_codes(codes, 2).reshape(128, 32)
    assert p2[0, 2] == 0b1100 and p2[0].sum() == 0b1100 and p2[1, 0] == 1
    p4 = o.pack_codes(codes, 4).reshape(128, 64)
    assert p4[0, 4] == 0x30 and p4[0].sum() == 0x30 and p4[1, 0] == 1
    # V tiles are stored transposed: token 17 of channel 0 sits in row 0, lane 1, offset 2
    v = np.zeros((128, 128), dtype=np.uint8)
    v[17, 0] = 3
    pv = o.pack_tile(v, 2, "V").reshape(128, 32)
    assert pv[0, 2] == 0b1100 and pv.sum() == 0b1100
    rng = np.random.default_rng(14)
    for bits in (2, 4):
        c = rng.integers(0, 2 ** bits, (128, 128)).astype(np.uint8)
        assert np.array_equal(o.unpack_codes(o.pack_codes(c, bits), bits), c)
        for kind in ("K", "V"):
            assert np.array_equal(o.unpack_tile(o.pack_tile(c, bits, kind), bits, kind), c)


def test_bit_accounting_against_printed_figures():
    gold = _golden("bit_accounting.txt")
    group = gold["group_size"]
    # codes + two FP8 scales + one FP16 zero-point per group, as the page counts it
    assert 2 + (8 + 8 + 16) / group == gold["bits_per_element_2bit"]
    assert o.bits_per_element(2) - 32 / 16384 == gold["bits_per_element_2bit"]
    assert round(o.bits_per_element(2), 1) == gold["bits_per_element_table"]
    assert round(100 * (1 - gold["bits_per_element_table"] / gold["fp16_bits"]), 1) == gold["memory_reduction_percent"]
    # the byte sizes of the format give the same figure
    for bits in (2, 4):
        tile_bits = 8 * (128 * 16 * bits + 512 + 4)
        assert tile_bits / 16384 == o.bits_per_element(bits)


# --- attention --------------------------------------------------------------------------------
def test_attention_matches_sdpa():
    rng = np.random.default_rng(15)
    for L in (1, 7, 300):
        q, k, v = rng.standard_normal(128), rng.standard_normal((L, 128)) * 3, rng.standard_normal((L, 128))
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[None, None, None], torch.from_numpy(k)[None, None],
            torch.from_numpy(v)[None, None], scale=0.2)[0, 0, 0].numpy()
        assert np.abs(o.attention_single_query(q, k, v, 0.2) - ref).max() <= 1e-12


@pytest.mark.parametrize("full_tail", [False, True])
def test_decode_attention_gqa_and_tail_against_sdpa_on_dequantised_cache(full_tail):
    rng = np.random.default_rng(16)
    bsz, hq, hkv, max_tiles = 2, 4, 2, 3
    n_tiles = bsz * hkv * max_tiles
    tiles = np.stack([_outlier_tile(100 + i) for i in range(n_tiles)])
    kc, kp, ks, _ = o.encode_blocks(tiles, "K", 4)
    vtiles = np.stack([_outlier_tile(200 + i) for i in range(n_tiles)])
    vc, vp, vs, _ = o.encode_blocks(vtiles, "V", 2)
    table = rng.permutation(n_tiles).reshape(bsz, hkv, max_tiles)
    lens = np.array([2 * 128 + 57, 3 * 128])
    k_tail = rng.standard_normal((bsz, hkv, 128, 128))
    v_tail = rng.standard_normal((bsz, hkv, 128, 128))
    q = rng.standard_normal((bsz, hq, 128))
    out = o.decode_attention(q, hq, hkv, kc, kp, ks, vc, vp, vs, table, lens, k_tail, v_tail,
                             0.1, 4, 2, full_tail=full_tail)
    kd = o.dequant_blocks(kc, kp, ks, "K", 4, original_basis=True)
    vd = o.dequant_blocks(vc, vp, vs, "V", 2, original_basis=True)
    for b in range(bsz):
        for h in range(hq):
            kv = h // 2
            # full window: the last ((L - 1) mod 128) + 1 tokens come from the tail
            nfull = (lens[b] - 1) // 128 if full_tail else lens[b] // 128
            tail = lens[b] - 128 * nfull
            kk = np.concatenate([kd[table[b, kv, i]] for i in range(nfull)] + [k_tail[b, kv, :tail]])
            vv = np.concatenate([vd[table[b, kv, i]] for i in range(nfull)] + [v_tail[b, kv, :tail]])
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[b, h])[None, None, None], torch.from_numpy(kk)[None, None],
                torch.from_numpy(vv)[None, None], scale=0.1)[0, 0, 0].numpy()
            assert np.abs(out[b, h] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_decode_attention_tail_only_is_unquantised_attention():
    rng = np.random.default_rng(17)
    q = rng.standard_normal((1, 2, 128))
    k_tail = rng.standard_normal((1, 1, 128, 128))
    v_tail = rng.standard_normal((1, 1, 128, 128))
    empty = np.zeros((0, 4096), np.uint8)
    for L, full_tail in ((0, False), (1, False), (127, False), (0, True), (1, True), (128, True)):
        out = o.decode_attention(q, 2, 1, empty, np.zeros((0, 512), np.uint8), np.zeros(0),
                                 empty, np.zeros((0, 512), np.uint8), np.zeros(0),
                                 np.zeros((1, 1, 1), np.int64), np.array([L]), k_tail, v_tail,
                                 0.3, 2, 2, full_tail=full_tail)
        for h in range(2):
            if L == 0:
                assert not out[0, h].any()
                continue
            s = 0.3 * k_tail[0, 0, :L] @ q[0, h]
            p = np.exp(s - s.max())
            assert np.abs(out[0, h] - (p / p.sum()) @ v_tail[0, 0, :L]).max() <= 1e-12


# --- error diagnostics ------------------------------------------------------------------------
def test_error_decomposition_identity_and_special_cases():
    rng = np.random.default_rng(50)
    x = rng.standard_normal((300, 128)) * np.exp(rng.standard_normal((300, 1)))
    xh = x + 0.1 * rng.standard_normal((300, 128))
    e_m, e_d = o.error_decomposition(x, xh)
    total = np.sum((x - xh) ** 2, axis=1)
    # E_D cancels terms of size |x|^2, so the identity holds to rounding of |x|^2
    scale = np.sum(x * x, axis=1)
    assert np.all(np.abs(e_m + e_d - total) <= 1e-13 * scale)
    assert np.all(e_m >= 0) and np.all(e_d >= -1e-13 * scale)
    # a pure rescaling is all magnitude error; a rotation of equal length is all direction error
    e_m, e_d = o.error_decomposition(x, 1.5 * x)
    assert np.all(np.abs(e_d) <= 1e-13 * scale)
    assert np.allclose(e_m, 0.25 * np.sum(x * x, axis=1), rtol=1e-12)
    rot = np.concatenate([x[:, 1:], x[:, :1]], axis=1)  # a permutation keeps the norm
    e_m, e_d = o.error_decomposition(x, rot)
    assert np.all(e_m <= 1e-24 * scale ** 2 + 1e-30)


def test_magnitude_share_and_token_scale_ratio_by_hand():
    e_m = np.array([0.0, 1.0, 3.0, 0.5])
    e_d = np.array([1.0, 1.0, 1.0, 0.5])
    s = o.magnitude_share_of_top_errors(e_m, e_d, fractions=(0.25, 0.5, 1.0))
    assert s[0.25] == 3.0 / 4.0                     # the largest total error is row 2 (4.0)
    assert s[0.5] == (3.0 + 1.0) / (4.0 + 2.0)      # rows 2 and 1
    assert s[1.0] == 4.5 / 8.0
    x = np.array([[3.0, 4.0], [0.0, 0.0], [1.0, 0.0]])
    xh = np.array([[6.0, 8.0], [0.0, 1.0], [0.0, 0.5]])
    assert np.allclose(o.token_scale_ratio(x, xh), [2.0, 1.0, 0.5])


def test_decode_attention_with_sink_against_sdpa():
    # FP16 sink rows come first, then the dequantised body tiles, then the tail
    rng = np.random.default_rng(18)
    bsz, hq, hkv, max_tiles = 3, 2, 1, 2
    n_tiles = bsz * hkv * max_tiles
    kc, kp, ks, _ = o.encode_blocks(np.stack([_outlier_tile(300 + i) for i in range(n_tiles)]), "K", 2)
    vc, vp, vs, _ = o.encode_blocks(np.stack([_outlier_tile(400 + i) for i in range(n_tiles)]), "V", 2)
    table = rng.permutation(n_tiles).reshape(bsz, hkv, max_tiles)
    lens = np.array([20, 32 + 128 + 5, 32 + 2 * 128 + 100])
    k_sink, v_sink = rng.standard_normal((bsz, hkv, 128, 128)), rng.standard_normal((bsz, hkv, 128, 128))
    k_tail, v_tail = rng.standard_normal((bsz, hkv, 128, 128)), rng.standard_normal((bsz, hkv, 128, 128))
    q = rng.standard_normal((bsz, hq, 128))
    out = o.decode_attention(q, hq, hkv, kc, kp, ks, vc, vp, vs, table, lens, k_tail, v_tail, 0.1, 2, 2,
                             k_sink=k_sink, v_sink=v_sink, sink_len=32)
    kd = o.dequant_blocks(kc, kp, ks, "K", 2, original_basis=True)
    vd = o.dequant_blocks(vc, vp, vs, "V", 2, original_basis=True)
    for b in range(bsz):
        ns = min(32, lens[b])
        body = lens[b] - ns
        nfull, tail = body // 128, body % 128
        kk = np.concatenate([k_sink[b, 0, :ns]] + [kd[table[b, 0, i]] for i in range(nfull)] + [k_tail[b, 0, :tail]])
        vv = np.concatenate([v_sink[b, 0, :ns]] + [vd[table[b, 0, i]] for i in range(nfull)] + [v_tail[b, 0, :tail]])
        for h in range(hq):
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[b, h])[None, None, None], torch.from_numpy(kk)[None, None],
                torch.from_numpy(vv)[None, None], scale=0.1)[0, 0, 0].numpy()
            assert np.abs(out[b, h] - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


@pytest.mark.parametrize("full_tail", [False, True])
def test_append_tokens_rebuilds_the_same_cache_as_one_shot(full_tail):
    # appending a token stream in random chunks gives the same tails and the same completed blocks
    # as cutting the whole stream at once
    rng = np.random.default_rng(60)
    total, hkv = 700, 2
    stream_k = rng.standard_normal((1, hkv, total, 128))
    stream_v = rng.standard_normal((1, hkv, total, 128))
    table = np.arange(8 * hkv).reshape(1, hkv, 8)
    lens = np.array([0])
    kt, vt = np.zeros((1, hkv, 128, 128)), np.zeros((1, hkv, 128, 128))
    got_blocks = {}
    pos = 0
    while pos < total:
        n_new = int(rng.integers(1, 129))
        acc = int(rng.integers(0, n_new + 1))
        acc = min(acc, total - pos)
        kn = np.zeros((1, hkv, n_new, 128))
        vn = np.zeros((1, hkv, n_new, 128))
        kn[:, :, :acc] = stream_k[:, :, pos:pos + acc]
        vn[:, :, :acc] = stream_v[:, :, pos:pos + acc]
        kn[:, :, acc:] = 1e9  # offered but rejected tokens must never enter the cache
        lens, kt, vt, blocks = o.append_tokens(kn, vn, [acc], lens, kt, vt, table, full_tail)
        for b, h, tile, kb, vb in blocks:
            assert tile not in got_blocks
            got_blocks[tile] = (kb, vb)
        pos += acc
    assert lens[0] == total
    n_full = ((total - 1) // 128 if full_tail else total // 128)
    assert sorted(got_blocks) == sorted(int(table[0, h, i]) for h in range(hkv) for i in range(n_full))
    for h in range(hkv):
        for i in range(n_full):
            kb, vb = got_blocks[int(table[0, h, i])]
            assert np.array_equal(kb, stream_k[0, h, 128 * i:128 * (i + 1)])
            assert np.array_equal(vb, stream_v[0, h, 128 * i:128 * (i + 1)])
        tail = total - 128 * n_full
        assert np.array_equal(kt[0, h, :tail], stream_k[0, h, 128 * n_full:])
        assert np.array_equal(vt[0, h, :tail], stream_v[0, h, 128 * n_full:])
