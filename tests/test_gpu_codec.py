"""GPU encode / dequant parity with the fp64 oracle, through the C-ABI."""
import numpy as np
import pytest
import torch

from oracle import kvarn_oracle as o
from tests._parity import compare_encode, rel_l2

pytestmark = pytest.mark.gpu


def _encode_gpu(kv, cfg, kind, x_tiles):
    n = x_tiles.shape[0]
    bits = cfg.k_bits if kind == kv.KVARN_KIND_K else cfg.v_bits
    codes = torch.empty(n, 128 * 16 * bits, dtype=torch.uint8, device="cuda")
    params = torch.empty(n, 512, dtype=torch.uint8, device="cuda")
    scale = torch.empty(n, dtype=torch.float32, device="cuda")
    kv.kvarn_encode_blocks(cfg, kind, x_tiles, codes, params, scale)
    torch.cuda.synchronize()
    assert kv.kvarn_device_error() == 0
    return codes, params, scale


def _check(kv, cfg, x_tiles, label, rotate=True, normalize=True, kinds=("K", "V")):
    xs = x_tiles.float().cpu().double().numpy()
    out = {}
    for kind, name in ((kv.KVARN_KIND_K, "K"), (kv.KVARN_KIND_V, "V")):
        if name not in kinds:
            continue
        bits = cfg.k_bits if name == "K" else cfg.v_bits
        codes, params, scale = _encode_gpu(kv, cfg, kind, x_tiles)
        st = compare_encode(xs, name, bits, codes.cpu().numpy(), params.cpu().numpy(),
                            scale.cpu().numpy(), cfg.sinkhorn_iters, rotate, normalize)
        print(label, name, st)
        out[name] = (codes, params, scale, st)
    return out


def test_config0_tiny_codec(kv):
    # one kv head, K and V of 1024 tokens (8 tiles each), 2-bit, seed 0
    k, v = kv.synthetic.outlier_kv(0, 1, 1024)
    cfg = kv.kvarn_config_from_preset("kvarn_k2v2_g128")
    _check(kv, cfg, k.reshape(8, 128, 128).cuda(), "config0")
    _check(kv, cfg, v.reshape(8, 128, 128).cuda(), "config0")


ALL_PRESETS = ["kvarn_k4v2_g128", "kvarn_k2v2_g128", "kvarn_k4v4_g128", "kvarn_k2v4_g128"]


@pytest.mark.parametrize("preset", ALL_PRESETS)
def test_config1_batched_encode_full(kv, preset):
    # 64 sequences x 8 kv heads x one 128-token block, seed 1: 512 K tiles and 512 V tiles through
    # the fused K+V call, every tile against the oracle (including the 4-bit V encoder of the K4/V4
    # and K2/V4 presets); the single-kind calls must give the same bytes
    k, v = kv.synthetic.outlier_kv(1, 64 * 8, 128, device="cuda")
    k, v = k.reshape(-1, 128, 128), v.reshape(-1, 128, 128)
    n = k.shape[0]
    cfg = kv.kvarn_config_from_preset(preset)
    outs = []
    for bits in (cfg.k_bits, cfg.v_bits):
        outs += [torch.full((n, 128 * 16 * bits), 7, dtype=torch.uint8, device="cuda"),
                 torch.full((n, 512), 7, dtype=torch.uint8, device="cuda"),
                 torch.full((n,), 7.0, dtype=torch.float32, device="cuda")]
    kv.kvarn_encode_kv_blocks(cfg, k, v, *outs)
    torch.cuda.synchronize()
    assert kv.kvarn_device_error() == 0
    sep = list(_encode_gpu(kv, cfg, kv.KVARN_KIND_K, k)) + list(_encode_gpu(kv, cfg, kv.KVARN_KIND_V, v))
    for got, want in zip(outs, sep):
        assert torch.equal(got, want)
    for name, x, (c, p_, sc), bits in (("K", k, outs[:3], cfg.k_bits), ("V", v, outs[3:], cfg.v_bits)):
        st = compare_encode(x.float().cpu().double().numpy(), name, bits, c.cpu().numpy(), p_.cpu().numpy(),
                            sc.cpu().numpy())
        print(preset, name, st)
        assert st["free_code_mismatch"] <= 1e-4 * st["elements"]


def test_edge_tiles(kv):
    cfg = kv.kvarn_config_from_preset("kvarn_k4v2_g128")
    base = kv.synthetic.outlier_kv(5, 1, 128)[0].reshape(1, 128, 128)
    tiles = [torch.zeros(128, 128), torch.full((128, 128), 3.0), base[0].float() * 2.0 ** 40,
             base[0].float() * 2.0 ** -40, torch.randn(128, 128, generator=torch.Generator().manual_seed(3))]
    t = torch.zeros(128, 128)
    t[:, 7] = 5.0  # one non-zero channel
    tiles.append(t)
    t = torch.zeros(128, 128)
    t[9, :] = -2.0  # one non-zero token
    tiles.append(t)
    x = torch.stack(tiles).to(torch.bfloat16).cuda()
    res = _check(kv, cfg, x, "edge")
    codes, params, scale, _ = res["K"]
    assert scale[0].item() == 1.0 and not codes[0].any()


@pytest.mark.parametrize("flags,iters", [(0, 0), (0, 1), (0, 20), (1, 8), (2, 8), (3, 0)])
def test_ablation_flags_and_iterations(kv, flags, iters):
    k, _ = kv.synthetic.outlier_kv(6, 3, 128)
    cfg = kv.make_config(4, 2, iters, flags)
    _check(kv, cfg, k.reshape(3, 128, 128).cuda(), f"flags={flags} iters={iters}",
           rotate=not (flags & 1), normalize=not (flags & 2))


def test_persistent_grid_many_tiles_and_empty(kv):
    cfg = kv.kvarn_config_from_preset("kvarn_k2v2_g128")
    k, _ = kv.synthetic.outlier_kv(7, 1, 128 * 333, device="cuda")
    x = k.reshape(333, 128, 128)
    codes, params, scale = _encode_gpu(kv, cfg, kv.KVARN_KIND_K, x)
    # every tile independent of its position in the grid: re-encode a few tiles alone
    for i in (0, 151, 152, 332):
        c1, p1, s1 = _encode_gpu(kv, cfg, kv.KVARN_KIND_K, x[i:i + 1].contiguous())
        assert torch.equal(c1[0], codes[i]) and torch.equal(p1[0], params[i]) and s1[0] == scale[i]
    empty = torch.empty(0, dtype=torch.uint8, device="cuda")
    kv.kvarn_encode_blocks(cfg, kv.KVARN_KIND_K, torch.empty(0, 128, 128, dtype=torch.bfloat16, device="cuda"),
                           empty, empty, torch.empty(0, device="cuda"))


@pytest.mark.parametrize("preset", ALL_PRESETS)
@pytest.mark.parametrize("n", [512, 77, 1])
def test_fused_kv_encode_equals_separate_calls(kv, preset, n):
    # one launch over K and V tiles gives the two single-kind results bit for bit; the first
    # fused tiles are also checked against the oracle directly
    k, v = kv.synthetic.outlier_kv(11, n, 128, device="cuda")
    k, v = k.reshape(n, 128, 128), v.reshape(n, 128, 128)
    cfg = kv.kvarn_config_from_preset(preset)
    ref_k = _encode_gpu(kv, cfg, kv.KVARN_KIND_K, k)
    ref_v = _encode_gpu(kv, cfg, kv.KVARN_KIND_V, v)
    out_k = [torch.full_like(t, 7) for t in ref_k]
    out_v = [torch.full_like(t, 7) for t in ref_v]
    kv.kvarn_encode_kv_blocks(cfg, k, v, *out_k, *out_v)
    torch.cuda.synchronize()
    assert kv.kvarn_device_error() == 0
    for got, want in zip(out_k + out_v, list(ref_k) + list(ref_v)):
        assert torch.equal(got, want)
    m = min(n, 4)
    for name, x, res, bits in (("K", k, out_k, cfg.k_bits), ("V", v, out_v, cfg.v_bits)):
        compare_encode(x[:m].float().cpu().double().numpy(), name, bits, res[0][:m].cpu().numpy(),
                       res[1][:m].cpu().numpy(), res[2][:m].cpu().numpy())


@pytest.mark.parametrize("preset", ALL_PRESETS)
def test_dequant_matches_oracle_on_identical_packed_input(kv, preset):
    cfg = kv.kvarn_config_from_preset(preset)
    k, v = kv.synthetic.outlier_kv(8, 40, 128, device="cuda")
    for kind, name, x in ((kv.KVARN_KIND_K, "K", k), (kv.KVARN_KIND_V, "V", v)):
        bits = cfg.k_bits if name == "K" else cfg.v_bits
        x = x.reshape(-1, 128, 128)
        codes, params, scale = _encode_gpu(kv, cfg, kind, x)
        for basis in (0, 1):
            out = torch.empty(x.shape[0], 128, 128, device="cuda")
            kv.kvarn_dequant(cfg, kind, codes, params, scale, out, original_basis=basis)
            torch.cuda.synchronize()
            ref = o.dequant_blocks(codes.cpu().numpy(), params.cpu().numpy(), scale.cpu().numpy(),
                                   name, bits, original_basis=bool(basis))
            got = out.cpu().double().numpy()
            for t in range(x.shape[0]):
                rms = np.sqrt(np.mean(ref[t] ** 2))
                assert np.abs(got[t] - ref[t]).max() <= 1e-3 * rms
        # reconstruction quality sanity: the codec estimate is close to the input
        assert rel_l2(got, x.float().cpu().double().numpy()) < (0.5 if bits == 2 else 0.15)


@pytest.mark.parametrize("flags", [0, 1])
@pytest.mark.parametrize("preset", ["kvarn_k4v2_g128", "kvarn_k2v4_g128"])
def test_mean_dominated_tiles(kv, preset, flags):
    # K with a per-channel bias of 30x, 100x and 300x its within-channel std, V with per-token
    # offsets of the same sizes: rows or columns whose variance is a small fraction of their mean
    # square, where a one-pass fp32 variance would lose most of its digits; with and without the
    # rotation (without it the biases reach the normalisation unrotated)
    from tests import _tiles

    base = kv.kvarn_config_from_preset(preset)
    cfg = kv.make_config(base.k_bits, base.v_bits, 8, flags)
    xk = _tiles.biased_k_tiles(61).cuda()
    xv = _tiles.offset_v_tiles(62).cuda()
    _check(kv, cfg, xk, f"biased K flags={flags}", rotate=not flags, kinds=("K",))
    _check(kv, cfg, xv, f"offset V flags={flags}", rotate=not flags, kinds=("V",))


@pytest.mark.parametrize("bits", [2, 4])
def test_degeneracy_threshold_rows_and_columns(kv, bits):
    # rows (and, in a second tile, columns) whose variance is 0.56x, 0.985x, 1.012x and 2.07x of
    # 1e-5 times their mean square when the normalisation first meets them: the ones below keep
    # their factor, the ones above are normalised, and the kernel must decide each as the oracle
    # does (no rotation, so the constructed rows reach the normalisation unchanged)
    from tests import _tiles

    cfg = kv.make_config(bits, bits, 8, 1)
    xr, rows = _tiles.threshold_row_tile(1)
    xc, cols = _tiles.threshold_column_tile(2)
    for x, where, axis in ((xr, rows, "token"), (xc, cols, "channel")):
        # precondition: the constructed rows / columns sit at their ratios, and no decision the
        # oracle takes on the tile is within 0.5% of the threshold
        trace = []
        o.dual_axis_normalize(x.float().double().numpy(), 8, trace=trace)
        first = trace[0 if axis == "token" else 1][2]
        for label, i in where.items():
            want = float(label[:-1])
            assert abs(first[i] / 1e-5 / want - 1) < 0.03, (axis, label, first[i])
        assert min(np.nanmin(np.abs(r[2] / 1e-5 - 1)) for r in trace) > 5e-3
        _check(kv, cfg, x[None].cuda(), f"threshold {axis}s", rotate=False)
