"""GPU error diagnostics (libkvarn encode + dequant, statistics in PyTorch) against the same
statistics of the oracle's own encode and dequantisation."""
import numpy as np
import pytest
import torch

from oracle import kvarn_oracle as o

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("preset", ["kivi_k2v2_g128", "hadamard_k2v2_g128", "kvarn_k2v2_g128", "kvarn_k4v2_g128"])
def test_diagnostics_match_oracle(kv, preset):
    from bit_kv_cache_kvarn_gb300 import diagnostics

    cfg = kv.kvarn_config_from_preset(preset)
    k, v = kv.synthetic.outlier_kv(30, 12, 128, device="cuda")
    k, v = k.reshape(12, 128, 128), v.reshape(12, 128, 128)
    got = diagnostics.run(kv, k, v, presets=(preset,))[preset]
    rotate, normalize = not (cfg.flags & 1), not (cfg.flags & 2)
    for kind, x, bits in (("K", k, cfg.k_bits), ("V", v, cfg.v_bits)):
        xs = x.float().cpu().double().numpy()
        c, p, s, _ = o.encode_blocks(xs, kind, bits, cfg.sinkhorn_iters, rotate, normalize)
        xh = o.dequant_blocks(c, p, s, kind, bits, original_basis=True, rotate=rotate)
        e_m, e_d = o.error_decomposition(xs.reshape(-1, 128), xh.reshape(-1, 128))
        mse = (e_m + e_d).sum() / xs.size
        g = got[kind]
        print(preset, kind, g["mse_per_element"], g["magnitude_share_of_top_errors"])
        assert abs(g["mse_per_element"] - mse) <= 1e-3 * mse
        assert abs(g["magnitude_share_of_all_error"] - e_m.sum() / (e_m + e_d).sum()) <= 2e-3
        share = o.magnitude_share_of_top_errors(e_m, e_d, diagnostics.FRACTIONS)
        for f in diagnostics.FRACTIONS[:3]:
            assert abs(g["magnitude_share_of_top_errors"][str(f)] - share[f]) <= 5e-3
        lr = np.abs(np.log2(o.token_scale_ratio(xs.reshape(-1, 128), xh.reshape(-1, 128))))
        assert abs(g["token_scale_abs_log2_ratio"]["mean"] - lr.mean()) <= 1e-3 * max(lr.mean(), 1e-6) + 1e-6
