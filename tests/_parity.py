"""Parity helpers: compare the CUDA codec with the fp64 oracle stage by stage.

Rounding decisions (an E4M3 scale, an FP16 zero-point, an integer code) are compared exactly,
except where the oracle's unrounded value lies within TIE_REL (relative) of a rounding boundary:
the kernel computes the same quantity in fp32, so such a decision may legitimately go the other
way.  Each stage is teacher-forced with the GPU's earlier decisions, so a flip upstream never
hides or excuses a mismatch downstream.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import kvarn_oracle as o

TIE_REL = 1e-5
CODE_MISMATCH_BUDGET = 1e-4  # total code mismatches allowed, as a fraction of elements

_E4M3_GRID = np.sort(torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn)
                     .to(torch.float64).numpy())
_FP16_GRID = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)


def _near(x, points, rel):
    x = np.abs(np.asarray(x, dtype=np.float64))
    idx = np.clip(np.searchsorted(points, x), 1, len(points) - 1)
    d = np.minimum(np.abs(x - points[idx - 1]), np.abs(points[idx] - x))
    return d <= rel * np.maximum(x, 1e-30)


def near_rn_tie(x, grid):
    mids = (grid[1:] + grid[:-1]) / 2
    return _near(x, mids, TIE_REL)


def near_grid_point(x, grid):
    return _near(x, grid, TIE_REL)


def code_tie(u):
    frac = np.abs(u - np.floor(u) - 0.5)
    return frac <= TIE_REL * np.maximum(1.0, np.abs(u))


def compare_encode(x_tiles, kind, bits, gpu_codes, gpu_params, gpu_scale, iters=8, rotate=True,
                   normalize=True):
    """x_tiles: [n,128,128] fp64 (the bf16 inputs); gpu_*: numpy arrays from the kernel.
    Returns a dict of counts; raises AssertionError on any unexcused difference."""
    n = x_tiles.shape[0]
    stats = dict(tiles=n, elements=n * 128 * 128, s2_flips=0, s1_flips=0, z_flips=0, g_diff=0,
                 code_ties=0, free_code_mismatch=0)
    for k in range(n):
        gs1, gs2, gz = o.unpack_params(gpu_params[k])
        gcodes = o.unpack_tile(gpu_codes[k], bits, kind)
        gg = float(gpu_scale[k])
        free = o.encode_tile(x_tiles[k], kind, bits, iters, rotate, normalize)
        stats["free_code_mismatch"] += int((free["codes"] != gcodes).sum())
        # stage 1: s2
        bad = gs2 != free["s2"]
        if bad.any():
            tie = near_rn_tie(free["s2_raw"], _E4M3_GRID)
            assert np.all(tie[bad]), f"tile {k}: s2 differs away from a rounding tie"
            stats["s2_flips"] += int(bad.sum())
        # stage 2: given the GPU's s2 -> g, S1, Z
        st2 = o.encode_tile(x_tiles[k], kind, bits, iters, rotate, normalize, forced={"s2": gs2})
        if gg != st2["g"]:
            stats["g_diff"] += 1
            raise AssertionError(f"tile {k}: tile factor {gg} != oracle {st2['g']}")
        bad = gs1 != st2["S1"]
        if bad.any():
            tie = near_grid_point(st2["S1_raw"], _E4M3_GRID)
            assert np.all(tie[bad]), f"tile {k}: S1 differs away from a rounding boundary"
            stats["s1_flips"] += int(bad.sum())
        bad = gz != st2["Z"]
        if bad.any():
            tie = near_rn_tie(st2["Z_raw"], _FP16_GRID)
            assert np.all(tie[bad]), f"tile {k}: Z differs away from a rounding tie"
            stats["z_flips"] += int(bad.sum())
        # stage 3: given all GPU parameters -> codes
        st3 = o.encode_tile(x_tiles[k], kind, bits, iters, rotate, normalize,
                            forced={"s2": gs2, "S1": gs1, "Z": gz, "g": gg})
        bad = gcodes != st3["codes"]
        if bad.any():
            tie = code_tie(st3["u"])
            assert np.all(tie[bad]), (
                f"tile {k}: {int((bad & ~tie).sum())} codes differ away from a rounding tie")
            stats["code_ties"] += int(bad.sum())
    frac = stats["free_code_mismatch"] / stats["elements"]
    assert frac <= CODE_MISMATCH_BUDGET, f"free-running code mismatch fraction {frac:.2e}"
    return stats


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)
