"""Hand-built input tiles for the encoder's hard cases (input generators only: no codec arithmetic).

* Mean-dominated tiles: K with a large per-channel bias (after the rotation every column is shifted
  by the rotated bias vector) and V with a per-token offset (after the rotation it lands in channel
  0, whose column becomes nearly constant).  Real key caches carry such channel biases.
* Degeneracy-threshold tiles (for the no-rotation flag, where the input reaches the normalisation
  unchanged): rows, or columns, whose values take two neighbouring bf16 levels c and c + 1 with k
  of 128 entries at c + 1, so that their variance over mean square, f (1 - f) / (c + f)^2 with
  f = k / 128, sits just below, just above, half and twice the 1e-5 threshold under which the
  normalisation leaves a row's or column's factor unchanged.
All values are exactly representable in bf16.
"""
from __future__ import annotations

import numpy as np
import torch

# (c, k): variance / mean square = f (1 - f) / ((c + f)^2 + f (1 - f)), f = k / 128
THRESHOLD_LEVELS = {"0.56x": (128, 13), "0.985x": (128, 26), "1.012x": (128, 27), "2.07x": (64, 12)}


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)


def biased_k_tiles(seed: int, ratios=(30, 100, 300), per_ratio=2) -> torch.Tensor:
    """K tiles with a per-channel bias `ratio` times the channel's within-tile std."""
    g = np.random.default_rng(seed)
    out = []
    for ratio in ratios:
        for _ in range(per_ratio):
            chan = np.exp(g.standard_normal(128))
            tok = np.exp(0.5 * g.standard_normal(128))
            x = g.standard_normal((128, 128)) * chan[None, :] * tok[:, None]
            bias = ratio * chan * np.where(g.random(128) < 0.5, -1.0, 1.0)
            out.append(x + bias[None, :])
    return _bf16(np.stack(out))


def offset_v_tiles(seed: int, ratios=(30, 100, 300), per_ratio=2) -> torch.Tensor:
    """V tiles with a positive per-token offset `ratio` times the typical channel std."""
    g = np.random.default_rng(seed)
    out = []
    for ratio in ratios:
        for _ in range(per_ratio):
            chan = np.exp(g.standard_normal(128))
            x = g.standard_normal((128, 128)) * chan[None, :]
            off = ratio * np.median(chan) * np.exp(0.3 * g.standard_normal(128))
            out.append(x + off[:, None])
    return _bf16(np.stack(out))


def _two_level(c: int, k: int, g) -> np.ndarray:
    v = np.full(128, float(c))
    v[g.permutation(128)[:k]] = c + 1.0
    return v


def threshold_row_tile(seed: int) -> tuple[torch.Tensor, dict]:
    """Gaussian tile whose rows 3, 40, 77, 114 are two-level rows at the THRESHOLD_LEVELS ratios.
    Returns the tile and {label: row}."""
    g = np.random.default_rng(seed)
    x = g.standard_normal((128, 128))
    rows = {}
    for (label, (c, k)), t in zip(THRESHOLD_LEVELS.items(), (3, 40, 77, 114)):
        x[t] = _two_level(c, k, g)
        rows[label] = t
    return _bf16(x), rows


def threshold_column_tile(seed: int) -> tuple[torch.Tensor, dict]:
    """Rows of a +-1024 Sylvester Hadamard pattern (every row has the same spread, so the token step
    gives every row the same factor) with columns 5, 33, 70, 101 replaced by two-level columns at
    the THRESHOLD_LEVELS ratios.  Returns the tile and {label: column}."""
    g = np.random.default_rng(seed)
    i = np.arange(128)
    h = np.where(np.vectorize(lambda v: bin(v).count("1") % 2)(i[:, None] & i[None, :]) == 0, 1.0, -1.0)
    h[0] = -h[1]  # the all-ones row would be constant
    x = 1024.0 * h
    cols = {}
    for (label, (c, k)), j in zip(THRESHOLD_LEVELS.items(), (5, 33, 70, 101)):
        x[:, j] = _two_level(c, k, g)
        cols[label] = j
    return _bf16(x), cols
