"""kvarn_decode_attention_static_ws: decode attention whose split-K scratch is a fixed device array
inside libkvarn, for callers that cannot allocate device memory where they run decode (inside a
host callback, in a plugin whose framework owns the allocator, or in a loop that must not pay
cudaMalloc's implicit synchronisation).  It must give the same output as kvarn_decode_attention
with a caller workspace, call after call, and refuse shapes whose scratch would not fit.

This file is collected last on purpose, so a run that stops at the first failure has already run
every other test; it also passes when run alone in a fresh process."""
import math

import pytest
import torch

from tests._parity import rel_l2
from tests.test_gpu_decode import DECODE_REL_L2, build_cache, run_gpu

pytestmark = pytest.mark.gpu


def _static(kv, cfg, q, hkv, c, scale):
    out = torch.full((q.shape[0], q.shape[1], 128), float("nan"), device="cuda")
    kc, kp, ks = c["pools"]["k"]
    vc, vp, vs = c["pools"]["v"]
    kv.kvarn_decode_attention_static_ws(cfg, q, hkv, kc, kp, ks, vc, vp, vs, c["table"],
                                        c["seq_lens"], c["k_tail"], c["v_tail"], scale, out,
                                        seq_lens_host=c["lens"])
    torch.cuda.synchronize()
    return out


def _same(a, b):
    a, b = a.cpu().double().numpy(), b.cpu().double().numpy()
    for bi in range(a.shape[0]):
        for h in range(a.shape[1]):
            if not b[bi, h].any():
                assert not a[bi, h].any()
                continue
            assert rel_l2(a[bi, h], b[bi, h]) <= DECODE_REL_L2, (bi, h)


def test_static_scratch_matches_caller_workspace_on_consecutive_calls(kv):
    scale = 1 / math.sqrt(128)
    # call 1: ragged lengths including an empty sequence and tail-only ones, K4/V2, GQA 4
    cfg1 = kv.kvarn_config_from_preset("kvarn_k4v2_g128")
    lens1 = [0, 100, 128, 17 * 128 + 9, 40 * 128 + 127]
    c1 = build_cache(kv, cfg1, len(lens1), 2, lens1, seed=21)
    q1 = kv.synthetic.queries(21, len(lens1), 8, device="cuda")
    # call 2 right after: a different shape, preset and cache, so stale partials from call 1
    # sit in the shared array
    cfg2 = kv.kvarn_config_from_preset("kvarn_k2v2_g128")
    lens2 = [64 * 128, 3 * 128 + 1, 50]
    c2 = build_cache(kv, cfg2, len(lens2), 4, lens2, seed=22)
    q2 = kv.synthetic.queries(22, len(lens2), 16, device="cuda")

    got1 = _static(kv, cfg1, q1, 2, c1, scale)
    got2 = _static(kv, cfg2, q2, 4, c2, scale)
    _same(got1, run_gpu(kv, cfg1, q1, 2, c1, scale))
    _same(got2, run_gpu(kv, cfg2, q2, 4, c2, scale))
    # and once more in the original order
    _same(_static(kv, cfg1, q1, 2, c1, scale), got1)


def test_static_scratch_rejects_shapes_beyond_its_size(kv):
    cfg = kv.kvarn_config_from_preset("kvarn_k2v2_g128")
    # 64 sequences x 32 query heads x 256 tiles of context needs 17.3 MB of partials > 8 MiB
    need = kv.kvarn_decode_workspace_size(cfg, 64, 32, 8, 256)
    assert need > 8 * 1024 * 1024
    dummy_u8 = torch.zeros(16, dtype=torch.uint8, device="cuda")
    table = torch.zeros(64, 8, 256, dtype=torch.int32, device="cuda")
    q = torch.zeros(64, 32, 128, dtype=torch.bfloat16, device="cuda")
    tail = torch.zeros(64, 8, 128, 128, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(64, dtype=torch.int32, device="cuda")
    out = torch.full((64, 32, 128), 7.0, device="cuda")
    with pytest.raises(kv.KvarnError) as ei:
        kv.kvarn_decode_attention_static_ws(cfg, q, 8, dummy_u8, dummy_u8, dummy_u8.float(), dummy_u8,
                                            dummy_u8, dummy_u8.float(), table, lens, tail, tail, 0.1, out)
    assert ei.value.status == 4 and "static scratch" in str(ei.value)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)  # nothing was launched
