"""Block pseudo-decode through libkvarn (encode of each finished block + attention over the packed
cache) against the fp64 oracle: free-running at a reduced size, teacher-forced at full size."""
import math

import numpy as np
import pytest
import torch

from oracle import pseudo_decode as opd
from oracle import kvarn_oracle as o
from tests._parity import rel_l2

pytestmark = pytest.mark.gpu


def _np_weights(w):
    return [{k: t.float().cpu().double().numpy() for k, t in wl.items()} for wl in w]


def test_reduced_stack_free_running_matches_oracle(kv):
    from bit_kv_cache_kvarn_gb300 import pseudo_decode as pd

    hq, hkv, hidden, layers, blocks = 4, 2, 256, 2, 4
    w = pd.make_weights(40, layers, hidden, hq, hkv)
    x = pd.make_input(40, blocks * 128, hidden)
    cfg = kv.kvarn_config_from_preset("kvarn_k2v2_g128")
    gq, _ = pd.run(kv, cfg, w, x, hq, hkv, quantised=True)
    gr, _ = pd.run(kv, None, w, x, hq, hkv, quantised=False)
    assert kv.kvarn_device_error() == 0
    wn, xn = _np_weights(w), x.float().cpu().double().numpy()
    oq = opd.run(wn, xn, hq, hkv, quantised=True, k_bits=2, v_bits=2)
    orf = opd.run(wn, xn, hq, hkv, quantised=False)
    worst_ref = worst_q = 0.0
    for j in range(blocks):
        for l in range(layers):
            worst_ref = max(worst_ref, rel_l2(gr[j][l].cpu().double().numpy(), orf[j][l]))
            worst_q = max(worst_q, rel_l2(gq[j][l].cpu().double().numpy(), oq[j][l]))
    mg = np.array(pd.mae_curves(gq, gr))
    mo = opd.mae_curves(oq, orf)
    print("rel-L2 reference run", worst_ref, "quantised run", worst_q)
    print("MAE per block x layer, GPU\n", mg, "\noracle\n", mo)
    # the model plumbing (fp32 on the GPU, fp64 in the oracle) agrees closely without quantisation
    assert worst_ref <= 1e-4
    # Free-running, the two quantised trajectories are not bit-identical: a K/V value whose fp32
    # and fp64 projections round to different bf16 neighbours can move its group's min/max and
    # with it that group's codes.  Their outputs stay close and the error curves -- the quantity
    # the evaluation reports -- agree to 1%; strict parity is the teacher-forced test below.
    assert worst_q <= 2e-2
    assert np.all(mo[0] == 0.0) and np.all(mg[0] <= 1e-6)  # block 0 reads no cache
    assert np.all(np.abs(mg[1:] - mo[1:]) <= 0.01 * mo[1:])


def test_config4_teacher_forced_against_oracle(kv):
    # 4 layers, 32q/8kv, hidden 4096, 64 blocks of 128 tokens, seed 4; the oracle recomputes
    # sampled queries' attention from the GPU's own packed cache, queries and block K/V
    from bit_kv_cache_kvarn_gb300 import pseudo_decode as pd

    hq, hkv, hidden, layers, blocks = 32, 8, 4096, 4, 64
    w = pd.make_weights(4, layers, hidden, hq, hkv)
    x = pd.make_input(4, blocks * 128, hidden)
    cfg = kv.kvarn_config_from_preset("kvarn_k2v2_g128")
    cap = {(1, 0): None, (32, 2): None, (63, 3): None}
    attn, secs = pd.run(kv, cfg, w, x, hq, hkv, quantised=True, capture=cap)
    assert kv.kvarn_device_error() == 0
    print(f"config 4 pseudo-decode: {secs:.3f} s on the GPU")
    scale = 1 / math.sqrt(128)
    for (j, l), c in cap.items():
        toks = [0, 77, 127]
        kc, kp, ks, vc, vp, vs = (t.cpu().numpy() for t in c["pools"])
        table = np.array([[[jj * hkv + h for jj in range(max(j, 1))] for h in range(hkv)]] * len(toks))
        kt = c["k_blk"].permute(1, 0, 2).float().cpu().double().numpy()
        vt = c["v_blk"].permute(1, 0, 2).float().cpu().double().numpy()
        ref = o.decode_attention(c["q"][toks].float().cpu().double().numpy(), hq, hkv, kc, kp, ks, vc, vp, vs,
                                 table, [128 * j + t + 1 for t in toks], np.stack([kt] * len(toks)),
                                 np.stack([vt] * len(toks)), scale, 2, 2, full_tail=True)
        got = c["attn"][toks].cpu().double().numpy()
        worst = max(rel_l2(got[i, h], ref[i, h]) for i in range(len(toks)) for h in range(hq))
        print(f"block {j} layer {l}: worst rel-L2 {worst:.2e}")
        assert worst <= 1e-3
        assert torch.equal(c["attn"], attn[j][l])


_ORACLE_CODEC = {"kvarn_k2v2_g128": dict(iters=8, rotate=True, normalize=True),
                 "hadamard_k2v2_g128": dict(iters=0, rotate=True, normalize=False),
                 "kivi_k2v2_g128": dict(iters=0, rotate=False, normalize=False)}


@pytest.mark.parametrize("preset", list(_ORACLE_CODEC))
def test_reduced_stack_with_kv_outliers_free_running_matches_oracle(kv, preset):
    # the variant whose K/V carry the cache recipe's outlier channels and tokens, through KVarN,
    # rotation only and plain RTN: GPU and oracle curves agree as for the plain stack
    from bit_kv_cache_kvarn_gb300 import pseudo_decode as pd
    from bit_kv_cache_kvarn_gb300 import synthetic

    hq, hkv, hidden, layers, blocks = 4, 2, 256, 2, 4
    w = pd.make_weights(41, layers, hidden, hq, hkv, kv_outliers=True)
    x = pd.make_input(41, blocks * 128, hidden)
    ts = synthetic.pseudo_decode_token_scales(41, blocks * 128)
    cfg = kv.kvarn_config_from_preset(preset)
    gq, _ = pd.run(kv, cfg, w, x, hq, hkv, quantised=True, kv_token_scale=ts)
    gr, _ = pd.run(kv, None, w, x, hq, hkv, quantised=False, kv_token_scale=ts)
    assert kv.kvarn_device_error() == 0
    wn, xn = _np_weights(w), x.float().cpu().double().numpy()
    tsn = ts.double().numpy()
    oq = opd.run(wn, xn, hq, hkv, quantised=True, k_bits=2, v_bits=2, kv_token_scale=tsn, **_ORACLE_CODEC[preset])
    orf = opd.run(wn, xn, hq, hkv, quantised=False, kv_token_scale=tsn)
    worst_ref = max(rel_l2(gr[j][l].cpu().double().numpy(), orf[j][l]) for j in range(blocks) for l in range(layers))
    worst_q = max(rel_l2(gq[j][l].cpu().double().numpy(), oq[j][l]) for j in range(blocks) for l in range(layers))
    mg, mo = np.array(pd.mae_curves(gq, gr)), opd.mae_curves(oq, orf)
    print(preset, "rel-L2 reference run", worst_ref, "quantised run", worst_q)
    print("MAE GPU\n", mg, "\noracle\n", mo)
    # The unquantised runs differ only by the fp32 (GPU) and fp64 (oracle) model plumbing, whose
    # q/k/v can round to neighbouring bf16 values; with outlier channels x20 and tokens x8 the
    # logits span ~10^3 and one such neighbour moves a sharp softmax by ~1e-4, so the bound here is
    # the decode tolerance.  The quantised trajectories part at those neighbours (a different code
    # then feeds every later block), so they are compared through their error curves -- the
    # quantity the evaluation reports -- and strictly only teacher-forced (the config-4 test).
    assert worst_ref <= 1e-3
    assert np.all(np.abs(mg[1:] - mo[1:]) <= 0.01 * mo[1:])


def test_config4_full_size_free_running_curves_against_stored_oracle(kv):
    # the full config-4 stack, free-running on the GPU, against the fp64 oracle's own free-running
    # MAE curves (tests/golden/config4_oracle_mae.json, written by make_config4_oracle_curves.py,
    # which runs only the oracle): plain stack with KVarN, and the outlier variant with KVarN,
    # rotation only and plain RTN
    import json
    import os

    from bit_kv_cache_kvarn_gb300 import pseudo_decode as pd
    from bit_kv_cache_kvarn_gb300 import synthetic

    with open(os.path.join(os.path.dirname(__file__), "golden", "config4_oracle_mae.json")) as f:
        gold = json.load(f)
    c = gold["config"]
    names = {"kvarn_k2v2": "kvarn_k2v2_g128", "hadamard_k2v2": "hadamard_k2v2_g128", "rtn_k2v2": "kivi_k2v2_g128"}
    for variant in ("plain", "kv_outliers"):
        out = variant == "kv_outliers"
        w = pd.make_weights(c["seed"], c["layers"], c["hidden"], c["hq"], c["hkv"], kv_outliers=out)
        x = pd.make_input(c["seed"], c["blocks"] * 128, c["hidden"])
        ts = synthetic.pseudo_decode_token_scales(c["seed"], c["blocks"] * 128) if out else None
        ref, _ = pd.run(kv, None, w, x, c["hq"], c["hkv"], quantised=False, kv_token_scale=ts)
        per_block = {}
        for name, preset in names.items():
            if name not in gold[variant]:
                continue
            a, _ = pd.run(kv, kv.kvarn_config_from_preset(preset), w, x, c["hq"], c["hkv"], quantised=True,
                          kv_token_scale=ts)
            mg = np.array(pd.mae_curves(a, ref))
            mo = np.array(gold[variant][name]["mae"])
            rel = np.abs(mg[1:] - mo[1:]) / mo[1:]
            lg, lo = mg[1:].mean(axis=1), mo[1:].mean(axis=1)  # per block, over the layers
            rel_block = np.abs(lg - lo) / lo
            print(variant, name, "curve difference per point: worst", float(rel.max()), "mean", float(rel.mean()),
                  "| per block (layer mean): worst", float(rel_block.max()))
            assert rel.mean() <= CURVE_MEAN_TOL, (variant, name)
            assert rel_block.max() <= CURVE_BLOCK_TOL, (variant, name)
            per_block[name] = (lg, lo)
        # the comparison the evaluation makes: each codec's error relative to KVarN's, block by block
        for name in per_block:
            if name == "kvarn_k2v2":
                continue
            rg = per_block[name][0] / per_block["kvarn_k2v2"][0]
            ro = per_block[name][1] / per_block["kvarn_k2v2"][1]
            print(variant, name, "/ kvarn_k2v2 ratio, GPU", rg.min(), rg.max(), "oracle", ro.min(), ro.max())
            assert np.all(np.abs(rg - ro) <= CURVE_BLOCK_TOL * ro), (variant, name)
    assert kv.kvarn_device_error() == 0


# Full-size free-running curves: the GPU (fp32 projections) and oracle (fp64) trajectories part at
# single bf16 rounding flips of K/V and then carry different quantisation realisations block after
# block, so single (block, layer) points of the deepest layer can differ by ~10%.  What the
# evaluation reports -- each block's error (here averaged over the layers) and the codecs' errors
# relative to one another -- must agree within 5%, well inside the 10% (rotation only) and 2x (RTN)
# gaps between codecs that the outlier variant shows; the per-point differences must average 2%.
CURVE_BLOCK_TOL = 0.05
CURVE_MEAN_TOL = 0.02
