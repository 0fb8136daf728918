"""Writes tests/golden/config4_oracle_mae.json: the fp64 oracle's free-running block pseudo-decode
MAE curves at the full config-4 size (4 layers, 32q/8kv heads, hidden 4096, 64 blocks of 128
tokens, seed 4), for the plain random-weight stack and for its outlier variant (K/V with the cache
recipe's outlier channels and tokens).

Only the oracle (oracle/) and the seeded input generators run here; nothing comes from the CUDA
path.  It takes several minutes of CPU:

    python tests/golden/make_config4_oracle_curves.py

With --time-only it runs the plain stack alone (reference and KVarN cache), prints the oracle's
wall times and the host's CPU count as one JSON line and writes nothing.
"""
from __future__ import annotations

import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from bit_kv_cache_kvarn_gb300 import synthetic  # noqa: E402
from oracle import pseudo_decode as opd  # noqa: E402

SEED, LAYERS, HIDDEN, HQ, HKV, BLOCKS = 4, 4, 4096, 32, 8, 64
# (name, k_bits, v_bits, iters, rotate, normalize): the presets of the GPU harness
CODECS = (("kvarn_k2v2", 2, 2, 8, True, True),
          ("hadamard_k2v2", 2, 2, 0, True, False),
          ("rtn_k2v2", 2, 2, 0, False, False))


def curves(kv_outliers: bool, codecs):
    w = synthetic.pseudo_decode_weights(SEED, LAYERS, HIDDEN, HQ, HKV, kv_outliers=kv_outliers)
    x = synthetic.pseudo_decode_input(SEED, BLOCKS * 128, HIDDEN)
    wn = [{k: t.float().double().numpy() for k, t in wl.items()} for wl in w]
    xn = x.float().double().numpy()
    ts = synthetic.pseudo_decode_token_scales(SEED, BLOCKS * 128).double().numpy() if kv_outliers else None
    t0 = time.time()
    ref = opd.run(wn, xn, HQ, HKV, quantised=False, kv_token_scale=ts)
    out = {"reference_seconds": round(time.time() - t0, 1)}
    for name, kb, vb, iters, rot, norm in codecs:
        t0 = time.time()
        a = opd.run(wn, xn, HQ, HKV, quantised=True, k_bits=kb, v_bits=vb, iters=iters, rotate=rot,
                    normalize=norm, kv_token_scale=ts)
        out[name] = {"seconds": round(time.time() - t0, 1), "mae": opd.mae_curves(a, ref).tolist(),
                     "mean_abs_reference": [[float(np.mean(np.abs(r))) for r in rr] for rr in ref]}
        print(name, "outliers" if kv_outliers else "plain", out[name]["seconds"], "s", flush=True)
    return out


def main():
    if "--time-only" in sys.argv[1:]:
        t0 = time.time()
        r = curves(False, CODECS[:1])
        print(json.dumps({"config4_plain_stack": {"reference_seconds": r["reference_seconds"],
                                                   "kvarn_k2v2_seconds": r["kvarn_k2v2"]["seconds"],
                                                   "total_seconds": round(time.time() - t0, 1),
                                                   "host_cpus": len(os.sched_getaffinity(0))}}))
        return
    res = {"config": dict(seed=SEED, layers=LAYERS, hidden=HIDDEN, hq=HQ, hkv=HKV, blocks=BLOCKS),
           "plain": curves(False, CODECS[:1]), "kv_outliers": curves(True, CODECS)}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "config4_oracle_mae.json")
    with open(path, "w") as f:
        json.dump(res, f)
    print("wrote", path)


if __name__ == "__main__":
    main()
