"""Pins of the pseudo-decode reference (oracle/pseudo_decode.py) against definitions that do not
share its code: PyTorch's bf16 cast and SDPA, RoPE's relative-position property, and ordinary
(unblocked) causal attention."""
import numpy as np
import torch

from oracle import kvarn_oracle as o
from oracle import pseudo_decode as pd


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(40)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(pd.bf16_round(x.astype(np.float64)), ref)


def test_rmsnorm_unit_rms():
    x = np.random.default_rng(41).standard_normal((5, 300)) * 7
    y = pd.rmsnorm(x, eps=0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-14)


def test_rope_is_a_rotation_with_relative_scores():
    rng = np.random.default_rng(42)
    q, k = rng.standard_normal((1, 1, 128)), rng.standard_normal((1, 1, 128))
    # norms preserved; q_m . k_n depends only on m - n
    assert np.isclose(np.linalg.norm(pd.rope(q, np.array([37]))), np.linalg.norm(q), rtol=1e-14)
    s1 = float(pd.rope(q, np.array([1000]))[0, 0] @ pd.rope(k, np.array([990]))[0, 0])
    s2 = float(pd.rope(q, np.array([10]))[0, 0] @ pd.rope(k, np.array([0]))[0, 0])
    assert abs(s1 - s2) <= 1e-9 * max(1.0, abs(s2))
    # position 0 is the identity
    assert np.array_equal(pd.rope(q, np.array([0])), q)


def test_causal_block_attention_matches_sdpa():
    rng = np.random.default_rng(43)
    t, p, hq, hkv = 16, 40, 4, 2
    q = rng.standard_normal((t, hq, 128))
    kp, vp = rng.standard_normal((p, hkv, 128)), rng.standard_normal((p, hkv, 128))
    kb, vb = rng.standard_normal((t, hkv, 128)), rng.standard_normal((t, hkv, 128))
    out = pd.causal_block_attention(q, kp, vp, kb, vb, 0.09)
    for h in range(hq):
        kv = h // 2
        keys = torch.from_numpy(np.concatenate([kp[:, kv], kb[:, kv]]))
        vals = torch.from_numpy(np.concatenate([vp[:, kv], vb[:, kv]]))
        mask = torch.ones(t, p + t, dtype=torch.bool)
        mask[:, p:] = torch.tril(torch.ones(t, t, dtype=torch.bool))
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[:, h])[None], keys[None], vals[None], attn_mask=mask[None], scale=0.09)[0]
        assert np.abs(out[:, h] - ref.numpy()).max() <= 1e-12


def _tiny_model(seed, layers=2, hidden=256, hq=4, hkv=2):
    rng = np.random.default_rng(seed)
    w = [dict(wq=rng.standard_normal((hq * 128, hidden)) * 0.02, wk=rng.standard_normal((hkv * 128, hidden)) * 0.02,
              wv=rng.standard_normal((hkv * 128, hidden)) * 0.02, wo=rng.standard_normal((hidden, hq * 128)) * 0.02)
         for _ in range(layers)]
    return w, rng.standard_normal((3 * 128, hidden))


def test_unquantised_pseudo_decode_is_plain_causal_attention():
    # without quantisation the block-by-block cache bookkeeping must vanish: each layer equals
    # ordinary causal attention over the whole sequence (block = 128 or 64 gives the same)
    w, x = _tiny_model(44)
    hq, hkv = 4, 2
    a128 = pd.run(w, x, hq, hkv, quantised=False)
    a64 = pd.run(w, x, hq, hkv, quantised=False, block=64)
    T = x.shape[0]
    h = x.copy()
    pos = np.arange(T)
    for l, wl in enumerate(w):
        n = pd.rmsnorm(h)
        q = pd.bf16_round(pd.rope((n @ wl["wq"].T).reshape(T, hq, 128), pos))
        k = pd.bf16_round(pd.rope((n @ wl["wk"].T).reshape(T, hkv, 128), pos))
        v = pd.bf16_round((n @ wl["wv"].T).reshape(T, hkv, 128))
        full = pd.causal_block_attention(q, np.zeros((0, hkv, 128)), np.zeros((0, hkv, 128)), k, v,
                                         1 / np.sqrt(128))
        for j in range(3):
            assert np.abs(a128[j][l] - full[128 * j:128 * (j + 1)]).max() <= 1e-12
            for half in range(2):
                blk = a64[2 * j + half][l]
                assert np.abs(blk - full[128 * j + 64 * half:128 * j + 64 * (half + 1)]).max() <= 1e-12
        h = h + full.reshape(T, hq * 128) @ wl["wo"].T
    assert np.all(pd.mae_curves(a128, a128) == 0.0)


def test_quantised_pseudo_decode_first_block_is_exact_and_error_appears_after():
    # block 0 reads no cache, so it equals the unquantised run; later blocks read the codec
    w, x = _tiny_model(45, layers=1)
    ref = pd.run(w, x, 4, 2, quantised=False)
    q = pd.run(w, x, 4, 2, quantised=True, k_bits=2, v_bits=2)
    m = pd.mae_curves(q, ref)
    assert m[0][0] == 0.0
    assert m[1][0] > 0 and m[2][0] > 0
    # and the quantised cache entries are exactly the oracle codec's dequantised tiles
    k = np.random.default_rng(46).standard_normal((128, 2, 128))
    got = pd.quantise_block(k, "K", 2, 8, True, True)
    e = o.encode_tile(k[:, 1], "K", 2)
    want = o.dequant_tile(e["codes"], e["S1"], e["s2"], e["Z"], e["g"], "K", original_basis=True)
    assert np.array_equal(got[:, 1], want)


def test_kv_token_scale_scales_the_keys_and_values_of_each_position():
    # the outlier variant's per-position multipliers act on the K and V projections only: with
    # them, the unquantised run equals ordinary causal attention (torch SDPA, fp64) over keys and
    # values scaled row by row, while the queries are unscaled
    w, x = _tiny_model(47, layers=1)
    hq, hkv, T = 4, 2, x.shape[0]
    ts = np.exp(np.random.default_rng(48).standard_normal(T))
    a = pd.run(w, x, hq, hkv, quantised=False, kv_token_scale=ts)
    wl, pos = w[0], np.arange(T)
    n = pd.rmsnorm(x)
    q = pd.bf16_round(pd.rope((n @ wl["wq"].T).reshape(T, hq, 128), pos))
    k = pd.bf16_round(pd.rope((n @ wl["wk"].T * ts[:, None]).reshape(T, hkv, 128), pos))
    v = pd.bf16_round((n @ wl["wv"].T * ts[:, None]).reshape(T, hkv, 128))
    mask = torch.tril(torch.ones(T, T, dtype=torch.bool))
    for h in range(hq):
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[:, h])[None], torch.from_numpy(k[:, h // 2])[None],
            torch.from_numpy(v[:, h // 2])[None], attn_mask=mask[None], scale=1 / np.sqrt(128))[0].numpy()
        for j in range(3):
            assert np.abs(a[j][0][:, h] - ref[128 * j:128 * (j + 1)]).max() <= 1e-12
    # all-ones multipliers are no multipliers
    plain = pd.run(w, x, hq, hkv, quantised=False)
    ones = pd.run(w, x, hq, hkv, quantised=False, kv_token_scale=np.ones(T))
    assert all(np.array_equal(p_, o_) for rp, ro in zip(plain, ones) for p_, o_ in zip(rp, ro))
