"""libkvarn's calls inside a CUDA graph: the library never allocates, never synchronises and launches
only on the stream it is given, so a serving loop can capture encode, append and decode once and
replay them without the per-call host cost.  A replay must give the same bytes as the eager call."""
import math

import pytest
import torch

from tests.test_gpu_decode import build_cache

pytestmark = pytest.mark.gpu


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()  # first call outside the capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    return g


def test_decode_and_encode_replay_bit_identical(kv):
    cfg = kv.kvarn_config_from_preset("kvarn_k2v2_g128")
    lens = [0, 77, 128, 5 * 128 + 3, 40 * 128 + 127]  # empty, tail only, one block, ragged
    B, hkv, hq = len(lens), 2, 8
    c = build_cache(kv, cfg, B, hkv, lens, seed=91)
    q = kv.synthetic.queries(91, B, hq, device="cuda")
    ws = torch.empty(kv.kvarn_decode_workspace_size(cfg, B, hq, hkv, c["nt"]), dtype=torch.uint8, device="cuda")
    out = torch.empty(B, hq, 128, device="cuda")
    kc, kp, ks = c["pools"]["k"]
    vc, vp, vs = c["pools"]["v"]

    def decode():
        kv.kvarn_decode_attention(cfg, q, hkv, kc, kp, ks, vc, vp, vs, c["table"], c["seq_lens"], c["k_tail"],
                                  c["v_tail"], 1 / math.sqrt(128), ws, out)

    decode()
    torch.cuda.synchronize()
    eager = out.clone()
    g = _capture(decode)
    out.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)

    x = kv.synthetic.outlier_kv(92, 6, 128, device="cuda")[0].reshape(6, 128, 128)
    outs = [torch.empty(6, 4096, dtype=torch.uint8, device="cuda"), torch.empty(6, 512, dtype=torch.uint8, device="cuda"),
            torch.empty(6, device="cuda")]
    outs += [torch.empty_like(t) for t in outs]

    def encode():
        kv.kvarn_encode_kv_blocks(cfg, x, x, *outs)

    encode()
    torch.cuda.synchronize()
    ref = [t.clone() for t in outs]
    g = _capture(encode)
    for t in outs:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(outs, ref))
    assert kv.kvarn_device_error() == 0


def test_append_replay_matches_eager_calls(kv):
    # the same sequence of one-token appends, eager and replayed, leaves identical tails, lengths
    # and pool tiles (a block completes along the way)
    cfg = kv.kvarn_config_from_preset("kvarn_k2v2_g128")
    B, hkv, mt, steps = 3, 2, 4, 140
    g = torch.Generator(device="cpu").manual_seed(93)
    toks = [torch.randn(B, hkv, 1, 128, generator=g).to(torch.bfloat16).cuda() for _ in range(steps)]
    table = torch.randperm(B * hkv * mt, generator=g).to(torch.int32).reshape(B, hkv, mt).cuda()

    def state():
        n = B * hkv * mt
        pools = [torch.zeros(n, 4096, dtype=torch.uint8, device="cuda"), torch.zeros(n, 512, dtype=torch.uint8, device="cuda"),
                 torch.zeros(n, device="cuda"), torch.zeros(n, 4096, dtype=torch.uint8, device="cuda"),
                 torch.zeros(n, 512, dtype=torch.uint8, device="cuda"), torch.zeros(n, device="cuda")]
        return dict(lens=torch.full((B,), 100, dtype=torch.int32, device="cuda"),
                    kt=torch.zeros(B, hkv, 128, 128, dtype=torch.bfloat16, device="cuda"),
                    vt=torch.zeros(B, hkv, 128, 128, dtype=torch.bfloat16, device="cuda"), pools=pools,
                    ws=torch.empty(kv.kvarn_append_workspace_size(B, hkv), dtype=torch.uint8, device="cuda"),
                    tok=torch.empty(B, hkv, 1, 128, dtype=torch.bfloat16, device="cuda"))

    eager, graph = state(), state()
    for t in toks:
        kv.kvarn_append_tokens(cfg, t, t, eager["lens"], eager["kt"], eager["vt"], *eager["pools"], table, eager["ws"])

    def step():
        s = graph
        kv.kvarn_append_tokens(cfg, s["tok"], s["tok"], s["lens"], s["kt"], s["vt"], *s["pools"], table, s["ws"])

    # the capture's warm-up call appends a token too: feed it the first one, then replay the rest
    graph["tok"].copy_(toks[0])
    gr = _capture(step)
    graph["lens"].fill_(101)  # the warm-up call appended toks[0]; the capture itself ran nothing
    for t in toks[1:]:
        graph["tok"].copy_(t)
        gr.replay()
    torch.cuda.synchronize()
    assert kv.kvarn_device_error() == 0
    assert torch.equal(eager["lens"], graph["lens"])
    assert torch.equal(eager["kt"], graph["kt"]) and torch.equal(eager["vt"], graph["vt"])
    assert all(torch.equal(a, b) for a, b in zip(eager["pools"], graph["pools"]))
