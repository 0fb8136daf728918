"""Appending decode-step tokens through libkvarn (tails, completed blocks encoded into their pool
slots, speculative accept counts) against the oracle's append semantics."""
import numpy as np
import pytest
import torch

from oracle import kvarn_oracle as o

pytestmark = pytest.mark.gpu


def _valid_rows(L, full_tail):
    if full_tail:
        return ((L - 1) % 128) + 1 if L > 0 else 0
    return L % 128


@pytest.mark.parametrize("k_bits,v_bits,flags", [(2, 2, 0), (4, 2, 4)])
def test_append_steps_match_oracle(kv, k_bits, v_bits, flags):
    cfg = kv.make_config(k_bits, v_bits, 8, flags)
    full = bool(flags & 4)
    B, Hkv, max_tiles = 5, 2, 6
    g = torch.Generator(device="cpu").manual_seed(70)
    lens = [0, 1, 127, 128, 300]
    kt = torch.zeros(B, Hkv, 128, 128, dtype=torch.bfloat16)
    vt = torch.zeros_like(kt)
    for b, L in enumerate(lens):
        r = _valid_rows(L, full)
        kt[b, :, :r] = torch.randn(Hkv, r, 128, generator=g).to(torch.bfloat16)
        vt[b, :, :r] = torch.randn(Hkv, r, 128, generator=g).to(torch.bfloat16)
    n_tiles = B * Hkv * max_tiles
    table = torch.randperm(n_tiles, generator=g).to(torch.int32).reshape(B, Hkv, max_tiles)
    pools = [torch.zeros(n_tiles, 2048 * k_bits, dtype=torch.uint8), torch.zeros(n_tiles, 512, dtype=torch.uint8),
             torch.zeros(n_tiles), torch.zeros(n_tiles, 2048 * v_bits, dtype=torch.uint8),
             torch.zeros(n_tiles, 512, dtype=torch.uint8), torch.zeros(n_tiles)]
    d_pools = [t.cuda() for t in pools]
    d_kt, d_vt, d_table = kt.cuda(), vt.cuda(), table.cuda()
    d_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ws = torch.empty(kv.kvarn_append_workspace_size(B, Hkv), dtype=torch.uint8, device="cuda")
    o_lens, o_kt, o_vt = np.array(lens), kt.float().numpy(), vt.float().numpy()
    written = {}
    for n_new, accept in ((1, None), (128, [128, 5, 0, 64, 1]), (7, None), (100, [100, 100, 28, 0, 99]),
                          (128, [127, 3, 128, 1, 0])):
        kn = torch.randn(B, Hkv, n_new, 128, generator=g).to(torch.bfloat16)
        vn = torch.randn(B, Hkv, n_new, 128, generator=g).to(torch.bfloat16)
        acc = None if accept is None else torch.tensor(accept, dtype=torch.int32, device="cuda")
        kv.kvarn_append_tokens(cfg, kn.cuda(), vn.cuda(), d_lens, d_kt, d_vt, *d_pools, d_table, ws, n_accept=acc)
        torch.cuda.synchronize()
        assert kv.kvarn_device_error() == 0
        o_lens, o_kt, o_vt, blocks = o.append_tokens(kn.float().numpy(), vn.float().numpy(),
                                                     accept if accept is not None else [n_new] * B, o_lens,
                                                     o_kt, o_vt, table.numpy(), full)
        assert d_lens.cpu().tolist() == list(o_lens)
        for b in range(B):
            r = _valid_rows(int(o_lens[b]), full)
            assert torch.equal(d_kt[b, :, :r].float().cpu(), torch.from_numpy(o_kt[b, :, :r]).float())
            assert torch.equal(d_vt[b, :, :r].float().cpu(), torch.from_numpy(o_vt[b, :, :r]).float())
        for b, h, tile, kb, vb in blocks:
            written[tile] = (kb, vb)
    # every completed block sits in its slot, encoded exactly as kvarn_encode_blocks encodes it
    assert len(written) > 0
    tiles = sorted(written)
    kb = torch.from_numpy(np.stack([written[t][0] for t in tiles])).to(torch.bfloat16).cuda()
    vb = torch.from_numpy(np.stack([written[t][1] for t in tiles])).to(torch.bfloat16).cuda()
    ref_k = [torch.empty(len(tiles), 2048 * k_bits, dtype=torch.uint8, device="cuda"),
             torch.empty(len(tiles), 512, dtype=torch.uint8, device="cuda"), torch.empty(len(tiles), device="cuda")]
    ref_v = [torch.empty(len(tiles), 2048 * v_bits, dtype=torch.uint8, device="cuda"),
             torch.empty(len(tiles), 512, dtype=torch.uint8, device="cuda"), torch.empty(len(tiles), device="cuda")]
    kv.kvarn_encode_blocks(cfg, kv.KVARN_KIND_K, kb, *ref_k)
    kv.kvarn_encode_blocks(cfg, kv.KVARN_KIND_V, vb, *ref_v)
    idx = torch.tensor(tiles, device="cuda")
    for got, want in zip(d_pools, ref_k + ref_v):
        assert torch.equal(got[idx], want)
    # slots no block was written to stay untouched
    untouched = torch.tensor(sorted(set(range(n_tiles)) - set(tiles)), device="cuda")
    assert torch.all(d_pools[0][untouched] == 0) and torch.all(d_pools[2][untouched] == 0)
    print("blocks written", len(tiles))


def test_append_without_a_block_table_slot_sets_the_device_error(kv):
    cfg = kv.make_config(2, 2, 8, 0)
    B, Hkv = 1, 1
    d_lens = torch.tensor([127], dtype=torch.int32, device="cuda")  # the next token completes block 0
    kt = torch.zeros(B, Hkv, 128, 128, dtype=torch.bfloat16, device="cuda")
    vt = torch.zeros_like(kt)
    pools = [torch.zeros(1, 4096, dtype=torch.uint8, device="cuda"), torch.zeros(1, 512, dtype=torch.uint8, device="cuda"),
             torch.zeros(1, device="cuda"), torch.zeros(1, 4096, dtype=torch.uint8, device="cuda"),
             torch.zeros(1, 512, dtype=torch.uint8, device="cuda"), torch.zeros(1, device="cuda")]
    table = torch.zeros(B, Hkv, 0, dtype=torch.int32, device="cuda")  # max_tiles = 0: no slot
    ws = torch.empty(kv.kvarn_append_workspace_size(B, Hkv), dtype=torch.uint8, device="cuda")
    kn = torch.ones(B, Hkv, 1, 128, dtype=torch.bfloat16, device="cuda")
    kv.kvarn_append_tokens(cfg, kn, kn, d_lens, kt, vt, *pools, table, ws)
    assert kv.kvarn_device_error() == 4
    assert d_lens.item() == 127 and torch.all(kt == 0)
