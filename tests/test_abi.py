"""The C-ABI library builds, loads and exports every call include/kvarn.h declares; host-side
argument validation returns the documented status without touching a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvarn.h")


@pytest.fixture(scope="module")
def lib():
    from bit_kv_cache_kvarn_gb300 import _build
    import bit_kv_cache_kvarn_gb300 as kv

    srcs = [os.path.join(_build.CSRC, s) for s in os.listdir(_build.CSRC)] + [HEADER]
    if not os.path.exists(_build.LIB) or os.path.getmtime(_build.LIB) < max(map(os.path.getmtime, srcs)):
        _build.build()
    return kv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvarn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for want in ("kvarn_encode_blocks", "kvarn_dequant", "kvarn_decode_attention",
                 "kvarn_decode_workspace_size", "kvarn_config_from_preset"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (kvarn_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_presets_and_sizes(lib):
    import bit_kv_cache_kvarn_gb300 as kv

    c = kv.kvarn_config_from_preset("kvarn_k4v2_g128")
    assert (c.k_bits, c.v_bits, c.sinkhorn_iters, c.flags) == (4, 2, 8, 0)
    c = kv.kvarn_config_from_preset("kvarn_k2v2_g128")
    assert (c.k_bits, c.v_bits, c.sinkhorn_iters) == (2, 2, 8)
    for name, want in (("kvarn_k4v4_g128", (4, 4, 8, 0)), ("kvarn_k2v4_g128", (2, 4, 8, 0)),
                       ("hadamard_k2v2_g128", (2, 2, 0, 2)), ("kivi_k2v2_g128", (2, 2, 0, 3))):
        c = kv.kvarn_config_from_preset(name)
        assert (c.k_bits, c.v_bits, c.sinkhorn_iters, c.flags) == want
    with pytest.raises(kv.KvarnError, match="unknown preset"):
        kv.kvarn_config_from_preset("kvarn_k3v3")
    assert kv.kvarn_tile_code_bytes(2) == 4096 and kv.kvarn_tile_code_bytes(4) == 8192
    assert kv.kvarn_tile_code_bytes(3) == 0 and kv.kvarn_tile_param_bytes() == 512
    for s in range(6):
        assert kv.kvarn_status_string(s).startswith("KVARN_")
    assert "TIMEOUT" in kv.kvarn_status_string(5)


def _cfg(**kw):
    import bit_kv_cache_kvarn_gb300 as kv

    return kv.make_config(**kw)


FAKE = 0x7F0000000000  # a 16-byte aligned address the calls must reject or never touch


def test_encode_validation_needs_no_gpu(lib):
    cfg = _cfg()
    enc = lib.kvarn_encode_blocks
    assert enc(None, 0, FAKE, 1, FAKE, FAKE, FAKE, None) == 1
    assert enc(ctypes.byref(_cfg(k_bits=3)), 0, FAKE, 1, FAKE, FAKE, FAKE, None) == 1
    assert enc(ctypes.byref(_cfg(sinkhorn_iters=65)), 0, FAKE, 1, FAKE, FAKE, FAKE, None) == 1
    assert enc(ctypes.byref(_cfg(flags=8)), 0, FAKE, 1, FAKE, FAKE, FAKE, None) == 1
    assert enc(ctypes.byref(cfg), 2, FAKE, 1, FAKE, FAKE, FAKE, None) == 1
    assert enc(ctypes.byref(cfg), 0, FAKE, -1, FAKE, FAKE, FAKE, None) == 1
    assert enc(ctypes.byref(cfg), 0, None, 1, FAKE, FAKE, FAKE, None) == 1
    assert enc(ctypes.byref(cfg), 0, FAKE + 8, 1, FAKE, FAKE, FAKE, None) == 1
    assert b"aligned" in lib.kvarn_last_error()
    assert enc(ctypes.byref(cfg), 0, FAKE, 1, FAKE, FAKE, FAKE + 2, None) == 1
    assert enc(ctypes.byref(cfg), 0, None, 0, None, None, None, None) == 0  # empty: no-op


def test_fused_encode_validation_needs_no_gpu(lib):
    cfg = _cfg()
    enc = lib.kvarn_encode_kv_blocks
    assert enc(None, FAKE, FAKE, 1, *[FAKE] * 6, None) == 1
    assert enc(ctypes.byref(cfg), FAKE, FAKE, -1, *[FAKE] * 6, None) == 1
    assert enc(ctypes.byref(cfg), FAKE, None, 1, *[FAKE] * 6, None) == 1
    assert b"v_bf16" in lib.kvarn_last_error()
    assert enc(ctypes.byref(cfg), FAKE, FAKE, 1, FAKE, FAKE, FAKE + 2, FAKE, FAKE, FAKE, None) == 1
    assert enc(ctypes.byref(cfg), FAKE, FAKE, 1, FAKE, FAKE, FAKE, FAKE + 8, FAKE, FAKE, None) == 1
    assert enc(ctypes.byref(_cfg(v_bits=3)), FAKE, FAKE, 1, *[FAKE] * 6, None) == 1
    assert enc(ctypes.byref(cfg), None, None, 0, *[None] * 6, None) == 0


def test_dequant_validation_needs_no_gpu(lib):
    cfg = _cfg()
    dq = lib.kvarn_dequant
    assert dq(ctypes.byref(cfg), 0, FAKE, FAKE, FAKE, 1, 2, FAKE, None) == 1
    assert dq(ctypes.byref(cfg), 0, FAKE, FAKE, FAKE, 2 ** 31, 0, FAKE, None) == 1
    assert dq(ctypes.byref(cfg), 0, FAKE, FAKE, FAKE, 1, 0, FAKE + 4, None) == 1
    assert dq(ctypes.byref(cfg), 1, None, None, None, 0, 1, None, None) == 0


def _decode(lib, cfg, B=2, Hq=8, Hkv=2, max_tiles=4, lens_host=None, ws=FAKE, ws_bytes=1 << 30,
            scale=0.1, tail=FAKE):
    host = None
    if lens_host is not None:
        arr = (ctypes.c_int32 * len(lens_host))(*lens_host)
        host = ctypes.cast(arr, ctypes.c_void_p)
    return lib.kvarn_decode_attention(ctypes.byref(cfg), FAKE, B, Hq, Hkv, FAKE, FAKE, FAKE, FAKE,
                                      FAKE, FAKE, FAKE, max_tiles, FAKE, host, tail, FAKE,
                                      ctypes.c_float(scale), ws, ws_bytes, FAKE, None)


def test_sink_decode_validation_needs_no_gpu(lib):
    cfg = _cfg()

    def call(sink_len, sink=FAKE, lens_host=None, B=2):
        host = None
        if lens_host is not None:
            arr = (ctypes.c_int32 * len(lens_host))(*lens_host)
            host = ctypes.cast(arr, ctypes.c_void_p)
        return lib.kvarn_decode_attention_sink(ctypes.byref(cfg), FAKE, B, 8, 2, FAKE, FAKE, FAKE, FAKE, FAKE,
                                               FAKE, FAKE, 4, FAKE, host, sink, sink, sink_len, FAKE, FAKE,
                                               ctypes.c_float(0.1), FAKE, 1 << 30, FAKE, None)

    assert call(129) == 1
    assert call(-1) == 1
    assert call(32, sink=None) == 1
    assert b"k_sink" in lib.kvarn_last_error()
    assert call(32, lens_host=[5, 32 + 4 * 128 + 128]) == 1  # body over 128*max_tiles + 127
    assert b"0..671" in lib.kvarn_last_error()
    assert call(32, B=0) == 0


def test_decode_validation_needs_no_gpu(lib):
    cfg = _cfg()
    assert _decode(lib, cfg, Hq=6, Hkv=4) == 1
    # any whole group is accepted (B = 0: validated, nothing enqueued)
    for hq, hkv in ((12, 4), (32, 2), (5, 1), (96, 8)):
        assert _decode(lib, cfg, B=0, Hq=hq, Hkv=hkv) == 0, (hq, hkv)
    assert _decode(lib, cfg, B=0, Hq=65536, Hkv=1) == 1
    assert _decode(lib, cfg, B=-1) == 1
    assert _decode(lib, cfg, max_tiles=-1) == 1
    assert _decode(lib, cfg, scale=float("inf")) == 1
    assert _decode(lib, cfg, tail=None) == 1
    assert _decode(lib, cfg, lens_host=[5, 4 * 128 + 128]) == 1  # over 128*max_tiles + 127
    assert _decode(lib, cfg, lens_host=[-1, 3]) == 1
    # the full FP16 window allows one more token per sequence, and only that
    full = _cfg(flags=4)
    assert _decode(lib, full, lens_host=[5, 4 * 128 + 129]) == 1
    assert b"0..640" in lib.kvarn_last_error()
    assert _decode(lib, _cfg(flags=8), lens_host=[5, 6]) == 1
    assert _decode(lib, cfg, ws_bytes=16) == 4
    assert b"workspace" in lib.kvarn_last_error()
    assert _decode(lib, cfg, B=0) == 0


def test_workspace_plan(lib):
    import bit_kv_cache_kvarn_gb300 as kv

    cfg = _cfg()

    def piece(units, m):
        # piece granularity P: 16, halved (down to 2) while B Hkv (table width) < 512 P
        p = 16
        while p > 2 and units * m < 512 * p:
            p //= 2
        return p

    def expected(B, Hq, Hkv, max_tiles):
        # enough for every table width up to max_tiles (a narrower table may take a finer P), 256-byte
        # multiple: the widest width of each finer granularity gives its largest slot count
        units = B * Hkv
        P = piece(units, max_tiles)
        s = max(1, -(-max_tiles // P))
        q = P // 2
        while q >= 2 and units > 0:
            m = min(max_tiles, -(-1024 * q // units) - 1)
            if m > 0:
                s = max(s, -(-m // q))
            q //= 2
        return (B * Hq * (s + 1) * 528 + 255) // 256 * 256

    assert kv.kvarn_decode_workspace_size(cfg, 16, 32, 8, 256) == expected(16, 32, 8, 256)
    assert kv.kvarn_decode_workspace_size(cfg, 4, 40, 10, 1024) == expected(4, 40, 10, 1024)
    assert kv.kvarn_decode_workspace_size(cfg, 1, 4, 1, 0) == expected(1, 4, 1, 0)
    # small calls take finer pieces: B = 1, 8 kv heads, 32 tiles -> P = 2, 17 slots per head
    assert kv.kvarn_decode_workspace_size(cfg, 1, 32, 8, 32) == expected(1, 32, 8, 32) == 32 * 17 * 528
    # 2 x 8 units x 256 tiles = 4096 stream tiles: P = 8 (33 slots), but a 255-tile table takes P = 4
    # (65 slots), so the workspace holds 65
    assert expected(2, 32, 8, 256) == 2 * 32 * 65 * 528
    assert kv.kvarn_decode_workspace_size(cfg, 2, 32, 8, 256) == expected(2, 32, 8, 256)
    assert kv.kvarn_decode_workspace_size(cfg, 1, 6, 4, 1) == 0


def test_workspace_covers_every_narrower_table(lib):
    # brute force: a workspace sized for max_tiles serves any table width m <= max_tiles, and it
    # never shrinks as max_tiles grows
    import bit_kv_cache_kvarn_gb300 as kv

    cfg = _cfg()

    def needed(B, Hq, Hkv, m):
        units, p = B * Hkv, 16
        while p > 2 and units * m < 512 * p:
            p //= 2
        return B * Hq * (max(1, -(-m // p)) + 1) * 528

    for B, Hkv in ((1, 1), (1, 8), (2, 8), (3, 5), (16, 8)):
        Hq = 2 * Hkv
        prev, worst = 0, 0
        for m in range(0, 1200):
            worst = max(worst, needed(B, Hq, Hkv, m))
            got = kv.kvarn_decode_workspace_size(cfg, B, Hq, Hkv, m)
            assert got >= worst, (B, Hkv, m, got, worst)
            assert got >= prev, (B, Hkv, m)
            prev = got


def test_append_validation_needs_no_gpu(lib):
    cfg = _cfg()

    def call(B=2, Hkv=2, n_new=4, ws_bytes=1 << 30, ws=FAKE, seq=FAKE, max_tiles=4):
        return lib.kvarn_append_tokens(ctypes.byref(cfg), B, Hkv, FAKE, FAKE, n_new, None, seq, FAKE, FAKE,
                                       FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, max_tiles, ws, ws_bytes, None)

    assert call(n_new=0) == 1 and call(n_new=129) == 1
    assert call(Hkv=0) == 1 and call(B=-1) == 1 and call(max_tiles=-1) == 1
    assert call(seq=None) == 1
    assert b"seq_lens" in lib.kvarn_last_error()
    assert call(ws=FAKE + 16) == 1  # the workspace must be 256-byte aligned
    assert call(ws_bytes=100) == 4
    assert call(B=0) == 0
    assert lib.kvarn_append_workspace_size(2, 2) >= 2 * 4 * 32768
    assert lib.kvarn_append_workspace_size(0, 0) == 0


def test_bounded_wait_check_validation_needs_no_gpu(lib):
    # the self-check's limit is validated on the host; nothing is enqueued on error
    assert lib.kvarn_check_bounded_wait(0, None) == 1
    assert lib.kvarn_check_bounded_wait(1000001, None) == 1
    assert b"limit_us" in lib.kvarn_last_error()
    assert lib.kvarn_status_string(5) == b"KVARN_ERR_TIMEOUT: a bounded device wait gave up"
