"""Python binding of libkvarn, the KVarN KV-cache codec for GB300 (sm_103a).

Argument marshalling only: every step of the codec runs in the CUDA kernels of libkvarn.so.  The
functions keep the C names and order of arguments; tensors are torch CUDA tensors (their
data_ptr() is passed) and the stream defaults to torch's current stream.  There is no fallback:
if the shared library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import synthetic  # noqa: F401  (seeded workload generators)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvarn.so")

KVARN_KIND_K = 0
KVARN_KIND_V = 1
KVARN_FLAG_NO_ROTATE = 1
KVARN_FLAG_NO_NORMALIZE = 2
KVARN_FLAG_FULL_TAIL = 4
PARAM_BYTES = 512
TILE = 128


KVARN_ERR_TIMEOUT = 5


class KvarnError(RuntimeError):
    def __init__(self, status: int, msg: str, code: int | None = None):
        super().__init__(f"{msg} (status {status})")
        self.status = status
        self.code = code  # kvarn_device_error's bits, for KVARN_ERR_TIMEOUT


class kvarn_config(ctypes.Structure):
    _fields_ = [("k_bits", ctypes.c_int32), ("v_bits", ctypes.c_int32),
                ("sinkhorn_iters", ctypes.c_int32), ("flags", ctypes.c_uint32)]

    def __repr__(self):
        return (f"kvarn_config(k_bits={self.k_bits}, v_bits={self.v_bits}, "
                f"sinkhorn_iters={self.sinkhorn_iters}, flags={self.flags})")


_lib = None
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t

_SIGNATURES = {
    "kvarn_config_from_preset": (_i32, [ctypes.c_char_p, ctypes.POINTER(kvarn_config)]),
    "kvarn_tile_code_bytes": (_sz, [_i32]),
    "kvarn_tile_param_bytes": (_sz, []),
    "kvarn_encode_blocks": (_i32, [ctypes.POINTER(kvarn_config), _i32, _vp, _i64, _vp, _vp, _vp, _vp]),
    "kvarn_encode_kv_blocks": (_i32, [ctypes.POINTER(kvarn_config), _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp,
                                      _vp, _vp]),
    "kvarn_dequant": (_i32, [ctypes.POINTER(kvarn_config), _i32, _vp, _vp, _vp, _i64, _i32, _vp, _vp]),
    "kvarn_decode_workspace_size": (_sz, [ctypes.POINTER(kvarn_config), _i32, _i32, _i32, _i32]),
    "kvarn_decode_attention": (_i32, [ctypes.POINTER(kvarn_config), _vp, _i32, _i32, _i32,
                                      _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp,
                                      ctypes.c_float, _vp, _sz, _vp, _vp]),
    "kvarn_decode_attention_sink": (_i32, [ctypes.POINTER(kvarn_config), _vp, _i32, _i32, _i32,
                                           _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp,
                                           _i32, _vp, _vp, ctypes.c_float, _vp, _sz, _vp, _vp]),
    "kvarn_decode_attention_static_ws": (_i32, [ctypes.POINTER(kvarn_config), _vp, _i32, _i32, _i32,
                                                _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp,
                                                _vp, _vp, ctypes.c_float, _vp, _vp]),
    "kvarn_device_error": (_i32, [ctypes.POINTER(ctypes.c_uint32)]),
    "kvarn_check_bounded_wait": (_i32, [ctypes.c_uint32, _vp]),
    "kvarn_append_workspace_size": (_sz, [_i32, _i32]),
    "kvarn_append_tokens": (_i32, [ctypes.POINTER(kvarn_config), _i32, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _vp,
                                   _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _sz, _vp]),
    "kvarn_status_string": (ctypes.c_char_p, [_i32]),
    "kvarn_last_error": (ctypes.c_char_p, []),
}


def load(path: str | None = None):
    """Load libkvarn.so (built by __graft_entry__.build()); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libkvarn.so not found at {path}: run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        lib = load()
        raise KvarnError(status, lib.kvarn_last_error().decode() or lib.kvarn_status_string(status).decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _need(t, dtype, numel, name):
    if not isinstance(t, torch.Tensor):
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")


def kvarn_config_from_preset(name: str) -> kvarn_config:
    cfg = kvarn_config()
    _check(load().kvarn_config_from_preset(name.encode(), ctypes.byref(cfg)))
    return cfg


def make_config(k_bits=2, v_bits=2, sinkhorn_iters=8, flags=0) -> kvarn_config:
    return kvarn_config(k_bits, v_bits, sinkhorn_iters, flags)


def kvarn_tile_code_bytes(bits: int) -> int:
    return int(load().kvarn_tile_code_bytes(bits))


def kvarn_tile_param_bytes() -> int:
    return int(load().kvarn_tile_param_bytes())


def kvarn_encode_blocks(cfg: kvarn_config, kind: int, x, codes, params, tile_scale, stream=None,
                        n_tiles: int | None = None):
    """x: [n, 128, 128] bf16 -> codes [n, code_bytes] u8, params [n, 512] u8, tile_scale [n] f32."""
    if n_tiles is None:
        n_tiles = x.shape[0]
    bits = cfg.k_bits if kind == KVARN_KIND_K else cfg.v_bits
    _need(x, torch.bfloat16, n_tiles * TILE * TILE, "x")
    _need(codes, torch.uint8, n_tiles * TILE * 16 * bits, "codes")
    _need(params, torch.uint8, n_tiles * PARAM_BYTES, "params")
    _need(tile_scale, torch.float32, n_tiles, "tile_scale")
    _check(load().kvarn_encode_blocks(ctypes.byref(cfg), kind, _ptr(x), n_tiles, _ptr(codes),
                                      _ptr(params), _ptr(tile_scale), _stream(stream)))


def kvarn_encode_kv_blocks(cfg: kvarn_config, k, v, k_codes, k_params, k_scale, v_codes, v_params,
                           v_scale, stream=None, n_tiles: int | None = None):
    """K and V blocks [n, 128, 128] bf16 encoded in one launch (same results as two
    kvarn_encode_blocks calls)."""
    if n_tiles is None:
        n_tiles = k.shape[0]
    for x, name in ((k, "k"), (v, "v")):
        _need(x, torch.bfloat16, n_tiles * TILE * TILE, name)
    _need(k_codes, torch.uint8, n_tiles * TILE * 16 * cfg.k_bits, "k_codes")
    _need(v_codes, torch.uint8, n_tiles * TILE * 16 * cfg.v_bits, "v_codes")
    for t, name in ((k_params, "k_params"), (v_params, "v_params")):
        _need(t, torch.uint8, n_tiles * PARAM_BYTES, name)
    for t, name in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, torch.float32, n_tiles, name)
    _check(load().kvarn_encode_kv_blocks(ctypes.byref(cfg), _ptr(k), _ptr(v), n_tiles, _ptr(k_codes),
                                         _ptr(k_params), _ptr(k_scale), _ptr(v_codes), _ptr(v_params),
                                         _ptr(v_scale), _stream(stream)))


def kvarn_append_workspace_size(B: int, Hkv: int) -> int:
    return int(load().kvarn_append_workspace_size(B, Hkv))


def kvarn_append_tokens(cfg: kvarn_config, k_new, v_new, seq_lens, k_tail, v_tail, k_codes, k_params, k_scale,
                        v_codes, v_params, v_scale, block_table, workspace, n_accept=None, stream=None):
    """Commit offered tokens k_new, v_new [B, Hkv, n_new, 128] bf16 (the first n_accept[b] of
    them, or all) to the tails / pools; seq_lens, tails and pools are updated in place."""
    B, Hkv, n_new = k_new.shape[0], k_new.shape[1], k_new.shape[2]
    max_tiles = block_table.shape[-1]
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, torch.bfloat16, B * Hkv * n_new * TILE, name)
    for t, name in ((k_tail, "k_tail"), (v_tail, "v_tail")):
        _need(t, torch.bfloat16, B * Hkv * TILE * TILE, name)
    _need(seq_lens, torch.int32, B, "seq_lens")
    _need(block_table, torch.int32, B * Hkv * max_tiles, "block_table")
    if n_accept is not None:
        _need(n_accept, torch.int32, B, "n_accept")
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load().kvarn_append_tokens(ctypes.byref(cfg), B, Hkv, _ptr(k_new), _ptr(v_new), n_new, _ptr(n_accept),
                                      _ptr(seq_lens), _ptr(k_tail), _ptr(v_tail), _ptr(k_codes), _ptr(k_params),
                                      _ptr(k_scale), _ptr(v_codes), _ptr(v_params), _ptr(v_scale),
                                      _ptr(block_table), max_tiles, _ptr(workspace), ws_bytes, _stream(stream)))


def kvarn_dequant(cfg: kvarn_config, kind: int, codes, params, tile_scale, out, original_basis=1,
                  stream=None, n_tiles: int | None = None):
    """Packed tiles -> float32 [n, 128, 128]."""
    if n_tiles is None:
        n_tiles = tile_scale.shape[0]
    bits = cfg.k_bits if kind == KVARN_KIND_K else cfg.v_bits
    _need(codes, torch.uint8, n_tiles * TILE * 16 * bits, "codes")
    _need(params, torch.uint8, n_tiles * PARAM_BYTES, "params")
    _need(tile_scale, torch.float32, n_tiles, "tile_scale")
    _need(out, torch.float32, n_tiles * TILE * TILE, "out")
    _check(load().kvarn_dequant(ctypes.byref(cfg), kind, _ptr(codes), _ptr(params),
                                _ptr(tile_scale), n_tiles, int(original_basis), _ptr(out),
                                _stream(stream)))


def kvarn_decode_workspace_size(cfg: kvarn_config, B: int, Hq: int, Hkv: int, max_tiles: int) -> int:
    return int(load().kvarn_decode_workspace_size(ctypes.byref(cfg), B, Hq, Hkv, max_tiles))


def kvarn_decode_attention(cfg: kvarn_config, q, Hkv: int, k_codes, k_params, k_scale, v_codes,
                           v_params, v_scale, block_table, seq_lens, k_tail, v_tail,
                           softmax_scale: float, workspace, out, seq_lens_host=None, stream=None,
                           k_sink=None, v_sink=None, sink_len: int = 0):
    """q: [B, Hq, 128] bf16; block_table: [B, Hkv, max_tiles] int32; seq_lens: [B] int32 (device);
    tails: [B, Hkv, 128, 128] bf16; out: [B, Hq, 128] float32.  With sink_len > 0 the first
    sink_len tokens come from k_sink / v_sink ([B, Hkv, 128, 128] bf16; kvarn_decode_attention_sink)."""
    B, Hq = q.shape[0], q.shape[1]
    max_tiles = block_table.shape[-1]
    _need(q, torch.bfloat16, B * Hq * TILE, "q")
    _need(block_table, torch.int32, B * Hkv * max_tiles, "block_table")
    _need(seq_lens, torch.int32, B, "seq_lens")
    _need(k_tail, torch.bfloat16, B * Hkv * TILE * TILE, "k_tail")
    _need(v_tail, torch.bfloat16, B * Hkv * TILE * TILE, "v_tail")
    _need(out, torch.float32, B * Hq * TILE, "out")
    host = None
    if seq_lens_host is not None:
        arr = (ctypes.c_int32 * B)(*[int(v) for v in seq_lens_host])
        host = ctypes.cast(arr, ctypes.c_void_p)
    ws_bytes = workspace.numel() * workspace.element_size() if isinstance(workspace, torch.Tensor) else 0
    if sink_len:
        _need(k_sink, torch.bfloat16, B * Hkv * TILE * TILE, "k_sink")
        _need(v_sink, torch.bfloat16, B * Hkv * TILE * TILE, "v_sink")
        _check(load().kvarn_decode_attention_sink(
            ctypes.byref(cfg), _ptr(q), B, Hq, Hkv, _ptr(k_codes), _ptr(k_params), _ptr(k_scale),
            _ptr(v_codes), _ptr(v_params), _ptr(v_scale), _ptr(block_table), max_tiles, _ptr(seq_lens),
            host, _ptr(k_sink), _ptr(v_sink), int(sink_len), _ptr(k_tail), _ptr(v_tail),
            float(softmax_scale), _ptr(workspace), ws_bytes, _ptr(out), _stream(stream)))
        return
    _check(load().kvarn_decode_attention(
        ctypes.byref(cfg), _ptr(q), B, Hq, Hkv, _ptr(k_codes), _ptr(k_params), _ptr(k_scale),
        _ptr(v_codes), _ptr(v_params), _ptr(v_scale), _ptr(block_table), max_tiles, _ptr(seq_lens),
        host, _ptr(k_tail), _ptr(v_tail), float(softmax_scale), _ptr(workspace), ws_bytes,
        _ptr(out), _stream(stream)))


def kvarn_decode_attention_static_ws(cfg: kvarn_config, q, Hkv: int, k_codes, k_params, k_scale,
                                     v_codes, v_params, v_scale, block_table, seq_lens, k_tail,
                                     v_tail, softmax_scale: float, out, seq_lens_host=None,
                                     stream=None):
    """kvarn_decode_attention without a workspace argument: the split-K scratch is a fixed device
    array owned by the library (for callers that cannot allocate device memory at this point)."""
    B, Hq = q.shape[0], q.shape[1]
    max_tiles = block_table.shape[-1]
    _need(q, torch.bfloat16, B * Hq * TILE, "q")
    _need(block_table, torch.int32, B * Hkv * max_tiles, "block_table")
    _need(seq_lens, torch.int32, B, "seq_lens")
    _need(k_tail, torch.bfloat16, B * Hkv * TILE * TILE, "k_tail")
    _need(v_tail, torch.bfloat16, B * Hkv * TILE * TILE, "v_tail")
    _need(out, torch.float32, B * Hq * TILE, "out")
    host = None
    if seq_lens_host is not None:
        arr = (ctypes.c_int32 * B)(*[int(v) for v in seq_lens_host])
        host = ctypes.cast(arr, ctypes.c_void_p)
    _check(load().kvarn_decode_attention_static_ws(
        ctypes.byref(cfg), _ptr(q), B, Hq, Hkv, _ptr(k_codes), _ptr(k_params), _ptr(k_scale),
        _ptr(v_codes), _ptr(v_params), _ptr(v_scale), _ptr(block_table), max_tiles, _ptr(seq_lens),
        host, _ptr(k_tail), _ptr(v_tail), float(softmax_scale), _ptr(out), _stream(stream)))


def kvarn_device_error() -> int:
    """The device error bits (read and cleared).  Raises KvarnError (status KVARN_ERR_TIMEOUT, the
    bits in .code) when a bounded device wait gave up."""
    v = ctypes.c_uint32(0)
    lib = load()
    st = lib.kvarn_device_error(ctypes.byref(v))
    if st == KVARN_ERR_TIMEOUT:
        raise KvarnError(st, lib.kvarn_last_error().decode(), code=int(v.value))
    _check(st)
    return int(v.value)


def kvarn_check_bounded_wait(limit_us: int, stream=None):
    """Enqueue the self-check kernel whose bounded wait gives up after limit_us microseconds."""
    _check(load().kvarn_check_bounded_wait(int(limit_us), _stream(stream)))


def kvarn_status_string(status: int) -> str:
    return load().kvarn_status_string(status).decode()
