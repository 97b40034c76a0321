"""Thin ctypes binding of libkvarn.so (include/kvarn.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. PyTorch supplies device memory and the current stream. There is no
fallback: if the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import _build

TILE = 128
DEFAULT_ITERS = 4
LAUNCH_PDL = 1       # KVARN_LAUNCH_PDL
LAUNCH_PREFETCH = 2  # KVARN_LAUNCH_PREFETCH
DEVERR_WAIT = 1      # KVARN_DEVERR_WAIT
DEVERR_RECORD = 2    # KVARN_DEVERR_RECORD
DEVERR_WINDOW = 4    # KVARN_DEVERR_WINDOW
DEVERR_SELFTEST = 8  # KVARN_DEVERR_SELFTEST

_lib = None


class KvarnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = _L().kvarn_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{fn} failed: {msg} ({status})")
        self.status = status


class Layout(ctypes.Structure):
    """Mirror of kvarn_layout_t."""
    _fields_ = [("version", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("tile_tokens", ctypes.c_int32), ("sinkhorn_iters", ctypes.c_int32),
                ("k_bits", ctypes.c_int32), ("v_bits", ctypes.c_int32),
                ("v_group", ctypes.c_int32), ("v_groups", ctypes.c_int32),
                ("record_bytes", ctypes.c_int64),
                ("off_k_codes", ctypes.c_int64), ("off_v_codes", ctypes.c_int64),
                ("off_k_delta", ctypes.c_int64), ("off_k_lo", ctypes.c_int64),
                ("off_k_s", ctypes.c_int64), ("off_k_r", ctypes.c_int64),
                ("off_v_delta", ctypes.c_int64), ("off_v_lo", ctypes.c_int64),
                ("off_v_r", ctypes.c_int64), ("off_v_s", ctypes.c_int64)]


def library_path() -> str:
    return _build.LIB


def _L():
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libkvarn.so is not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        vp, i64, c_int, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        u32, f32, lay = ctypes.c_uint, ctypes.c_float, ctypes.POINTER(Layout)
        lib.kvarn_status_string.restype = ctypes.c_char_p
        lib.kvarn_status_string.argtypes = [c_int]
        lib.kvarn_layout.argtypes = [c_int, c_int, lay]
        lib.kvarn_layout_scales.argtypes = [c_int, c_int, c_int, lay]
        lib.kvarn_layout_ex.argtypes = [c_int, c_int, c_int, c_int, lay]
        lib.kvarn_get_device_error.argtypes = [ctypes.POINTER(u32), c_int]
        lib.kvarn_selftest_bounded_wait.argtypes = [u32, vp]
        lib.kvarn_rotate_query.argtypes = [vp, vp, i64, c_int, vp]
        lib.kvarn_compress_tile.argtypes = [vp, vp, i64, i64, vp, vp, i64, vp, i64, lay, vp]
        lib.kvarn_append_window.argtypes = [vp, vp, i64, vp, vp, c_int, vp, vp, c_int, c_int, c_int,
                                            u32, vp]
        lib.kvarn_decode_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int, c_int, c_int,
                                                     ctypes.POINTER(sz)]
        lib.kvarn_decode_attention.argtypes = [vp, vp, i64, vp, vp, vp, vp, vp, vp, c_int, c_int,
                                               c_int, c_int, c_int, c_int, f32, lay, vp, sz, vp,
                                               u32, vp]
        lib.kvarn_decode_attention_noalloc.argtypes = [vp, vp, i64, vp, vp, vp, vp, vp, vp, c_int,
                                                       c_int, c_int, c_int, c_int, c_int, f32, lay,
                                                       vp, u32, vp]
        lib.kvarn_decode_split.argtypes = [vp, vp, i64, vp, vp, vp, vp, vp, vp, c_int, c_int, c_int,
                                           c_int, c_int, c_int, f32, lay, vp, sz, u32, vp]
        lib.kvarn_decode_combine.argtypes = [vp, sz, c_int, c_int, c_int, c_int, c_int, c_int, vp,
                                             u32, vp]
        lib.kvarn_window_advance.argtypes = [vp, vp, vp, c_int, c_int, c_int, c_int, u32, vp]
        lib.kvarn_prefill_attention.argtypes = [vp, c_int, i64, vp, i64, vp, c_int, c_int, vp, vp,
                                                c_int, c_int, c_int, c_int, c_int, c_int, f32, lay,
                                                vp, sz, vp, vp]
        lib.kvarn_prefill_attention_cached.argtypes = [vp, c_int, i64, vp, i64, vp, c_int, c_int,
                                                       vp, vp, c_int, c_int, c_int, c_int, c_int,
                                                       c_int, f32, lay, vp, sz, c_int, c_int, vp, vp]
        lib.kvarn_prefill_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int, ctypes.POINTER(sz)]
        for name in ("kvarn_layout", "kvarn_layout_scales", "kvarn_layout_ex", "kvarn_rotate_query",
                     "kvarn_compress_tile", "kvarn_get_device_error", "kvarn_selftest_bounded_wait",
                     "kvarn_append_window", "kvarn_decode_workspace_bytes",
                     "kvarn_decode_attention", "kvarn_decode_attention_noalloc",
                     "kvarn_decode_split", "kvarn_decode_combine", "kvarn_window_advance",
                     "kvarn_prefill_attention", "kvarn_prefill_workspace_bytes",
                     "kvarn_prefill_attention_cached"):
            getattr(lib, name).restype = c_int
        _lib = lib
    return _lib


def declared_functions(header: str) -> list:
    """Names of the functions include/kvarn.h declares."""
    with open(header) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(kvarn_\w+)\s*\(", text, flags=re.M)))


def _check(fn: str, rc: int):
    if rc != 0:
        raise KvarnError(fn, rc)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, name, dtype, device=None):
    """A contiguous CUDA tensor of `dtype` (on `device`, when given): anything
    else would reach the kernels as a pointer they cannot use."""
    if not (isinstance(t, torch.Tensor) and t.is_cuda):
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def _all_dev(device, **tensors):
    """_dev for several (tensor, dtype) pairs that must share one device."""
    for name, (t, dtype) in tensors.items():
        _dev(t, name, dtype, device)


def device_error(clear: bool = True) -> int:
    """KVARN_DEVERR_* bits that kernels of this library set on the current
    device since the word was last cleared (kvarn_get_device_error; this
    synchronises the device)."""
    bits = ctypes.c_uint()
    _check("kvarn_get_device_error", _L().kvarn_get_device_error(ctypes.byref(bits), int(bool(clear))))
    return int(bits.value)


def selftest_bounded_wait(timeout_us: int, stream=None):
    """One kernel whose wait runs out after timeout_us and reports
    DEVERR_SELFTEST (kvarn_selftest_bounded_wait)."""
    _check("kvarn_selftest_bounded_wait",
           _L().kvarn_selftest_bounded_wait(int(timeout_us), _stream(stream)))


def layout(head_dim: int, iters: int = DEFAULT_ITERS, scale_bits: int = 32,
           v_bits: int = 2) -> Layout:
    """Record layout: fp32 scale fields (scale_bits 32, the default) or
    binary16 ones (16, the f16-scale layout; same codes), and 2-bit value
    codes (the k4v2 preset) or 4-bit ones (v_bits 4, the k4v4 variant)."""
    L = Layout()
    _check("kvarn_layout_ex",
           _L().kvarn_layout_ex(head_dim, iters, scale_bits, v_bits, ctypes.byref(L)))
    return L


def rotate_query(q: torch.Tensor, out: torch.Tensor = None, stream=None) -> torch.Tensor:
    """H q for every row (last axis = head_dim)."""
    _dev(q, "q", torch.float32)
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", torch.float32)
    D = q.shape[-1]
    _check("kvarn_rotate_query",
           _L().kvarn_rotate_query(_ptr(q), _ptr(out), q.numel() // D, D, _stream(stream)))
    return out


def compress_tile(k_raw, v_raw, src_row0, tiles, dst_record, lay: Layout, stream=None):
    """k_raw, v_raw: fp32 [n_rows][row_stride] (2-D view of any row-major
    buffer); src_row0, dst_record: int64 [n_units] on the device."""
    _dev(k_raw, "k_raw", torch.float32)
    _all_dev(k_raw.device, v_raw=(v_raw, torch.float32), src_row0=(src_row0, torch.int64),
             dst_record=(dst_record, torch.int64), tiles=(tiles, torch.uint8))
    if k_raw.shape != v_raw.shape:
        raise ValueError("k_raw and v_raw must have the same shape")
    if src_row0.numel() != dst_record.numel():
        raise ValueError("src_row0 and dst_record must have one entry per unit")
    row_stride = k_raw.shape[-1]
    n_rows = k_raw.numel() // row_stride
    _check("kvarn_compress_tile",
           _L().kvarn_compress_tile(_ptr(k_raw), _ptr(v_raw), row_stride, n_rows, _ptr(src_row0),
                                    _ptr(tiles), tiles.numel(), _ptr(dst_record), src_row0.numel(),
                                    ctypes.byref(lay), _stream(stream)))


def append_window(k_new, v_new, win_k, win_v, win_start, win_len, stream=None, flags=0):
    """k_new, v_new: fp32 [n_seq][n_new][Hkv][D]; win_k, win_v: fp32
    [n_seq][Hkv][cap][D]; win_start, win_len: int32 [n_seq]."""
    _dev(k_new, "k_new", torch.float32)
    _all_dev(k_new.device, v_new=(v_new, torch.float32), win_k=(win_k, torch.float32),
             win_v=(win_v, torch.float32), win_start=(win_start, torch.int32),
             win_len=(win_len, torch.int32))
    n_seq, n_new, hkv, D = k_new.shape
    if v_new.shape != k_new.shape or win_k.shape != win_v.shape or win_k.shape[:2] != (n_seq, hkv) \
            or win_k.shape[3] != D or win_start.numel() != n_seq or win_len.numel() != n_seq:
        raise ValueError("append_window: inconsistent shapes")
    cap = win_k.shape[2]
    _check("kvarn_append_window",
           _L().kvarn_append_window(_ptr(k_new), _ptr(v_new), n_new, _ptr(win_k), _ptr(win_v), cap,
                                    _ptr(win_start), _ptr(win_len), n_seq, hkv, D, int(flags),
                                    _stream(stream)))


def decode_workspace_bytes(B, Hq, Hkv, head_dim, max_tiles, win_capacity) -> int:
    n = ctypes.c_size_t()
    _check("kvarn_decode_workspace_bytes",
           _L().kvarn_decode_workspace_bytes(B, Hq, Hkv, head_dim, max_tiles, win_capacity,
                                             ctypes.byref(n)))
    return n.value


def _decode_inputs(q, tiles, tile_table, n_tiles, win_k, win_v, win_start, win_len, what):
    """Checks the decode inputs (q fp32 [B][Hq][D]; tile_table int64
    [B][Hkv][max_tiles]; n_tiles int32 [B]; win_k/v fp32 [B][Hkv][cap][D];
    win_start/len int32 [B]) and returns (B, Hq, D, Hkv, max_tiles, cap)."""
    _dev(q, "q", torch.float32)
    _all_dev(q.device, tiles=(tiles, torch.uint8), tile_table=(tile_table, torch.int64),
             n_tiles=(n_tiles, torch.int32), win_k=(win_k, torch.float32),
             win_v=(win_v, torch.float32), win_start=(win_start, torch.int32),
             win_len=(win_len, torch.int32))
    B, Hq, D = q.shape
    Hkv, max_tiles = tile_table.shape[1], tile_table.shape[2]
    cap = win_k.shape[2]
    if (tile_table.shape[0] != B or n_tiles.numel() != B or win_start.numel() != B
            or win_len.numel() != B or win_k.shape != win_v.shape
            or tuple(win_k.shape[:2]) != (B, Hkv) or win_k.shape[3] != D):
        raise ValueError(f"{what}: inconsistent shapes")
    return B, Hq, D, Hkv, max_tiles, cap


def decode_attention(q, tiles, tile_table, n_tiles, win_k, win_v, win_start, win_len,
                     lay: Layout, softmax_scale=None, ws=None, out=None, stream=None, flags=0):
    """q fp32 [B][Hq][D]; tiles uint8 record pool; tile_table int64
    [B][Hkv][max_tiles]; n_tiles int32 [B]; win_k/v fp32 [B][Hkv][cap][D];
    win_start/len int32 [B]; flags: LAUNCH_* bits of this call."""
    B, Hq, D, Hkv, max_tiles, cap = _decode_inputs(q, tiles, tile_table, n_tiles, win_k, win_v,
                                                   win_start, win_len, "decode_attention")
    if softmax_scale is None:
        softmax_scale = D ** -0.5
    need = decode_workspace_bytes(B, Hq, Hkv, D, max_tiles, cap)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    _all_dev(q.device, ws=(ws, torch.uint8), out=(out, torch.float32))
    _check("kvarn_decode_attention",
           _L().kvarn_decode_attention(_ptr(q), _ptr(tiles), tiles.numel(), _ptr(tile_table),
                                       _ptr(n_tiles), _ptr(win_k), _ptr(win_v), _ptr(win_start),
                                       _ptr(win_len), cap, B, Hq, Hkv, D, max_tiles,
                                       float(softmax_scale), ctypes.byref(lay), _ptr(ws),
                                       ws.numel(), _ptr(out), int(flags), _stream(stream)))
    return out


def decode_split(q, tiles, tile_table, n_tiles, win_k, win_v, win_start, win_len, lay: Layout,
                 ws, softmax_scale=None, stream=None, flags=0):
    """First decode kernel: per-item partials into ws (see decode_attention)."""
    B, Hq, D, Hkv, max_tiles, cap = _decode_inputs(q, tiles, tile_table, n_tiles, win_k, win_v,
                                                   win_start, win_len, "decode_split")
    _dev(ws, "ws", torch.uint8, q.device)
    if softmax_scale is None:
        softmax_scale = D ** -0.5
    _check("kvarn_decode_split",
           _L().kvarn_decode_split(_ptr(q), _ptr(tiles), tiles.numel(), _ptr(tile_table),
                                   _ptr(n_tiles), _ptr(win_k), _ptr(win_v), _ptr(win_start),
                                   _ptr(win_len), cap, B, Hq, Hkv, D, max_tiles,
                                   float(softmax_scale), ctypes.byref(lay), _ptr(ws), ws.numel(),
                                   int(flags), _stream(stream)))


def decode_combine(ws, out, Hkv, max_tiles, win_capacity, stream=None, flags=0):
    """Second decode kernel: LSE combine of the partials in ws into out [B][Hq][D]."""
    _dev(out, "out", torch.float32)
    _dev(ws, "ws", torch.uint8, out.device)
    B, Hq, D = out.shape
    _check("kvarn_decode_combine",
           _L().kvarn_decode_combine(_ptr(ws), ws.numel(), B, Hq, Hkv, D, max_tiles, win_capacity,
                                     _ptr(out), int(flags), _stream(stream)))
    return out


def window_advance(win_start, win_len, n_tiles, d_len, promote, win_capacity, stream=None, flags=0):
    """Device-side window bookkeeping (length += d_len, then promote tiles)."""
    _dev(win_start, "win_start", torch.int32)
    _dev(win_len, "win_len", torch.int32, win_start.device)
    if n_tiles is not None:
        _dev(n_tiles, "n_tiles", torch.int32, win_start.device)
    _check("kvarn_window_advance",
           _L().kvarn_window_advance(_ptr(win_start), _ptr(win_len), _ptr(n_tiles),
                                     win_start.numel(), int(d_len), int(promote),
                                     int(win_capacity), int(flags), _stream(stream)))


def prefill_workspace_bytes(n_tiles, win_len, Hkv, head_dim) -> int:
    n = ctypes.c_size_t()
    _check("kvarn_prefill_workspace_bytes",
           _L().kvarn_prefill_workspace_bytes(int(n_tiles), int(win_len), Hkv, head_dim,
                                              ctypes.byref(n)))
    return n.value


def prefill_attention(q_chunk, pos0, tiles, tile_table, n_tiles, win_k, win_v, win_start,
                      win_len, lay: Layout, softmax_scale=None, ws=None, out=None, stream=None,
                      ws_blocks=None, cached_tiles=0):
    """Causal attention of a chunk of one sequence: q_chunk fp32 [C][Hq][D] at
    positions pos0 + i; tile_table int64 [Hkv][stride]; win_k/v fp32
    [Hkv][cap][D]; n_tiles, win_start, win_len host ints; ws a uint8 device
    workspace of prefill_workspace_bytes() (allocated here when None). With
    ws_blocks (images per KV head of a ws kept for the whole prompt), the call
    goes through kvarn_prefill_attention_cached and converts only the tiles
    from cached_tiles on."""
    _dev(q_chunk, "q_chunk", torch.float32)
    _all_dev(q_chunk.device, tiles=(tiles, torch.uint8), tile_table=(tile_table, torch.int64),
             win_k=(win_k, torch.float32), win_v=(win_v, torch.float32))
    C, Hq, D = q_chunk.shape
    Hkv, stride = tile_table.shape
    cap = win_k.shape[1]
    if win_k.shape != win_v.shape or win_k.shape[0] != Hkv or win_k.shape[2] != D:
        raise ValueError("prefill_attention: inconsistent shapes")
    if softmax_scale is None:
        softmax_scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q_chunk)
    if ws is None:
        need = prefill_workspace_bytes(n_tiles, win_len, Hkv, D)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=q_chunk.device)
    _all_dev(q_chunk.device, ws=(ws, torch.uint8), out=(out, torch.float32))
    if ws_blocks is not None:
        _check("kvarn_prefill_attention_cached",
               _L().kvarn_prefill_attention_cached(
                   _ptr(q_chunk), C, int(pos0), _ptr(tiles), tiles.numel(), _ptr(tile_table),
                   stride, int(n_tiles), _ptr(win_k), _ptr(win_v), int(win_start), int(win_len),
                   cap, Hq, Hkv, D, float(softmax_scale), ctypes.byref(lay), _ptr(ws),
                   ws.numel(), int(ws_blocks), int(cached_tiles), _ptr(out), _stream(stream)))
        return out
    _check("kvarn_prefill_attention",
           _L().kvarn_prefill_attention(_ptr(q_chunk), C, int(pos0), _ptr(tiles), tiles.numel(),
                                        _ptr(tile_table), stride, int(n_tiles), _ptr(win_k),
                                        _ptr(win_v), int(win_start), int(win_len), cap, Hq, Hkv, D,
                                        float(softmax_scale), ctypes.byref(lay), _ptr(ws),
                                        ws.numel(), _ptr(out), _stream(stream)))
    return out


def decode_attention_noalloc(q, tiles, tile_table, n_tiles, win_k, win_v, win_start, win_len,
                             lay: Layout, softmax_scale=None, out=None, stream=None, flags=0):
    """decode_attention for callers that cannot allocate device memory: the
    partials go to the library's own fixed scratch array instead of a
    workspace (see kvarn_decode_attention_noalloc in include/kvarn.h).
    `out` must be passed by such callers; it is created here only as a
    convenience for everyone else."""
    B, Hq, D, Hkv, max_tiles, cap = _decode_inputs(q, tiles, tile_table, n_tiles, win_k, win_v,
                                                   win_start, win_len, "decode_attention_noalloc")
    if softmax_scale is None:
        softmax_scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", torch.float32, q.device)
    _check("kvarn_decode_attention_noalloc",
           _L().kvarn_decode_attention_noalloc(
               _ptr(q), _ptr(tiles), tiles.numel(), _ptr(tile_table), _ptr(n_tiles), _ptr(win_k),
               _ptr(win_v), _ptr(win_start), _ptr(win_len), cap, B, Hq, Hkv, D, max_tiles,
               float(softmax_scale), ctypes.byref(lay), _ptr(out), int(flags), _stream(stream)))
    return out
