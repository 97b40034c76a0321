"""CPU-side checks of the C ABI: the library loads, exports every function
include/kvarn.h declares, and rejects bad arguments on the host before any
launch (no GPU needed: validation precedes every CUDA call)."""
import ctypes
import os

import pytest

import oracle
from kv_cache_quantization_token_gb300 import _build, kvarn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvarn.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kvarn._L()


def test_library_exports_every_declared_function(lib):
    names = kvarn.declared_functions(HEADER)
    assert {"kvarn_layout", "kvarn_compress_tile", "kvarn_decode_attention",
            "kvarn_rotate_query", "kvarn_append_window"} <= set(names)
    raw = ctypes.CDLL(_build.LIB)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in kvarn.h but not exported"


@pytest.mark.parametrize("D", [64, 128, 256])
def test_layout_agrees_with_oracle_record_size(lib, D):
    L = kvarn.layout(D)
    assert L.record_bytes == oracle.record_bytes(D)
    assert L.version == 1 and L.tile_tokens == 128 and L.sinkhorn_iters == 4
    assert (L.k_bits, L.v_bits, L.v_group) == (4, 2, min(D, 128))
    offs = [L.off_k_codes, L.off_v_codes, L.off_k_delta, L.off_k_lo, L.off_k_s, L.off_k_r,
            L.off_v_delta, L.off_v_lo, L.off_v_r, L.off_v_s]
    assert offs == sorted(offs) and all(o % 16 == 0 for o in offs)
    assert L.off_v_codes == 64 * D and L.off_k_delta == 96 * D


def test_layout_rejects_unsupported(lib):
    L = kvarn.Layout()
    for D, it in ((96, 4), (32, 4), (512, 4), (128, 0), (128, 17)):
        assert lib.kvarn_layout(D, it, ctypes.byref(L)) == -3
    assert lib.kvarn_layout(128, 4, None) == -1


def test_status_strings(lib):
    for s in range(-7, 1):
        assert lib.kvarn_status_string(s)


def test_host_validation_rejects_before_launch(lib):
    L = kvarn.layout(128)
    p = ctypes.c_void_p(16)
    bad = ctypes.c_void_p(8)
    # compress: null, misaligned, bad stride, a pool smaller than one record
    rb = L.record_bytes
    assert lib.kvarn_compress_tile(None, p, 128, 256, p, p, rb, p, 1, ctypes.byref(L), None) == -1
    assert lib.kvarn_compress_tile(bad, p, 128, 256, p, p, rb, p, 1, ctypes.byref(L), None) == -2
    assert lib.kvarn_compress_tile(p, p, 130, 256, p, p, rb, p, 1, ctypes.byref(L), None) == -2
    assert lib.kvarn_compress_tile(p, p, 64, 256, p, p, rb, p, 1, ctypes.byref(L), None) == -4
    assert lib.kvarn_compress_tile(p, p, 128, 256, p, p, rb - 16, p, 1, ctypes.byref(L), None) == -4
    assert lib.kvarn_compress_tile(p, p, 128, 256, p, p, -1, p, 1, ctypes.byref(L), None) == -4
    assert lib.kvarn_compress_tile(p, p, 128, 256, p, p, rb, p, 0, ctypes.byref(L), None) == 0
    tampered = kvarn.layout(128)
    tampered.record_bytes += 16
    assert lib.kvarn_compress_tile(p, p, 128, 256, p, p, rb, p, 1, ctypes.byref(tampered), None) == -3
    # rotate: unsupported dim, overlap
    assert lib.kvarn_rotate_query(p, p, 4, 96, None) == -3
    assert lib.kvarn_rotate_query(ctypes.c_void_p(4096), ctypes.c_void_p(4096 + 256), 4, 128, None) == -4
    # append: too many new tokens for the ring; unknown launch flags
    assert lib.kvarn_append_window(p, p, 300, p, p, 256, p, p, 1, 8, 128, 0, None) == -4
    assert lib.kvarn_append_window(p, p, 3, p, p, 256, p, p, 1, 8, 128, 8, None) == -4
    # decode: GQA group too large, non-divisible heads, workspace too small
    n = ctypes.c_size_t()
    assert lib.kvarn_decode_workspace_bytes(1, 32, 2, 128, 8, 128, ctypes.byref(n)) == -3
    assert lib.kvarn_decode_workspace_bytes(1, 30, 8, 128, 8, 128, ctypes.byref(n)) == -4
    assert lib.kvarn_decode_workspace_bytes(1, 32, 8, 128, 8, 128, ctypes.byref(n)) == 0
    assert n.value > 0
    def dargs(ws_bytes=16, flags=0, tiles_bytes=1 << 30):
        return ([p, p, tiles_bytes] + [p] * 6 + [128, 1, 32, 8, 128, 8, ctypes.c_float(0.088),
                                                 ctypes.byref(L), p, ws_bytes, p, flags, None])
    assert lib.kvarn_decode_attention(*dargs()) == -5
    assert lib.kvarn_decode_attention(*dargs(1 << 30, flags=4)) == -4   # unknown flag bit
    assert lib.kvarn_decode_attention(*dargs(1 << 30, tiles_bytes=-1)) == -4
    assert lib.kvarn_decode_attention_noalloc(*(dargs(flags=2)[:17] + [p, 2, None])) == -4


def test_prefill_host_validation(lib):
    L = kvarn.layout(128)
    p = ctypes.c_void_p(4096)
    args = lambda C, pos0, nt, wl, D=128, Hq=32, lay=L, wsb=1 << 40: (
        p, C, pos0, p, ctypes.c_int64(1 << 40), p, 64, nt, p, p, 0, wl, 768, Hq, 8, D,
        ctypes.c_float(0.088), ctypes.byref(lay), p, ctypes.c_size_t(wsb), p, None)
    f = lib.kvarn_prefill_attention
    f.argtypes = None
    assert f(*args(512, 2000, 10, 300)) == -4          # chunk beyond the cache
    L256 = kvarn.layout(256)
    assert f(*args(16, 0, 1, 16, D=256, lay=L)) == -3     # layout of another head_dim
    assert f(*args(16, 0, 1, 16, D=96, lay=L256)) == -3   # head_dim 96
    assert f(*args(0, 0, 1, 16, D=256, lay=L256)) == 0    # head_dim 256: empty chunk
    assert f(*args(16, 0, 1, 16, Hq=80)) == -3            # GQA group of 10
    assert f(*args(0, 0, 0, 0)) == 0                      # empty chunk enqueues nothing
    # the workspace bound covers every tile and window block of 8 KV heads ...
    need = ctypes.c_size_t()
    assert lib.kvarn_prefill_workspace_bytes(10, 300, 8, 128, ctypes.byref(need)) == 0
    blk = 4 * 128 * 128 * 2
    assert need.value == (10 + 3) * 8 * blk
    assert lib.kvarn_prefill_workspace_bytes(10, 300, 4, 256, ctypes.byref(need)) == 0
    assert need.value == (10 + 3) * 4 * 4 * 128 * 256 * 2
    # ... a chunk at 1000..1511 sees the 10 tiles and 2 of the window's 3 blocks
    assert f(*args(512, 1000, 10, 300, wsb=12 * 8 * blk - 1)) == -5



def test_launch_flags_are_per_call(lib):
    """Launch flags are an argument of each decode-path call: unknown bits and
    PREFETCH without PDL are refused by that call, and nothing is left set
    between calls."""
    p = ctypes.c_void_p(4096)
    adv = lib.kvarn_window_advance
    assert adv(p, p, p, 1, 1, 0, 128, kvarn.LAUNCH_PREFETCH, None) == -4
    assert adv(p, p, p, 1, 1, 0, 128, 8, None) == -4
    assert adv(p, p, p, 0, 1, 0, 128, kvarn.LAUNCH_PDL | kvarn.LAUNCH_PREFETCH, None) == 0
    assert lib.kvarn_decode_combine(p, 1 << 30, 1, 32, 8, 128, 8, 128, p, 16, None) == -4
    assert not hasattr(kvarn, "set_launch_flags")
    raw = ctypes.CDLL(_build.LIB)
    assert not hasattr(raw, "kvarn_set_launch_flags")


def test_device_error_api_rejects_bad_arguments(lib):
    assert lib.kvarn_get_device_error(None, 0) == -1
    assert lib.kvarn_selftest_bounded_wait(0, None) == -4
    assert lib.kvarn_selftest_bounded_wait(2000000, None) == -4


@pytest.mark.parametrize("D", [64, 128, 256])
def test_f16_scale_layout_agrees_with_oracle(lib, D):
    L = kvarn.layout(D, scale_bits=16)
    assert L.version == 2 and L.record_bytes == oracle.record_bytes(D, 16)
    assert L.record_bytes % 128 == 0 and L.off_k_delta == 96 * D
    assert L.off_k_lo - L.off_k_delta == 2 * D and L.off_v_s + 2 * D == L.record_bytes
    assert (L.k_bits, L.v_bits) == (4, 2)
    M = kvarn.Layout()
    assert lib.kvarn_layout_scales(D, 4, 8, ctypes.byref(M)) == -3
    assert lib.kvarn_layout_scales(D, 4, 32, ctypes.byref(M)) == 0 and M.version == 1
    # a layout claiming f16 scales with fp32 offsets is not one the library made
    M.version = 2
    p = ctypes.c_void_p(16)
    assert lib.kvarn_compress_tile(p, p, D, 256, p, p, 1 << 20, p, 1, ctypes.byref(M), None) == -3


def test_prefill_cached_host_validation(lib):
    L = kvarn.layout(128)
    p = ctypes.c_void_p(4096)
    blk = 4 * 128 * 128 * 2
    f = lib.kvarn_prefill_attention_cached
    f.argtypes = None
    args = lambda wsb, wsblocks, cached, nt=10: (
        p, 512, 1000, p, ctypes.c_int64(1 << 40), p, 64, nt, p, p, 0, 300, 768, 32, 8, 128,
        ctypes.c_float(0.088), ctypes.byref(L), p, ctypes.c_size_t(wsb), wsblocks, cached, p, None)
    assert f(*args(1 << 40, 0, 0)) == -4           # ws_blocks must be positive
    assert f(*args(1 << 40, 11, 0)) == -5          # fewer images per head than the 12 blocks seen
    assert f(*args(16 * 8 * blk - 1, 16, 0)) == -5  # workspace smaller than ws_blocks images
    assert f(*args(1 << 40, 16, 11)) == -4         # more cached tiles than tiles
    assert f(*args(1 << 40, 16, -1)) == -4


@pytest.mark.parametrize("D", [64, 128, 256])
def test_v4_layout_agrees_with_oracle(lib, D):
    for sb in (32, 16):
        L = kvarn.layout(D, scale_bits=sb, v_bits=4)
        assert L.v_bits == 4 and L.record_bytes == oracle.record_bytes(D, sb, 4)
        assert L.off_k_delta == 128 * D and L.record_bytes % 128 == 0
    M = kvarn.Layout()
    assert lib.kvarn_layout_ex(D, 4, 32, 1, ctypes.byref(M)) == -3
    assert lib.kvarn_layout_ex(D, 4, 32, 8, ctypes.byref(M)) == -3


@pytest.mark.parametrize("D", [64, 128, 256])
def test_v3_layout_agrees_with_oracle(lib, D):
    """k4v3: token rows of 3 D / 8 bytes (a bit stream); the library's layout
    and the oracle's record size agree."""
    for sb in (32, 16):
        L = kvarn.layout(D, scale_bits=sb, v_bits=3)
        assert L.v_bits == 3 and L.record_bytes == oracle.record_bytes(D, sb, 3)
        assert L.off_k_delta == 112 * D and L.record_bytes % 128 == 0


def test_prefill_accepts_v4_records(lib):
    """k4v4 records pass the prefill entry's layout check: an empty chunk is a
    no-op and a bad head ratio is reported as such, not as an unsupported
    record format."""
    L = kvarn.layout(128, v_bits=4)
    p = ctypes.c_void_p(4096)
    f = lib.kvarn_prefill_attention
    f.argtypes = None
    big = ctypes.c_int64(1 << 40)
    assert f(p, 0, 0, p, big, p, 64, 1, p, p, 0, 16, 768, 32, 8, 128, ctypes.c_float(0.088),
             ctypes.byref(L), p, ctypes.c_size_t(1 << 40), p, None) == 0
    assert f(p, 16, 0, p, big, p, 64, 1, p, p, 0, 16, 768, 33, 8, 128, ctypes.c_float(0.088),
             ctypes.byref(L), p, ctypes.c_size_t(1 << 40), p, None) == -4
