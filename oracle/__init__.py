"""fp64 CPU oracle of the KVarN hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its binding) never calls it and shares no code with it.

The arithmetic lives in ``kvarn_oracle.c`` (plain C, fp64); this module only
marshals numpy arrays and keeps the bookkeeping of the cache state machine,
which holds no arithmetic beyond counting tokens.

Sources, by the pages' titles:
  * SharpInference issue #180 "Implement KVarN variance-normalized KV-cache
    quantization (2-bit values)", section "Algorithm (per 128-token tile)".
  * SharpInference PR #434 "KVarN variance-normalized KV-cache quantization:
    CPU + CUDA (#180)", commits 82efc4f (core quantizer), 6040076 (FP32
    window as staging, whole-tile promotion), 99c3773 (chunked prefill,
    schedule-independent tiles).
  * SharpInference issue #433 "KVarN follow-ups", item 2 (split-tile decode
    with LSE combine and a deferred inverse rotation).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

TILE = 128
K_BITS = 4
V_BITS = 2
DEFAULT_ITERS = 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvarn_oracle.c")
_LIB_PATH = os.path.join(_HERE, f"_build_{platform.machine()}", "liboracle.so")
_lib = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile the C oracle for this machine (gcc, fp64, no FMA contraction so
    that x86 and Arm hosts round alike)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                lib = ctypes.CDLL(build())
                i64, c_int = ctypes.c_int64, ctypes.c_int
                lib.orc_hadamard_entry.restype = ctypes.c_double
                lib.orc_hadamard_entry.argtypes = [c_int, c_int, c_int]
                lib.orc_wht_rows.argtypes = [_dp, _dp, i64, c_int]
                lib.orc_sinkhorn.argtypes = [_dp, c_int, c_int, c_int, _dp, _dp, _dp]
                lib.orc_rtn_group.argtypes = [_dp, c_int, i64, c_int, _dp, _dp, _u8p, _dp]
                lib.orc_quantize_tensor.argtypes = [_fp, i64, c_int, c_int, c_int, c_int,
                                                    _dp, _dp, _dp, _dp, _u8p, _dp]
                lib.orc_record_bytes.restype = i64
                lib.orc_record_bytes.argtypes = [c_int]
                lib.orc_pack_record.argtypes = [c_int, _u8p, _u8p] + [_dp] * 8 + [_u8p]
                lib.orc_unpack_record.argtypes = [c_int, _u8p, _u8p, _u8p] + [_dp] * 8
                lib.orc_compress_unit.argtypes = [_fp, _fp, i64, c_int, c_int, _u8p] + [_dp] * 10
                lib.orc_dequant_record.argtypes = [c_int, _u8p, _dp, _dp]
                lib.orc_record_bytes_fmt.restype = i64
                lib.orc_record_bytes_fmt.argtypes = [c_int, c_int, c_int]
                lib.orc_pack_record_fmt.argtypes = [c_int, c_int, c_int, _u8p, _u8p] + [_dp] * 8 + [_u8p]
                lib.orc_unpack_record_fmt.argtypes = [c_int, c_int, c_int, _u8p, _u8p, _u8p] + [_dp] * 8
                lib.orc_compress_unit_fmt.argtypes = ([_fp, _fp, i64, c_int, c_int, c_int, c_int, _u8p]
                                                      + [_dp] * 10)
                lib.orc_dequant_record_fmt.argtypes = [c_int, c_int, c_int, _u8p, _dp, _dp]
                lib.orc_f64_to_f16_bits.restype = ctypes.c_uint16
                lib.orc_f64_to_f16_bits.argtypes = [ctypes.c_double]
                lib.orc_f16_bits_to_f64.restype = ctypes.c_double
                lib.orc_f16_bits_to_f64.argtypes = [ctypes.c_uint16]
                lib.orc_attend.argtypes = [_dp, _dp, _dp, i64, c_int, ctypes.c_double, _dp]
                _lib = lib
    return _lib


def _ptr(a: np.ndarray, kind):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(kind)


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


# --------------------------------------------------------------------------
# c1 -- Walsh-Hadamard rotation
def hadamard_entry(i: int, j: int, D: int) -> float:
    return _L().orc_hadamard_entry(i, j, D)


def wht_rows(x: np.ndarray) -> np.ndarray:
    """H x for every row of x (last axis D): H the Sylvester matrix / sqrt(D)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    D = x.shape[-1]
    y = np.empty_like(x)
    _check(_L().orc_wht_rows(_ptr(x, _dp), _ptr(y, _dp), x.size // D, D), "wht")
    return y


# --------------------------------------------------------------------------
# c2 -- Sinkhorn normalisation
def sinkhorn(Y: np.ndarray, iters: int = DEFAULT_ITERS):
    """Returns (s[D], r[T], Yn[T][D]) for one rotated tensor Y[T][D]."""
    Y = np.ascontiguousarray(Y, dtype=np.float64)
    T, D = Y.shape
    s, r, yn = np.empty(D), np.empty(T), np.empty_like(Y)
    _check(_L().orc_sinkhorn(_ptr(Y, _dp), T, D, iters, _ptr(s, _dp), _ptr(r, _dp),
                             _ptr(yn, _dp)), "sinkhorn")
    return s, r, yn


# --------------------------------------------------------------------------
# c3 -- round to nearest
def rtn_group(y: np.ndarray, bits: int):
    """Returns (delta, lo, codes u8, vpre) for one group of values."""
    y = np.ascontiguousarray(y, dtype=np.float64).ravel()
    codes = np.empty(y.size, np.uint8)
    vpre = np.empty(y.size)
    d, lo = ctypes.c_double(), ctypes.c_double()
    _check(_L().orc_rtn_group(_ptr(y, _dp), y.size, 1, bits, ctypes.byref(d), ctypes.byref(lo),
                              _ptr(codes, _u8p), _ptr(vpre, _dp)), "rtn")
    return d.value, lo.value, codes, vpre


def quantize_tensor(x: np.ndarray, per_channel: bool, bits: int, iters: int = DEFAULT_ITERS):
    """Rotate, normalise and quantise one [128][D] fp32 tensor of a tile."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    T, D = x.shape
    assert T == TILE
    gv = D // min(D, 128)
    s, r = np.empty(D), np.empty(T)
    n_groups = D if per_channel else T * gv
    delta, lo = np.empty(n_groups), np.empty(n_groups)
    codes = np.empty((T, D), np.uint8)
    vpre = np.empty((T, D))
    _check(_L().orc_quantize_tensor(_ptr(x, _fp), D, D, iters, int(per_channel), bits,
                                    _ptr(s, _dp), _ptr(r, _dp), _ptr(delta, _dp), _ptr(lo, _dp),
                                    _ptr(codes, _u8p), _ptr(vpre, _dp)), "quantize")
    return dict(s=s, r=r, delta=delta, lo=lo, codes=codes, vpre=vpre)


# --------------------------------------------------------------------------
# c4 -- packed record. scale_bits = 32: the default layout (fp32 scales);
# 16: the f16-scale layout (SharpInference issue #433, item 3), same codes.
# v_bits = 2: the method's k4v2 preset; 3 and 4: k4v3 and k4v4 variants (other
# K/V bit widths, gmlx PR #116), the same packing rule: each token's V codes
# are a little-endian bit stream, channel c at bits v_bits*c .. (a 3-bit code
# can straddle two bytes).
def _sw(scale_bits: int) -> int:
    if scale_bits not in (16, 32):
        raise ValueError(f"scale_bits must be 16 or 32, not {scale_bits}")
    return scale_bits // 8


def f16_bits(v: float) -> int:
    """IEEE binary16 bits of v, rounded to nearest with ties to even."""
    return int(_L().orc_f64_to_f16_bits(float(v)))


def f16_value(bits: int) -> float:
    return float(_L().orc_f16_bits_to_f64(int(bits)))


def _vb(v_bits: int) -> int:
    if v_bits not in (2, 3, 4):
        raise ValueError(f"v_bits must be 2, 3 or 4, not {v_bits}")
    return v_bits


def record_bytes(D: int, scale_bits: int = 32, v_bits: int = 2) -> int:
    n = _L().orc_record_bytes_fmt(D, _sw(scale_bits), _vb(v_bits))
    if n < 0:
        raise ValueError(f"unsupported head_dim {D}")
    return int(n)


def pack_record(D, k_codes, v_codes, k_delta, k_lo, k_s, k_r, v_delta, v_lo, v_r, v_s,
                scale_bits: int = 32, v_bits: int = 2):
    rec = np.empty(record_bytes(D, scale_bits, v_bits), np.uint8)
    args = [np.ascontiguousarray(a, dtype=np.float64) for a in
            (k_delta, k_lo, k_s, k_r, v_delta, v_lo, v_r, v_s)]
    kc = np.ascontiguousarray(k_codes, dtype=np.uint8)
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
    _check(_L().orc_pack_record_fmt(D, _sw(scale_bits), _vb(v_bits), _ptr(kc, _u8p),
                                    _ptr(vc, _u8p), *[_ptr(a, _dp) for a in args],
                                    _ptr(rec, _u8p)), "pack")
    return rec


def unpack_record(rec: np.ndarray, D: int, scale_bits: int = 32, v_bits: int = 2) -> dict:
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    gv = D // min(D, 128)
    out = dict(k_codes=np.empty((TILE, D), np.uint8), v_codes=np.empty((TILE, D), np.uint8),
               k_delta=np.empty(D), k_lo=np.empty(D), k_s=np.empty(D), k_r=np.empty(TILE),
               v_delta=np.empty(TILE * gv), v_lo=np.empty(TILE * gv), v_r=np.empty(TILE),
               v_s=np.empty(D))
    names = ("k_delta", "k_lo", "k_s", "k_r", "v_delta", "v_lo", "v_r", "v_s")
    _check(_L().orc_unpack_record_fmt(D, _sw(scale_bits), _vb(v_bits), _ptr(rec, _u8p),
                                      _ptr(out["k_codes"], _u8p), _ptr(out["v_codes"], _u8p),
                                      *[_ptr(out[n], _dp) for n in names]), "unpack")
    return out


def compress_unit(k: np.ndarray, v: np.ndarray, iters: int = DEFAULT_ITERS,
                  scale_bits: int = 32, v_bits: int = 2) -> dict:
    """Compress one (tile, KV head): k, v fp32 [128][D]. Returns the record
    bytes plus fp64 scales and pre-rounding values for the parity checks."""
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    T, D = k.shape
    assert T == TILE and v.shape == k.shape
    gv = D // min(D, 128)
    o = dict(record=np.empty(record_bytes(D, scale_bits, v_bits), np.uint8),
             k_s=np.empty(D), k_r=np.empty(T), k_delta=np.empty(D), k_lo=np.empty(D),
             k_vpre=np.empty((T, D)), v_s=np.empty(D), v_r=np.empty(T),
             v_delta=np.empty(T * gv), v_lo=np.empty(T * gv), v_vpre=np.empty((T, D)))
    names = ("k_s", "k_r", "k_delta", "k_lo", "k_vpre", "v_s", "v_r", "v_delta", "v_lo", "v_vpre")
    _check(_L().orc_compress_unit_fmt(_ptr(k, _fp), _ptr(v, _fp), D, D, iters, _sw(scale_bits),
                                      _vb(v_bits), _ptr(o["record"], _u8p),
                                      *[_ptr(o[n], _dp) for n in names]), "compress")
    return o


# --------------------------------------------------------------------------
# c5 -- reconstruction
def dequant_record(rec: np.ndarray, D: int, scale_bits: int = 32, v_bits: int = 2):
    """Unrotated fp64 K and V rows ([128][D] each) of one record."""
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    k, v = np.empty((TILE, D)), np.empty((TILE, D))
    _check(_L().orc_dequant_record_fmt(D, _sw(scale_bits), _vb(v_bits), _ptr(rec, _u8p),
                                       _ptr(k, _dp), _ptr(v, _dp)), "dequant")
    return k, v


# --------------------------------------------------------------------------
# c7 / c8 -- exact attention
def attend(q: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float64)
    keys = np.ascontiguousarray(keys, dtype=np.float64)
    values = np.ascontiguousarray(values, dtype=np.float64)
    D = q.shape[-1]
    n = keys.shape[0] if keys.size else 0
    out = np.empty(D)
    kp = keys if n else np.zeros((1, D))
    vp = values if n else np.zeros((1, D))
    _check(_L().orc_attend(_ptr(q, _dp), _ptr(kp, _dp), _ptr(vp, _dp), n, D, float(scale),
                           _ptr(out, _dp)), "attend")
    return out


def window_rows(win: np.ndarray, start: int, length: int) -> np.ndarray:
    """The `length` oldest-first rows of a ring window win[Wcap][D]."""
    cap = win.shape[0]
    idx = (start + np.arange(length)) % cap
    return np.asarray(win[idx], dtype=np.float64)


def kv_head_tokens(pool: np.ndarray, table_row, n_tiles: int, win_k, win_v, start, length, D,
                   scale_bits: int = 32, v_bits: int = 2):
    """All cached (k, v) rows of one KV head, in position order: the tiles'
    reconstructed rows, then the window's raw rows."""
    ks, vs = [], []
    rb = record_bytes(D, scale_bits, v_bits)
    for i in range(n_tiles):
        off = int(table_row[i])
        k, v = dequant_record(pool[off:off + rb], D, scale_bits, v_bits)
        ks.append(k)
        vs.append(v)
    ks.append(window_rows(win_k, start, length))
    vs.append(window_rows(win_v, start, length))
    return np.concatenate(ks, 0), np.concatenate(vs, 0)


def decode_attention(q, pool, tile_table, n_tiles, win_k, win_v, win_start, win_len, scale,
                     heads=None, scale_bits: int = 32, v_bits: int = 2):
    """Exact decode attention (c7) for every (b, h) in `heads` (default: all).
    q [B][Hq][D]; tile_table [B][Hkv][max_tiles]; win_k/v [B][Hkv][Wcap][D].
    Returns {(b, h): out[D]} in fp64."""
    B, Hq, D = q.shape
    Hkv = tile_table.shape[1]
    G = Hq // Hkv
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(Hq)]
    cache = {}
    res = {}
    for b, h in heads:
        kvh = h // G
        if (b, kvh) not in cache:
            cache[(b, kvh)] = kv_head_tokens(pool, tile_table[b, kvh], int(n_tiles[b]),
                                             win_k[b, kvh], win_v[b, kvh], int(win_start[b]),
                                             int(win_len[b]), D, scale_bits, v_bits)
        keys, values = cache[(b, kvh)]
        res[(b, h)] = attend(q[b, h], keys, values, scale)
    return res


def prefill_attention(q_chunk, pos0, pool, table, n_tiles, win_k, win_v, win_start, win_len,
                      scale, rows=None, scale_bits: int = 32, v_bits: int = 2):
    """Exact causal attention (c8) of a chunk of queries of ONE sequence.
    q_chunk [C][Hq][D] at positions pos0 + i; tokens of tile k sit at positions
    [128k, 128k+128), window token j at 128*n_tiles + j; query i sees positions
    <= pos0 + i. table [Hkv][max_tiles]; win_k/v [Hkv][Wcap][D].
    rows: iterable of (i, h); default all. Returns {(i, h): out[D]}."""
    C, Hq, D = q_chunk.shape
    Hkv = table.shape[0]
    G = Hq // Hkv
    if rows is None:
        rows = [(i, h) for i in range(C) for h in range(Hq)]
    cache = {}
    res = {}
    for i, h in rows:
        kvh = h // G
        if kvh not in cache:
            cache[kvh] = kv_head_tokens(pool, table[kvh], int(n_tiles), win_k[kvh], win_v[kvh],
                                        int(win_start), int(win_len), D, scale_bits, v_bits)
        keys, values = cache[kvh]
        visible = pos0 + i + 1
        res[(i, h)] = attend(q_chunk[i, h], keys[:visible], values[:visible], scale)
    return res


# --------------------------------------------------------------------------
# c6 -- cache state machine (bookkeeping only)
class CacheStateMachine:
    """FP32 staging window plus promoted tiles of one sequence, all KV heads.

    Reading of PR #434 commit 6040076 ("the FP32 window is the staging; whole-
    tile promotion"): after each append, while the window holds at least W
    tokens, its oldest 128 tokens are compressed into the next tile. Step
    order: append, then promote, then attend.
    """

    def __init__(self, n_kv_heads: int, head_dim: int, W: int = 128, iters: int = DEFAULT_ITERS):
        assert W % TILE == 0 and W >= TILE
        self.Hkv, self.D, self.W, self.iters = n_kv_heads, head_dim, W, iters
        self.k_hist = np.zeros((n_kv_heads, 0, head_dim), np.float32)
        self.v_hist = np.zeros((n_kv_heads, 0, head_dim), np.float32)
        self.n_tiles = 0
        self.records = []  # [tile][kv head] -> record bytes

    @property
    def n_tokens(self) -> int:
        return self.k_hist.shape[1]

    @property
    def win_len(self) -> int:
        return self.n_tokens - TILE * self.n_tiles

    def append(self, k_new: np.ndarray, v_new: np.ndarray):
        """k_new, v_new: [n_new][Hkv][D]. Appends, then promotes."""
        k_new = np.asarray(k_new, np.float32).transpose(1, 0, 2)
        v_new = np.asarray(v_new, np.float32).transpose(1, 0, 2)
        self.k_hist = np.concatenate([self.k_hist, k_new], 1)
        self.v_hist = np.concatenate([self.v_hist, v_new], 1)
        promoted = []
        while self.win_len >= self.W:
            t0 = TILE * self.n_tiles
            recs = [compress_unit(self.k_hist[h, t0:t0 + TILE], self.v_hist[h, t0:t0 + TILE],
                                  self.iters)["record"] for h in range(self.Hkv)]
            self.records.append(recs)
            self.n_tiles += 1
            promoted.append(self.n_tiles - 1)
        return promoted

    def window(self, h: int):
        t0 = TILE * self.n_tiles
        return self.k_hist[h, t0:], self.v_hist[h, t0:]
