"""The product path has no CPU or PyTorch fallback: host tensors are refused
before anything is enqueued, and a missing library is an error, not a
silent substitute."""
import os
import subprocess
import sys

import pytest
import torch

from kv_cache_quantization_token_gb300 import kvarn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_host_tensors_are_refused():
    D = 128
    lay = kvarn.layout(D)
    x = torch.zeros(128, D)
    i64 = torch.zeros(1, dtype=torch.int64)
    u8 = torch.zeros(lay.record_bytes, dtype=torch.uint8)
    with pytest.raises(TypeError, match="CUDA tensor"):
        kvarn.compress_tile(x, x, i64, u8, i64, lay)
    with pytest.raises(TypeError, match="CUDA tensor"):
        kvarn.rotate_query(torch.zeros(4, D))
    q = torch.zeros(1, 8, D)
    tab = torch.zeros(1, 2, 1, dtype=torch.int64)
    n = torch.ones(1, dtype=torch.int32)
    win = torch.zeros(1, 2, 128, D)
    with pytest.raises(TypeError, match="CUDA tensor"):
        kvarn.decode_attention(q, u8, tab, n, win, win, n, n, lay)
    with pytest.raises(TypeError, match="CUDA tensor"):
        kvarn.prefill_attention(torch.zeros(4, 8, D), 0, u8, tab[0], 1, win[0], win[0], 0, 4, lay)


class _CudaStandIn(torch.Tensor):
    """A host tensor that reports itself as a CUDA tensor on cuda:0, so the
    binding's checks of the later arguments can be reached on a machine
    without a GPU. It is never handed to the library: each case below puts a
    plain host tensor in one position, which the binding must refuse first."""

    @property
    def is_cuda(self):
        return True

    @property
    def device(self):
        return torch.device("cuda", 0)


def _fake(t):
    return torch.Tensor._make_subclass(_CudaStandIn, t)


def _refuses(fn, args, kwargs, position):
    """fn with a host tensor in `position` (the others stand-ins) raises a
    TypeError naming that argument."""
    with pytest.raises(TypeError, match=f"{position} must be a CUDA tensor"):
        fn(*[a[1] if n == position else a[0] for n, a in args],
           **{k: (v[1] if k == position else v[0]) for k, v in kwargs.items()})


def _pair(t):
    return (_fake(t), t)


@pytest.mark.parametrize("position", ["q", "tiles", "tile_table", "n_tiles", "win_k", "win_v",
                                      "win_start", "win_len"])
def test_decode_refuses_a_host_tensor_in_every_position(position):
    D = 128
    lay = kvarn.layout(D)
    args = [("q", _pair(torch.zeros(1, 8, D))),
            ("tiles", _pair(torch.zeros(lay.record_bytes, dtype=torch.uint8))),
            ("tile_table", _pair(torch.zeros(1, 2, 1, dtype=torch.int64))),
            ("n_tiles", _pair(torch.ones(1, dtype=torch.int32))),
            ("win_k", _pair(torch.zeros(1, 2, 128, D))), ("win_v", _pair(torch.zeros(1, 2, 128, D))),
            ("win_start", _pair(torch.zeros(1, dtype=torch.int32))),
            ("win_len", _pair(torch.zeros(1, dtype=torch.int32)))]
    for fn in (kvarn.decode_attention, kvarn.decode_attention_noalloc):
        _refuses(lambda *a: fn(*a, lay), args, {}, position)
    ws = _fake(torch.zeros(1 << 16, dtype=torch.uint8))
    _refuses(lambda *a: kvarn.decode_split(*a, lay, ws), args, {}, position)


@pytest.mark.parametrize("position", ["q_chunk", "tiles", "tile_table", "win_k", "win_v"])
def test_prefill_refuses_a_host_tensor_in_every_position(position):
    D = 128
    lay = kvarn.layout(D)
    q = _pair(torch.zeros(4, 8, D))
    tiles = _pair(torch.zeros(lay.record_bytes, dtype=torch.uint8))
    tab = _pair(torch.zeros(2, 1, dtype=torch.int64))
    wk, wv = _pair(torch.zeros(2, 128, D)), _pair(torch.zeros(2, 128, D))
    args = [("q_chunk", q), ("pos0", (0, 0)), ("tiles", tiles), ("tile_table", tab),
            ("n_tiles", (1, 1)), ("win_k", wk), ("win_v", wv), ("win_start", (0, 0)),
            ("win_len", (4, 4))]
    _refuses(lambda *a: kvarn.prefill_attention(*a, lay), args, {}, position)


@pytest.mark.parametrize("position", ["k_raw", "v_raw", "src_row0", "tiles", "dst_record"])
def test_compress_refuses_a_host_tensor_in_every_position(position):
    lay = kvarn.layout(128)
    args = [("k_raw", _pair(torch.zeros(128, 128))), ("v_raw", _pair(torch.zeros(128, 128))),
            ("src_row0", _pair(torch.zeros(1, dtype=torch.int64))),
            ("tiles", _pair(torch.zeros(lay.record_bytes, dtype=torch.uint8))),
            ("dst_record", _pair(torch.zeros(1, dtype=torch.int64)))]
    _refuses(lambda *a: kvarn.compress_tile(*a, lay), args, {}, position)


@pytest.mark.parametrize("position", ["k_new", "v_new", "win_k", "win_v", "win_start", "win_len"])
def test_append_refuses_a_host_tensor_in_every_position(position):
    args = [("k_new", _pair(torch.zeros(1, 1, 2, 128))), ("v_new", _pair(torch.zeros(1, 1, 2, 128))),
            ("win_k", _pair(torch.zeros(1, 2, 128, 128))), ("win_v", _pair(torch.zeros(1, 2, 128, 128))),
            ("win_start", _pair(torch.zeros(1, dtype=torch.int32))),
            ("win_len", _pair(torch.zeros(1, dtype=torch.int32)))]
    _refuses(kvarn.append_window, args, {}, position)


def test_wrong_dtype_and_non_contiguous_are_refused():
    lay = kvarn.layout(128)
    q = _fake(torch.zeros(1, 8, 128))
    tiles = _fake(torch.zeros(64, dtype=torch.uint8))
    tab32 = _fake(torch.zeros(1, 2, 1, dtype=torch.int32))
    n = _fake(torch.ones(1, dtype=torch.int32))
    win = _fake(torch.zeros(1, 2, 128, 128))
    with pytest.raises(TypeError, match="tile_table must be torch.int64"):
        kvarn.decode_attention(q, tiles, tab32, n, win, win, n, n, lay)
    wt = _fake(torch.zeros(1, 2, 128, 128).transpose(2, 3))
    tab = _fake(torch.zeros(1, 2, 1, dtype=torch.int64))
    with pytest.raises(ValueError, match="win_k must be contiguous"):
        kvarn.decode_attention(q, tiles, tab, n, wt, win, n, n, lay)


def test_missing_library_raises():
    """With the library path pointing nowhere, the first call raises."""
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "from kv_cache_quantization_token_gb300 import kvarn\n"
        "kvarn._lib = None\n"
        "kvarn.library_path = lambda: '/nonexistent/libkvarn.so'\n"
        "try:\n"
        "    kvarn.layout(128)\n"
        "except RuntimeError as e:\n"
        "    print('raised:', e)\n"
        "else:\n"
        "    print('no error')\n" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.startswith("raised:"), r.stdout
