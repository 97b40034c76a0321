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
