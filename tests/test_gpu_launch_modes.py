"""Decode under the three launch modes of kvarn_set_launch_flags gives
bit-identical results, eagerly and inside a captured CUDA graph."""
import numpy as np
import pytest
import torch

from kv_cache_quantization_token_gb300 import kvarn, synth
from kvarn_helpers import Cache

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MODES = [0, kvarn.LAUNCH_PDL, kvarn.LAUNCH_PDL | kvarn.LAUNCH_PREFETCH]


@pytest.fixture(autouse=True)
def _reset_flags():
    yield
    kvarn.set_launch_flags(0)


def _layers(n_layers=3):
    caches = [Cache("qwen3_8b_decode", 30 + l, [128 * 9 + 70, 128 * 4 + 5], Hkv=8, D=128)
              for l in range(n_layers)]
    qs = [torch.from_numpy(synth.queries("qwen3_8b_decode", 30 + l, (2, 32, 128))).to(DEV)
          for l in range(n_layers)]
    kn = [torch.from_numpy(synth.queries("qwen3_8b_decode", 60 + l, (2, 1, 8, 128))).to(DEV)
          for l in range(n_layers)]
    return caches, qs, kn


def _step(caches, qs, kn, outs, ws):
    # per layer: attend, then append the layer's next token (as a decode loop does)
    for c, q, k, o in zip(caches, qs, kn, outs):
        kvarn.decode_split(q, c.tiles, c.tile_table, c.n_tiles, c.win_k, c.win_v, c.win_start,
                           c.win_len, c.lay, ws)
        kvarn.decode_combine(ws, o, c.Hkv, c.max_tiles, c.cap)
        kvarn.append_window(k, k, c.win_k, c.win_v, c.win_start, c.win_len)


def _run(mode, graph):
    kvarn.set_launch_flags(mode)
    caches, qs, kn = _layers()
    c0 = caches[0]
    ws = torch.empty(kvarn.decode_workspace_bytes(2, 32, 8, 128, c0.max_tiles, c0.cap) + 256,
                     dtype=torch.uint8, device=DEV)
    outs = [torch.empty(2, 32, 128, device=DEV) for _ in caches]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            _step(caches, qs, kn, outs, ws)
        g.replay()
    else:
        with torch.cuda.stream(stream):
            _step(caches, qs, kn, outs, ws)
    torch.cuda.synchronize()
    return [o.cpu() for o in outs] + [c.win_k.cpu() for c in caches]


@pytest.mark.parametrize("graph", [False, True])
def test_launch_modes_bit_identical(graph):
    ref = _run(0, graph)
    for mode in MODES[1:]:
        got = _run(mode, graph)
        for a, b in zip(ref, got):
            assert torch.equal(a, b), f"mode {mode} graph {graph}"
    assert all(np.isfinite(r.numpy()).all() for r in ref)


def test_first_layer_matches_oracle_under_prefetch():
    kvarn.set_launch_flags(kvarn.LAUNCH_PDL | kvarn.LAUNCH_PREFETCH)
    c = Cache("qwen3_8b_decode", 40, [128 * 6 + 30], Hkv=8, D=128)
    q = synth.queries("qwen3_8b_decode", 40, (1, 32, 128))
    out = c.decode(torch.from_numpy(q).to(DEV)).cpu().numpy()
    ref = c.oracle_decode(q)
    for h in range(32):
        err = np.linalg.norm(out[0, h] - ref[0, h]) / np.linalg.norm(ref[0, h])
        assert err < 1e-4, (h, err)
