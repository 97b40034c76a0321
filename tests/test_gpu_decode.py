"""GPU decode attention (split + LSE combine) vs the fp64 oracle, computed on
the GPU's own packed records."""
import numpy as np
import pytest
import torch

from kv_cache_quantization_token_gb300 import kvarn, synth
from tests.kvarn_helpers import ATTN_RTOL, Cache, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _check(cache, Hq, heads=None, scale=None, seed=0):
    q = synth.queries(cache.workload, seed, (cache.B, Hq, cache.D))
    out = cache.decode(torch.from_numpy(q).to(DEV), scale=scale).cpu().numpy()
    ref = cache.oracle_decode(q, heads=heads, scale=scale)
    worst = 0.0
    for (b, h), r in ref.items():
        e = rel_l2(out[b, h], r)
        worst = max(worst, e)
        assert e <= ATTN_RTOL, f"(b={b}, h={h}) rel-L2 {e:.3e}"
    return out, worst


def test_single_tile_plus_17_window():
    c = Cache("single_tile", 0, [128 + 17], Hkv=1, D=128)
    _check(c, Hq=1)


@pytest.mark.parametrize("w", [0, 1, 127, 77])
def test_qwen3_0p6b_like_3k(w):
    """16q/8kv, D=128, 3072 + w tokens (24 tiles + w-token window)."""
    c = Cache("qwen3_0p6b_decode", 4, [3072 + w], Hkv=8, D=128)
    _check(c, Hq=16, heads=[(0, h) for h in (0, 5, 10, 15)])


@pytest.mark.parametrize("ctx", [4096, 4096 + 77])
def test_qwen3_8b_like(ctx):
    c = Cache("qwen3_8b_decode", 1, [ctx], Hkv=8, D=128)
    _check(c, Hq=32, heads=[(0, h) for h in (0, 3, 17, 31)])


def test_qwen3_8b_like_16k_sampled_heads():
    c = Cache("qwen3_8b_decode", 2, [16384], Hkv=8, D=128)
    _check(c, Hq=32, heads=[(0, 0), (0, 13), (0, 30)])


def test_ragged_batch32_d256():
    ctxs = [900, 128 * 5 + 3, 256, 1500]
    c = Cache("batched_d256_decode", 0, ctxs, Hkv=4, D=256)
    _check(c, Hq=16, heads=[(b, h) for b in range(4) for h in (0, 7, 15)])


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (24, 8), (8, 1)])
def test_gqa_groups(Hq, Hkv):
    """G = 1, 3 (padded group of 4) and 8."""
    c = Cache("qwen3_8b_decode", 6, [600], Hkv=Hkv, D=128)
    _check(c, Hq=Hq)


def test_d64_and_window_wraparound():
    c = Cache("single_tile", 7, [128 * 3 + 200], Hkv=2, D=64, W=256, cap=384, win_start=[256])
    assert c.wl == [200] and c.cap == 384
    _check(c, Hq=4)


def test_empty_and_window_only_and_tiles_only():
    c = Cache("qwen3_8b_decode", 8, [0, 50, 256, 128], Hkv=2, D=128)
    out, _ = _check(c, Hq=4)
    assert np.all(out[0] == 0.0)


def test_custom_scale_and_determinism():
    c = Cache("qwen3_8b_decode", 9, [1000], Hkv=2, D=128)
    q = torch.from_numpy(synth.queries("qwen3_8b_decode", 1, (1, 8, 128))).to(DEV)
    a = c.decode(q, scale=0.3)
    b = c.decode(q, scale=0.3)
    assert torch.equal(a, b)
    _check(c, Hq=8, scale=0.3, seed=1)


def test_offset_not_multiple_of_128_poisons_only_that_head():
    c = Cache("qwen3_8b_decode", 11, [128 * 3 + 10], Hkv=2, D=128)
    q = torch.from_numpy(synth.queries("qwen3_8b_decode", 11, (1, 8, 128))).to(DEV)
    good = c.decode(q).cpu().numpy()
    n = c.tiles.numel()
    pool = torch.zeros(n + c.rb + 256, dtype=torch.uint8, device=DEV)
    pool[:n] = c.tiles
    pool[n + 16:n + 16 + c.rb] = c.tiles[int(c.tile_table[0, 1, 0]):int(c.tile_table[0, 1, 0]) + c.rb]
    table = c.tile_table.clone()
    table[0, 1, 0] = n + 16  # 16-byte aligned, not a multiple of 128
    out = kvarn.decode_attention(q, pool, table, c.n_tiles, c.win_k, c.win_v, c.win_start,
                                 c.win_len, c.lay).cpu().numpy()
    assert np.isnan(out[0, 4:]).all()          # query heads of KV head 1
    assert np.array_equal(out[0, :4], good[0, :4])


@pytest.mark.parametrize("workload,Hq,Hkv,D,ctx", [("single_tile", 8, 8, 64, 128 * 80 + 33),
                                                  ("qwen3_8b_decode", 8, 1, 128, 128 * 620 + 5)])
def test_four_tiles_per_item_path(workload, Hq, Hkv, D, ctx):
    """Grids with at least 4 tiles per SM take the 8-warp, 4-tiles-per-item
    split kernel: head_dim 64, and a GQA group of 8 (two n8-tiles of columns)."""
    c = Cache(workload, 12, [ctx], Hkv=Hkv, D=D)
    assert Hkv * c.max_tiles >= 4 * 152
    _check(c, Hq=Hq, heads=[(0, h) for h in range(0, Hq, 3)])


@pytest.mark.parametrize("workload,Hq,Hkv,D,ctx", [("qwen3_8b_decode", 8, 1, 128, 128 * 1400 + 9),
                                                  ("qwen3_8b_decode", 16, 2, 128, 128 * 1330 + 100),
                                                  ("batched_d256_decode", 16, 4, 256, 128 * 460 + 77)])
def test_multi_round_items(workload, Hq, Hkv, D, ctx):
    """Grids with many more tiles than the SMs hold at once take the split
    kernel in which each warp group works through several tiles in turn while
    its next record is copied into a second slot (head_dim 128: more than 8
    tiles per SM; head_dim 256: at least 12). Tile counts leave the last item
    and the last round of some groups partly empty."""
    c = Cache(workload, 13, [ctx], Hkv=Hkv, D=D)
    per_sm = Hkv * c.max_tiles // 152
    assert per_sm > (8 if D == 128 else 11)
    _check(c, Hq=Hq, heads=[(0, h) for h in range(0, Hq, 5)])
