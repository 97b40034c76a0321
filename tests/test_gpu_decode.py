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
    kvarn.device_error(clear=True)
    out = kvarn.decode_attention(q, pool, table, c.n_tiles, c.win_k, c.win_v, c.win_start,
                                 c.win_len, c.lay).cpu().numpy()
    assert np.isnan(out[0, 4:]).all()          # query heads of KV head 1
    assert np.array_equal(out[0, :4], good[0, :4])
    assert kvarn.device_error(clear=True) == kvarn.DEVERR_RECORD  # reported, then cleared


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


def test_qwen3_8b_like_32k_sampled_heads():
    """The 32k point of the 8B-like sweep (32q/8kv, 257 tiles per KV head):
    the multi-round split kernel on one GB300."""
    c = Cache("qwen3_8b_decode", 3, [32768 + 77], Hkv=8, D=128)
    _check(c, Hq=32, heads=[(0, 0), (0, 11), (0, 29)])


def test_batched_d256_full_config_sampled():
    """The benchmarked batched decode: 32 sequences with contexts uniform in
    [8192, 32768] (the same seeded draw), 16q/4kv, head_dim 256. Every
    sequence's tiles repeat a pool of 64 compressed tiles per KV head (as in
    the benchmark); sampled (sequence, head) outputs against the oracle."""
    import oracle
    B, Hq, Hkv, D, cap, pool_tiles = 32, 16, 4, 256, 128, 64
    ctxs = synth.uniform_ints(4242, 8192, 32768, B)
    ntl, wlen = ctxs // 128, ctxs % 128
    mt = int(ntl.max()) + 1
    lay = kvarn.layout(D)
    rb = lay.record_bytes
    ks, vs = synth.kv_layer("batched_d256_decode", 0, Hkv, 128 * pool_tiles + cap, D)
    pool = torch.zeros(Hkv * pool_tiles * rb, dtype=torch.uint8, device=DEV)
    src = np.array([h * (128 * pool_tiles + cap) + 128 * t for h in range(Hkv) for t in range(pool_tiles)])
    kvarn.compress_tile(torch.from_numpy(ks.reshape(-1, D)).to(DEV), torch.from_numpy(vs.reshape(-1, D)).to(DEV),
                        torch.from_numpy(src.astype(np.int64)).to(DEV), pool,
                        torch.arange(Hkv * pool_tiles, dtype=torch.int64, device=DEV) * rb, lay)
    table = ((np.arange(Hkv)[None, :, None] * pool_tiles + (np.arange(mt)[None, None, :] % pool_tiles))
             * rb * np.ones((B, 1, 1), np.int64)).astype(np.int64)
    win_k = np.broadcast_to(ks[None, :, 128 * pool_tiles:], (B, Hkv, cap, D)).copy()
    win_v = np.broadcast_to(vs[None, :, 128 * pool_tiles:], (B, Hkv, cap, D)).copy()
    q = synth.queries("batched_d256_decode", 0, (B, Hq, D))
    out = kvarn.decode_attention(torch.from_numpy(q).to(DEV), pool, torch.from_numpy(table).to(DEV),
                                 torch.from_numpy(ntl.astype(np.int32)).to(DEV),
                                 torch.from_numpy(win_k).to(DEV), torch.from_numpy(win_v).to(DEV),
                                 torch.zeros(B, dtype=torch.int32, device=DEV),
                                 torch.from_numpy(wlen.astype(np.int32)).to(DEV), lay).cpu().numpy()
    heads = [(b, h) for b in (0, 7, 19, 31) for h in (0, 9, 15)]
    ref = oracle.decode_attention(q, pool.cpu().numpy(), table, [int(x) for x in ntl], win_k, win_v,
                                  [0] * B, [int(x) for x in wlen], D ** -0.5, heads=heads)
    for (b, h), r in ref.items():
        e = rel_l2(out[b, h], r)
        assert e <= ATTN_RTOL, f"(b={b}, h={h}) rel-L2 {e:.3e}"


@pytest.mark.parametrize("workload,ctxs,Hq,Hkv,D", [("single_tile", [128 + 17], 1, 1, 128),
                                                   ("qwen3_8b_decode", [16384 + 40], 32, 8, 128),
                                                   ("qwen3_8b_decode", [600, 1000], 8, 1, 128),
                                                   ("batched_d256_decode", [900, 128 * 5 + 3], 16, 4, 256),
                                                   ("single_tile", [128 * 3 + 50], 4, 2, 64)])
def test_f16_scale_records(workload, ctxs, Hq, Hkv, D):
    """Decode over records of the f16-scale layout (binary16 scale fields,
    14,336-byte records at head_dim 128): the oracle dequantises the same
    records with the stored binary16 values."""
    c = Cache(workload, 14, ctxs, Hkv=Hkv, D=D, scale_bits=16)
    assert c.rb == 96 * D + 2 * (4 * D + 256 + 256 * (D // min(D, 128)))
    heads = [(b, h) for b in range(len(ctxs)) for h in range(0, Hq, max(1, Hq // 4))]
    _check(c, Hq=Hq, heads=heads)


def test_f16_scale_records_multi_round():
    """The multi-round split kernel (more than 8 tiles per SM) on f16-scale records."""
    c = Cache("qwen3_8b_decode", 15, [128 * 1400 + 9], Hkv=1, D=128, scale_bits=16)
    _check(c, Hq=8, heads=[(0, h) for h in range(0, 8, 3)])


@pytest.mark.parametrize("workload,ctxs,Hq,Hkv,D,sb", [("single_tile", [128 + 17], 1, 1, 128, 32),
                                                      ("qwen3_8b_decode", [16384 + 40], 32, 8, 128, 32),
                                                      ("qwen3_8b_decode", [600, 1000], 8, 1, 128, 16),
                                                      ("batched_d256_decode", [900, 128 * 5 + 3], 16, 4, 256, 32),
                                                      ("single_tile", [128 * 3 + 50], 4, 2, 64, 32),
                                                      ("qwen3_8b_decode", [700], 24, 8, 128, 32)])
def test_v4_records(workload, ctxs, Hq, Hkv, D, sb):
    """Decode over k4v4 records (4-bit values, 20,480-byte records at
    head_dim 128 with fp32 scales): the value contraction reads two channels
    per code byte; the oracle dequantises the same records."""
    c = Cache(workload, 16, ctxs, Hkv=Hkv, D=D, scale_bits=sb, v_bits=4)
    heads = [(b, h) for b in range(len(ctxs)) for h in range(0, Hq, max(1, Hq // 4))]
    _check(c, Hq=Hq, heads=heads)


@pytest.mark.parametrize("D,Hq,Hkv,ctx", [(128, 8, 1, 128 * 1400 + 9), (256, 16, 4, 128 * 460 + 77)])
def test_v4_records_multi_round(D, Hq, Hkv, ctx):
    """The multi-round split kernel on k4v4 records."""
    c = Cache("qwen3_8b_decode", 17, [ctx], Hkv=Hkv, D=D, v_bits=4)
    _check(c, Hq=Hq, heads=[(0, h) for h in range(0, Hq, 5)])


@pytest.mark.parametrize("workload,ctxs,Hq,Hkv,D,sb", [("single_tile", [128 + 17], 1, 1, 128, 32),
                                                      ("qwen3_8b_decode", [16384 + 40], 32, 8, 128, 32),
                                                      ("qwen3_8b_decode", [600, 1000], 8, 1, 128, 16),
                                                      ("batched_d256_decode", [900, 128 * 5 + 3], 16, 4, 256, 32),
                                                      ("single_tile", [128 * 3 + 50], 4, 2, 64, 32)])
def test_v3_records(workload, ctxs, Hq, Hkv, D, sb):
    """Decode over k4v3 records (3-bit values straddling bytes, 18,432-byte
    records at head_dim 128 with fp32 scales): after the scores, the warp
    group rewrites a record's value codes as 4-bit rows over its K codes and
    the value contraction reads those; the oracle dequantises the records."""
    c = Cache(workload, 18, ctxs, Hkv=Hkv, D=D, scale_bits=sb, v_bits=3)
    heads = [(b, h) for b in range(len(ctxs)) for h in range(0, Hq, max(1, Hq // 4))]
    _check(c, Hq=Hq, heads=heads)


@pytest.mark.parametrize("D,Hq,Hkv,ctx", [(128, 8, 1, 128 * 1400 + 9), (256, 16, 4, 128 * 460 + 77)])
def test_v3_records_multi_round(D, Hq, Hkv, ctx):
    """The multi-round split kernel (records double-buffered) on k4v3 records."""
    c = Cache("qwen3_8b_decode", 19, [ctx], Hkv=Hkv, D=D, v_bits=3)
    _check(c, Hq=Hq, heads=[(0, h) for h in range(0, Hq, 5)])
