"""GPU tile compression vs the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_quantization_token_gb300 import kvarn, synth
from tests.kvarn_helpers import compare_record

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _compress(k_rows, v_rows, units, D, iters=4, row_stride=None):
    """k_rows/v_rows: fp32 [n][D]; units: list of first rows. Returns records."""
    lay = kvarn.layout(D, iters)
    rb = lay.record_bytes
    n = k_rows.shape[0]
    if row_stride is not None and row_stride != D:
        kp = np.zeros((n, row_stride), np.float32)
        vp = np.zeros((n, row_stride), np.float32)
        kp[:, :D], vp[:, :D] = k_rows, v_rows
        kp[:, D:], vp[:, D:] = 1e30, -1e30  # padding must never be read
        k_rows, v_rows = kp, vp
    tiles = torch.full((len(units) * rb,), 0xAB, dtype=torch.uint8, device=DEV)
    # records go to a permuted order of slots: placement must not matter
    slots = np.random.default_rng(len(units)).permutation(len(units))
    kvarn.compress_tile(torch.from_numpy(k_rows).to(DEV), torch.from_numpy(v_rows).to(DEV),
                        torch.tensor(units, dtype=torch.int64, device=DEV), tiles,
                        torch.tensor(slots * rb, dtype=torch.int64, device=DEV), lay)
    host = tiles.cpu().numpy()
    return [host[s * rb:(s + 1) * rb] for s in slots]


@pytest.mark.parametrize("workload,D,n_heads,n_tiles", [("single_tile", 128, 1, 1), ("qwen3_0p6b_decode", 128, 2, 4), ("qwen3_8b_decode", 128, 2, 4),
                                                    ("batched_d256_decode", 256, 2, 3), ("qwen3_8b_decode", 64, 2, 3), ("single_tile", 64, 1, 2),
                                                    ("batched_d256_decode", 128, 1, 2)])
def test_compress_matches_oracle(workload, D, n_heads, n_tiles):
    ks, vs = synth.kv_layer(workload, 3, n_heads, 128 * n_tiles, D)
    k_rows, v_rows = ks.reshape(-1, D), vs.reshape(-1, D)
    units = [128 * i for i in range(n_heads * n_tiles)]
    recs = _compress(k_rows, v_rows, units, D)
    flips = total = 0
    for u, rec in zip(units, recs):
        ref = oracle.compress_unit(k_rows[u:u + 128], v_rows[u:u + 128])
        st = compare_record(rec, ref, D)
        flips += st["band_flips"]
        total += st["codes"]
    print(f"{workload} D{D}: {flips} boundary-band flips of {total} codes")


def test_compress_strided_rows_and_offsets():
    D = 128
    ks, vs = synth.kv_layer("qwen3_8b_decode", 5, 1, 128 * 3 + 40, D)
    k_rows, v_rows = ks[0], vs[0]
    units = [0, 40, 128 + 40, 256]  # overlapping and unaligned-to-128 starts
    recs = _compress(k_rows, v_rows, units, D, row_stride=D + 8)
    for u, rec in zip(units, recs):
        compare_record(rec, oracle.compress_unit(k_rows[u:u + 128], v_rows[u:u + 128]), D)


@pytest.mark.parametrize("iters", [1, 2, 7])
def test_compress_other_iteration_counts(iters):
    D = 128
    ks, vs = synth.kv_layer("single_tile", 2, 1, 256, D)
    recs = _compress(ks[0], vs[0], [0, 128], D, iters=iters)
    for u, rec in zip([0, 128], recs):
        compare_record(rec, oracle.compress_unit(ks[0, u:u + 128], vs[0, u:u + 128], iters), D)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_compress_degenerate_tiles(D):
    """All-zero tile; a tile of identical tokens (every channel constant); a
    tile with zero tokens and a zero channel."""
    rng = np.random.default_rng(D)
    zero = np.zeros((128, D), np.float32)
    same = np.tile(rng.standard_normal(D).astype(np.float32), (128, 1))
    holes = rng.standard_normal((128, D)).astype(np.float32)
    holes[::7] = 0.0
    holes[:, 3] = 0.0
    k_rows = np.concatenate([zero, same, holes])
    v_rows = np.concatenate([zero, same[::-1] * 2, holes * 0.5])
    recs = _compress(k_rows, v_rows, [0, 128, 256], D)
    for u, rec in zip([0, 128, 256], recs):
        compare_record(rec, oracle.compress_unit(k_rows[u:u + 128], v_rows[u:u + 128]), D)
    z = oracle.unpack_record(recs[0], D)
    assert np.all(z["k_codes"] == 0) and np.all(z["k_delta"] == 0) and np.all(z["k_s"] == 1)


def test_compress_is_deterministic_and_schedule_independent():
    D = 128
    ks, vs = synth.kv_layer("qwen3_8b_decode", 9, 1, 128 * 8, D)
    units = [128 * i for i in range(8)]
    a = _compress(ks[0], vs[0], units, D)
    b = _compress(ks[0], vs[0], units[::-1], D)[::-1]
    c = _compress(ks[0], vs[0], units[3:4], D)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert np.array_equal(a[3], c[0])


def test_compress_bulk_launch_sampled():
    """The benchmarked bulk launch: 256 tiles x 8 KV heads of 32k-token
    8B-like caches (2048 units, 256 MiB of input) in one call; a seeded sample
    of the units is checked against the oracle."""
    D, n_tiles, n_heads = 128, 256, 8
    ks, vs = synth.kv_layer("qwen3_8b_decode", 99, n_heads, 128 * n_tiles, D)
    k_rows, v_rows = ks.reshape(-1, D), vs.reshape(-1, D)
    units = [128 * i for i in range(n_heads * n_tiles)]
    lay = kvarn.layout(D)
    rb = lay.record_bytes
    tiles = torch.zeros(len(units) * rb, dtype=torch.uint8, device=DEV)
    kvarn.compress_tile(torch.from_numpy(k_rows).to(DEV), torch.from_numpy(v_rows).to(DEV),
                        torch.tensor(units, dtype=torch.int64, device=DEV), tiles,
                        torch.arange(len(units), dtype=torch.int64, device=DEV) * rb, lay)
    host = tiles.cpu().numpy()
    pick = np.random.default_rng(2048).choice(len(units), 12, replace=False)
    for i in sorted(pick.tolist()) + [0, len(units) - 1]:
        u = units[i]
        compare_record(host[i * rb:(i + 1) * rb],
                       oracle.compress_unit(k_rows[u:u + 128], v_rows[u:u + 128]), D)


@pytest.mark.parametrize("workload,D,n_heads,n_tiles", [("qwen3_8b_decode", 128, 2, 4),
                                                       ("batched_d256_decode", 256, 2, 3),
                                                       ("single_tile", 64, 1, 2)])
def test_compress_f16_scales_matches_oracle(workload, D, n_heads, n_tiles):
    """The f16-scale layout: the same codes, every scale field binary16."""
    from tests.kvarn_helpers import compare_record_f16
    ks, vs = synth.kv_layer(workload, 4, n_heads, 128 * n_tiles, D)
    k_rows, v_rows = ks.reshape(-1, D), vs.reshape(-1, D)
    units = [128 * i for i in range(n_heads * n_tiles)]
    lay = kvarn.layout(D, scale_bits=16)
    rb = lay.record_bytes
    assert rb == oracle.record_bytes(D, 16)
    tiles = torch.full((len(units) * rb,), 0xAB, dtype=torch.uint8, device=DEV)
    kvarn.compress_tile(torch.from_numpy(k_rows).to(DEV), torch.from_numpy(v_rows).to(DEV),
                        torch.tensor(units, dtype=torch.int64, device=DEV), tiles,
                        torch.arange(len(units), dtype=torch.int64, device=DEV) * rb, lay)
    host = tiles.cpu().numpy()
    flips = 0
    for i, u in enumerate(units):
        ref = oracle.compress_unit(k_rows[u:u + 128], v_rows[u:u + 128], scale_bits=16)
        flips += compare_record_f16(host[i * rb:(i + 1) * rb], ref, D)["scale_flips"]
    print(f"{workload} D{D} f16 scales: {flips} binary16 rounding-midpoint flips")


@pytest.mark.parametrize("workload,D,n_heads,n_tiles,sb", [("qwen3_8b_decode", 128, 2, 4, 32),
                                                          ("batched_d256_decode", 256, 2, 3, 32),
                                                          ("single_tile", 64, 1, 2, 32),
                                                          ("qwen3_8b_decode", 128, 1, 3, 16)])
def test_compress_v4_matches_oracle(workload, D, n_heads, n_tiles, sb):
    """The k4v4 variant: 4-bit values (16 levels per token group), packed
    token-major two channels per byte; keys as in the k4v2 record."""
    from tests.kvarn_helpers import compare_record_f16
    ks, vs = synth.kv_layer(workload, 8, n_heads, 128 * n_tiles, D)
    k_rows, v_rows = ks.reshape(-1, D), vs.reshape(-1, D)
    units = [128 * i for i in range(n_heads * n_tiles)]
    lay = kvarn.layout(D, scale_bits=sb, v_bits=4)
    rb = lay.record_bytes
    assert rb == oracle.record_bytes(D, sb, 4)
    tiles = torch.full((len(units) * rb,), 0xAB, dtype=torch.uint8, device=DEV)
    kvarn.compress_tile(torch.from_numpy(k_rows).to(DEV), torch.from_numpy(v_rows).to(DEV),
                        torch.tensor(units, dtype=torch.int64, device=DEV), tiles,
                        torch.arange(len(units), dtype=torch.int64, device=DEV) * rb, lay)
    host = tiles.cpu().numpy()
    flips = 0
    for i, u in enumerate(units):
        ref = oracle.compress_unit(k_rows[u:u + 128], v_rows[u:u + 128], scale_bits=sb, v_bits=4)
        rec = host[i * rb:(i + 1) * rb]
        st = compare_record(rec, ref, D, v_bits=4) if sb == 32 else compare_record_f16(rec, ref, D, 4)
        flips += st["band_flips"]
    print(f"{workload} D{D} k4v4 sb{sb}: {flips} boundary-band flips")


@pytest.mark.parametrize("workload,D,n_heads,n_tiles,sb", [("qwen3_8b_decode", 128, 2, 4, 32),
                                                          ("batched_d256_decode", 256, 2, 3, 32),
                                                          ("single_tile", 64, 1, 2, 32),
                                                          ("qwen3_8b_decode", 128, 1, 3, 16)])
def test_compress_v3_matches_oracle(workload, D, n_heads, n_tiles, sb):
    """The k4v3 variant: 3-bit values (8 levels per token group), each token
    row a bit stream in which 3-bit codes straddle bytes; keys as in k4v2."""
    from tests.kvarn_helpers import compare_record_f16
    ks, vs = synth.kv_layer(workload, 9, n_heads, 128 * n_tiles, D)
    k_rows, v_rows = ks.reshape(-1, D), vs.reshape(-1, D)
    units = [128 * i for i in range(n_heads * n_tiles)]
    lay = kvarn.layout(D, scale_bits=sb, v_bits=3)
    rb = lay.record_bytes
    assert rb == oracle.record_bytes(D, sb, 3)
    tiles = torch.full((len(units) * rb,), 0xAB, dtype=torch.uint8, device=DEV)
    kvarn.compress_tile(torch.from_numpy(k_rows).to(DEV), torch.from_numpy(v_rows).to(DEV),
                        torch.tensor(units, dtype=torch.int64, device=DEV), tiles,
                        torch.arange(len(units), dtype=torch.int64, device=DEV) * rb, lay)
    host = tiles.cpu().numpy()
    flips = 0
    for i, u in enumerate(units):
        ref = oracle.compress_unit(k_rows[u:u + 128], v_rows[u:u + 128], scale_bits=sb, v_bits=3)
        rec = host[i * rb:(i + 1) * rb]
        st = compare_record(rec, ref, D, v_bits=3) if sb == 32 else compare_record_f16(rec, ref, D, 3)
        flips += st["band_flips"]
    print(f"{workload} D{D} k4v3 sb{sb}: {flips} boundary-band flips")
