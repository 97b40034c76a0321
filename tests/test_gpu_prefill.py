"""GPU chunked-prefill attention (tcgen05) vs the fp64 oracle's causal
attention, evaluated on the GPU's own tiles and window."""
import numpy as np
import pytest
import torch

from kv_cache_quantization_token_gb300 import kvarn, synth
from tests.kvarn_helpers import ATTN_RTOL, Cache, PrefillRun, rel_l2

pytestmark = pytest.mark.gpu


def _rows(C, heads, step=37):
    idx = sorted(set([0, 1, 2, 63, 64, 127, 128, 255, 256, 511, C - 1] + list(range(0, C, step))))
    return [(i, h) for i in idx if i < C for h in heads]


def test_prefill_15k_prompt_prefix_chunks():
    """32q/8kv, D=128, W=256, 512-token chunks over a 2188-token prefix."""
    run = PrefillRun("qwen3_8b_prefill", 0, 2048 + 140, Hq=32, Hkv=8, D=128)
    worst = max(run.check(p, _rows(run.snap[p]["C"], (0, 5, 18, 31))) for p in run.snap)
    print(f"prefill D128 worst rel-L2 {worst:.2e}")


@pytest.mark.parametrize("Hq,Hkv,D,n,chunk,W", [(8, 8, 64, 700, 256, 128), (16, 2, 128, 900, 300, 256),
                                                 (12, 4, 64, 650, 200, 128), (4, 4, 128, 300, 96, 128)])
def test_prefill_shapes(Hq, Hkv, D, n, chunk, W):
    """GQA groups 1, 8 and 3 (padded rows), D=64, ragged chunks, windows that wrap."""
    run = PrefillRun("qwen3_8b_decode", 1, n, Hq=Hq, Hkv=Hkv, D=D, W=W, chunk=chunk)
    for p in run.snap:
        run.check(p, _rows(run.snap[p]["C"], range(0, Hq, 3), step=19))


def test_prefill_chunk_of_one_equals_decode():
    """A one-token chunk is a decode step over the same cache (both within
    1e-4 of the oracle, so within 2e-4 of each other)."""
    n = 128 * 3 + 40
    run = PrefillRun("qwen3_8b_decode", 2, n, Hq=8, Hkv=2, D=128, W=128, chunk=1, keep=[n - 1])
    s = run.snap[n - 1]
    dev = torch.device("cuda:0")
    q = torch.from_numpy(run.q[n - 1:n]).to(dev)
    dec = kvarn.decode_attention(q, run.tiles, run.table[None], torch.tensor([s["n_tiles"]],
                                 dtype=torch.int32, device=dev),
                                 torch.from_numpy(s["win_k"])[None].to(dev),
                                 torch.from_numpy(s["win_v"])[None].to(dev),
                                 torch.tensor([s["start"]], dtype=torch.int32, device=dev),
                                 torch.tensor([s["length"]], dtype=torch.int32, device=dev),
                                 run.lay).cpu().numpy()
    for h in range(8):
        assert rel_l2(s["out"][0, h], dec[0, h].astype(np.float64)) <= 2e-4
    run.check(n - 1, [(0, h) for h in range(8)])


def test_prefill_15k_prompt_full_sampled():
    """15,500 tokens = 30 x 512 + 140; every 64th row of the last chunk and a
    middle chunk, two KV heads' query heads."""
    n = 15500
    run = PrefillRun("qwen3_8b_prefill", 3, n, Hq=32, Hkv=8, D=128, keep=[512 * 15, 512 * 30])
    assert run.n_tiles == (n - 256) // 128 + 1
    for p in run.snap:
        C = run.snap[p]["C"]
        rows = [(i, h) for i in list(range(0, C, 64)) + [C - 1] for h in (0, 3, 28, 31)]
        w = run.check(p, rows)
        print(f"15.5k chunk {p}: worst rel-L2 {w:.2e}")


@pytest.mark.parametrize("Hq,Hkv,D,n,chunk,W", [(16, 2, 128, 900, 300, 256), (8, 8, 64, 700, 256, 128)])
def test_prefill_f16_scale_records(Hq, Hkv, D, n, chunk, W):
    """Chunked prefill over records of the f16-scale layout."""
    run = PrefillRun("qwen3_8b_decode", 5, n, Hq=Hq, Hkv=Hkv, D=D, W=W, chunk=chunk, scale_bits=16)
    for p in run.snap:
        run.check(p, _rows(run.snap[p]["C"], range(0, Hq, 3), step=19))


@pytest.mark.parametrize("Hq,Hkv,D,n,chunk,W,sb", [(32, 8, 128, 2188, 512, 256, 32),
                                                  (12, 4, 64, 650, 200, 128, 32),
                                                  (16, 2, 128, 900, 300, 256, 16)])
def test_prefill_cached_images_match_uncached(Hq, Hkv, D, n, chunk, W, sb):
    """kvarn_prefill_attention_cached with one workspace for the whole prompt
    (each chunk converts only the newly promoted tiles) gives the same bits as
    converting every visible tile in every chunk, and matches the oracle."""
    a = PrefillRun("qwen3_8b_prefill", 6, n, Hq=Hq, Hkv=Hkv, D=D, W=W, chunk=chunk, scale_bits=sb)
    b = PrefillRun("qwen3_8b_prefill", 6, n, Hq=Hq, Hkv=Hkv, D=D, W=W, chunk=chunk, scale_bits=sb,
                   cached=True)
    assert a.snap.keys() == b.snap.keys()
    for p in a.snap:
        np.testing.assert_array_equal(a.snap[p]["out"], b.snap[p]["out"])
    last = max(b.snap)
    b.check(last, _rows(b.snap[last]["C"], range(0, Hq, 5), step=29))


@pytest.mark.parametrize("Hq,Hkv,D,n,chunk,W,sb,cached,vb", [(32, 8, 128, 1400, 512, 256, 32, True, 4),
                                                            (8, 8, 64, 700, 256, 128, 32, False, 4),
                                                            (16, 2, 128, 900, 300, 256, 16, True, 4),
                                                            (32, 8, 128, 1400, 512, 256, 32, True, 3),
                                                            (8, 8, 64, 700, 256, 128, 16, False, 3)])
def test_prefill_v4_records(Hq, Hkv, D, n, chunk, W, sb, cached, vb):
    """Chunked prefill over k4v4 records (4-bit value codes, two channels per
    byte) and k4v3 records (3-bit codes straddling bytes), with fp32 or f16
    scale fields, cached or per-chunk images."""
    run = PrefillRun("qwen3_8b_prefill", 7, n, Hq=Hq, Hkv=Hkv, D=D, W=W, chunk=chunk,
                     scale_bits=sb, v_bits=vb, cached=cached)
    for p in run.snap:
        run.check(p, _rows(run.snap[p]["C"], range(0, Hq, 3), step=23))


@pytest.mark.parametrize("Hq,Hkv,n,chunk,W,sb,vb,cached", [
    (16, 4, 1400, 512, 256, 32, 2, False),   # the batched-decode head shape: 10 tiles + window
    (16, 4, 1400, 512, 256, 32, 2, True),
    (16, 2, 700, 256, 256, 16, 2, True),     # GQA group 8, f16 scales
    (4, 4, 450, 100, 128, 32, 4, False),     # group 1, k4v4, ragged chunks, window wraps
    (8, 4, 700, 256, 256, 32, 3, True),      # k4v3 records
    (32, 8, 1100, 512, 256, 32, 2, False),   # 128 row blocks: no key split
])
def test_prefill_head_dim_256(Hq, Hkv, n, chunk, W, sb, vb, cached):
    """head_dim 256: keys stream through the attention kernel in 64-key
    sub-blocks, the rotations pair two threads per row; grids of at most
    half the SMs split each row block's keys over a two-CTA cluster."""
    run = PrefillRun("batched_d256_decode", 8, n, Hq=Hq, Hkv=Hkv, D=256, W=W, chunk=chunk,
                     scale_bits=sb, v_bits=vb, cached=cached)
    for p in run.snap:
        run.check(p, _rows(run.snap[p]["C"], range(0, Hq, 3), step=17))


def test_prefill_head_dim_256_chunk_of_one_equals_decode():
    """A one-token chunk at head_dim 256 is a decode step over the same cache."""
    n = 128 * 2 + 40
    run = PrefillRun("batched_d256_decode", 9, n, Hq=8, Hkv=2, D=256, W=128, chunk=1, keep=[n - 1])
    s = run.snap[n - 1]
    dev = torch.device("cuda:0")
    q = torch.from_numpy(run.q[n - 1:n]).to(dev)
    dec = kvarn.decode_attention(q, run.tiles, run.table[None], torch.tensor([s["n_tiles"]],
                                 dtype=torch.int32, device=dev),
                                 torch.from_numpy(s["win_k"])[None].to(dev),
                                 torch.from_numpy(s["win_v"])[None].to(dev),
                                 torch.tensor([s["start"]], dtype=torch.int32, device=dev),
                                 torch.tensor([s["length"]], dtype=torch.int32, device=dev),
                                 run.lay).cpu().numpy()
    for h in range(8):
        assert rel_l2(s["out"][0, h], dec[0, h].astype(np.float64)) <= 2e-4
    run.check(n - 1, [(0, h) for h in range(8)])


def test_prefill_repeat_is_bit_identical():
    """The same 6,000-token prompt twice: every chunk's output is bit-identical
    (the warp roles hand off through barriers only; nothing depends on timing)."""
    a = PrefillRun("qwen3_8b_prefill", 10, 6000, Hq=32, Hkv=8, D=128, cached=True)
    b = PrefillRun("qwen3_8b_prefill", 10, 6000, Hq=32, Hkv=8, D=128, cached=True)
    for p in a.snap:
        np.testing.assert_array_equal(a.snap[p]["out"], b.snap[p]["out"])
    last = max(a.snap)
    a.check(last, _rows(a.snap[last]["C"], (0, 7, 30), step=41))


@pytest.mark.parametrize("Hq,Hkv,D,n,chunk,W", [(32, 8, 128, 1400, 512, 256), (16, 4, 256, 1100, 512, 256)])
def test_prefill_graph_replay_matches_direct_call(Hq, Hkv, D, n, chunk, W):
    """A prefill call captured in a CUDA graph (its attention kernel a
    programmatic dependent of its dequantisation grid; at head_dim 256 also a
    two-CTA cluster) replays to the direct call's output bit for bit: with
    every block converted, with only the window blocks converted, and with
    nothing to convert (a one-token chunk at the last tile position: no
    dequantisation grid in front, a plain launch)."""
    run = PrefillRun("qwen3_8b_prefill", 11, n, Hq=Hq, Hkv=Hkv, D=D, W=W, chunk=chunk)
    last = max(run.snap)
    s = run.snap[last]
    dev = torch.device("cuda:0")
    q_last = torch.from_numpy(run.q[last:last + s["C"]]).to(dev)
    p_tile = 128 * s["n_tiles"] - 1
    q_tile = torch.from_numpy(run.q[p_tile:p_tile + 1]).to(dev)
    wk = torch.from_numpy(s["win_k"]).to(dev)
    wv = torch.from_numpy(s["win_v"]).to(dev)
    cap = wk.shape[1]
    ws_blocks = s["n_tiles"] + cap // 128
    ws = torch.empty(kvarn.prefill_workspace_bytes(s["n_tiles"], cap, Hkv, D), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.Stream(device=dev)

    def call(q, pos0, out, cached):
        return kvarn.prefill_attention(q, pos0, run.tiles, run.table, s["n_tiles"], wk, wv,
                                       s["start"], s["length"], run.lay, ws=ws, out=out,
                                       ws_blocks=ws_blocks, cached_tiles=cached)

    for q, pos0, cached in [(q_last, last, 0), (q_last, last, s["n_tiles"]),
                            (q_tile, p_tile, s["n_tiles"])]:
        direct = torch.full(q.shape, float("nan"), device=dev)
        replay = torch.full(q.shape, float("nan"), device=dev)
        with torch.cuda.stream(stream):
            call(q, pos0, direct, 0)  # every image rebuilt: the reference output
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                call(q, pos0, replay, cached)
            g.replay()
        torch.cuda.synchronize()
        assert torch.equal(direct, replay), f"pos0={pos0} cached={cached}: graph replay differs"
        if pos0 == last:
            np.testing.assert_array_equal(replay.cpu().numpy(), s["out"])
