"""Device-side failure reporting: a kernel that gives up sets its bit in the
library's error word (read with kvarn_get_device_error), poisons or skips
what depends on it, and leaves the CUDA context usable. No case faults the
GPU: the bad inputs are refused by the kernels' own checks before any access,
and the wait that runs out waits on a barrier nothing completes, for a
bounded time."""
import numpy as np
import pytest
import torch

from kv_cache_quantization_token_gb300 import kvarn, synth
from tests.kvarn_helpers import ATTN_RTOL, Cache, PrefillRun, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _clear_word():
    torch.cuda.synchronize()
    kvarn.device_error(clear=True)
    yield
    torch.cuda.synchronize()
    kvarn.device_error(clear=True)


def _decode_ok(seed=90):
    """A small decode checked against the oracle: the context still works."""
    c = Cache("qwen3_8b_decode", seed, [128 * 3 + 9], Hkv=2, D=128)
    q = synth.queries("qwen3_8b_decode", seed, (1, 8, 128))
    out = c.decode(torch.from_numpy(q).to(DEV)).cpu().numpy()
    ref = c.oracle_decode(q)
    for (b, h), r in ref.items():
        assert rel_l2(out[b, h], r) <= ATTN_RTOL


def test_wait_that_runs_out_is_reported_and_the_context_survives():
    assert kvarn.device_error() == 0
    kvarn.selftest_bounded_wait(2000)  # 2 ms on a barrier nothing completes
    torch.cuda.synchronize()
    assert kvarn.device_error(clear=False) == kvarn.DEVERR_SELFTEST
    assert kvarn.device_error(clear=True) == kvarn.DEVERR_SELFTEST  # read, then cleared
    assert kvarn.device_error() == 0
    _decode_ok()
    assert kvarn.device_error() == 0


@pytest.mark.parametrize("bad", ["past_pool", "misaligned", "negative"])
def test_decode_refuses_a_table_entry_outside_the_pool(bad):
    c = Cache("qwen3_8b_decode", 91, [128 * 4 + 20, 128 * 2 + 3], Hkv=2, D=128)
    off = {"past_pool": c.tiles.numel(), "misaligned": 64, "negative": -128}[bad]
    c.tile_table[0, 1, 1] = off  # sequence 0, KV head 1, tile 1
    q = synth.queries("qwen3_8b_decode", 91, (2, 8, 128))
    out = c.decode(torch.from_numpy(q).to(DEV)).cpu().numpy()
    assert kvarn.device_error() == kvarn.DEVERR_RECORD
    assert np.isnan(out[0, 4:8]).all()            # the query heads of KV head 1
    assert np.isfinite(out[0, :4]).all() and np.isfinite(out[1]).all()
    _decode_ok(92)


def test_prefill_refuses_a_table_entry_outside_the_pool():
    run = PrefillRun("qwen3_8b_decode", 93, 700, Hq=8, Hkv=2, D=128, W=256, chunk=256, keep=[])
    assert kvarn.device_error() == 0
    table = run.table.clone()
    table[1, 0] = run.tiles.numel() - 64  # KV head 1, tile 0: runs past the pool
    s = 384  # positions 384..447 lie in the four tiles (no window needed)
    assert run.n_tiles == 4
    q = torch.from_numpy(run.q[s:s + 64]).to(DEV)
    win = torch.zeros(2, 512, 128, device=DEV)
    out = kvarn.prefill_attention(q, s, run.tiles, table, run.n_tiles, win, win, 0, 0,
                                  run.lay).cpu().numpy()
    assert kvarn.device_error() == kvarn.DEVERR_RECORD
    assert np.isnan(out[:, 4:8]).all() and np.isfinite(out[:, :4]).all()


def test_compress_skips_units_outside_its_buffers():
    lay = kvarn.layout(128)
    k, v = synth.kv_stream("single_tile", 0, 0, 256, 128)
    kd, vd = torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV)
    tiles = torch.zeros(2 * lay.record_bytes, dtype=torch.uint8, device=DEV)
    i64 = lambda xs: torch.tensor(xs, dtype=torch.int64, device=DEV)
    # unit 0 is fine; unit 1 would write past the pool; unit 2 would read past the rows
    kvarn.compress_tile(kd, vd, i64([0, 0, 129]), tiles,
                        i64([0, lay.record_bytes + 16, lay.record_bytes]), lay)
    torch.cuda.synchronize()
    assert kvarn.device_error() == kvarn.DEVERR_RECORD
    t = tiles.cpu().numpy()
    assert t[:lay.record_bytes].any() and not t[lay.record_bytes:].any()


def test_append_refuses_to_overfill_a_window():
    D, cap = 128, 128
    win_k = torch.zeros(2, 1, cap, D, device=DEV)
    win_v = torch.zeros_like(win_k)
    start = torch.zeros(2, dtype=torch.int32, device=DEV)
    length = torch.tensor([cap - 1, cap], dtype=torch.int32, device=DEV)  # sequence 1 is full
    new = torch.ones(2, 1, 1, D, device=DEV)
    kvarn.append_window(new, new, win_k, win_v, start, length)
    torch.cuda.synchronize()
    assert kvarn.device_error() == kvarn.DEVERR_WINDOW
    assert (win_k[0, 0, cap - 1] == 1).all()       # sequence 0 had room for its row
    assert not win_k[1].any()                      # sequence 1's ring is untouched
