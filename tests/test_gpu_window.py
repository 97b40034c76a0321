"""Query rotation and window append on the GPU; the cache state machine run
through the C ABI against the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_quantization_token_gb300 import kvarn, synth
from tests.kvarn_helpers import compare_record

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("D", [64, 128, 256])
def test_rotate_query_matches_oracle(D):
    q = synth.queries("qwen3_8b_decode", 0, (3, 5, D))
    got = kvarn.rotate_query(torch.from_numpy(q).to(DEV)).cpu().numpy()
    want = oracle.wht_rows(q.reshape(-1, D).astype(np.float64)).reshape(q.shape)
    assert np.max(np.abs(got - want)) <= 1e-5 * np.max(np.abs(want))
    t = torch.from_numpy(q).to(DEV)
    kvarn.rotate_query(t, out=t)  # in place
    assert torch.equal(t.cpu(), torch.from_numpy(got))


def test_append_window_ring_slots():
    D, hkv, cap = 128, 2, 256
    k = torch.randn(2, 5, hkv, D, device=DEV)
    v = torch.randn(2, 5, hkv, D, device=DEV)
    wk = torch.zeros(2, hkv, cap, D, device=DEV)
    wv = torch.zeros_like(wk)
    start = torch.tensor([128, 0], dtype=torch.int32, device=DEV)
    length = torch.tensor([126, 3], dtype=torch.int32, device=DEV)
    kvarn.append_window(k, v, wk, wv, start, length)
    for s, (st, ln) in enumerate(((128, 126), (0, 3))):
        for i in range(5):
            slot = (st + ln + i) % cap
            assert torch.equal(wk[s, :, slot], k[s, i]) and torch.equal(wv[s, :, slot], v[s, i])
    assert int((wk != 0).any(-1).sum()) == 2 * 5 * hkv


@pytest.mark.parametrize("W,chunk", [(128, 1), (128, 200), (256, 512), (256, 37)])
def test_state_machine_through_the_abi(W, chunk):
    """append -> promote -> (attend) over a 700-token stream: GPU tiles equal
    the oracle state machine's within the rounding band, for any chunking."""
    D, hkv, n = 64, 2, 700
    cap = 128 * ((W + chunk + 127) // 128)
    ks, vs = synth.kv_layer("single_tile", 11, hkv, n, D)
    lay = kvarn.layout(D)
    rb = lay.record_bytes
    wk = torch.zeros(1, hkv, cap, D, device=DEV)
    wv = torch.zeros_like(wk)
    start, length = 0, 0
    tiles = torch.zeros(hkv * 8 * rb, dtype=torch.uint8, device=DEV)
    n_tiles = 0
    sm = oracle.CacheStateMachine(hkv, D, W=W)
    for i0 in range(0, n, chunk):
        kn = ks[:, i0:i0 + chunk].transpose(1, 0, 2)
        vn = vs[:, i0:i0 + chunk].transpose(1, 0, 2)
        m = kn.shape[0]
        kvarn.append_window(torch.from_numpy(np.ascontiguousarray(kn[None])).to(DEV),
                            torch.from_numpy(np.ascontiguousarray(vn[None])).to(DEV), wk, wv,
                            torch.tensor([start], dtype=torch.int32, device=DEV),
                            torch.tensor([length], dtype=torch.int32, device=DEV))
        length += m
        sm.append(kn, vn)
        while length >= W:
            rows = wk.view(hkv * cap, D)
            src = torch.tensor([h * cap + start for h in range(hkv)], dtype=torch.int64, device=DEV)
            dst = torch.tensor([(n_tiles * hkv + h) * rb for h in range(hkv)], dtype=torch.int64,
                               device=DEV)
            kvarn.compress_tile(rows, wv.view(hkv * cap, D), src, tiles, dst, lay)
            n_tiles += 1
            start = (start + 128) % cap
            length -= 128
    assert n_tiles == sm.n_tiles
    host = tiles.cpu().numpy()
    for t in range(n_tiles):
        for h in range(hkv):
            o = (t * hkv + h) * rb
            t0 = 128 * t
            ref = oracle.compress_unit(ks[h, t0:t0 + 128], vs[h, t0:t0 + 128])
            compare_record(host[o:o + rb], ref, D)
