"""The decode entry point for callers that cannot allocate device memory
(kvarn_decode_attention_noalloc) against the workspace entry point.

Such callers run where cudaMalloc is off limits (inside another runtime's
memory arena, or under a host framework that owns every allocation); the
entry point keeps its scratch in the library's own device memory instead.
This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

from kv_cache_quantization_token_gb300 import kvarn, synth
from tests.kvarn_helpers import ATTN_RTOL, Cache, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    c = Cache("qwen3_8b_decode", 21, [2000, 777], Hkv=8, D=128)
    for call in range(2):  # the scratch keeps the previous call's contents
        q = torch.from_numpy(synth.queries("qwen3_8b_decode", 40 + call, (2, 32, 128))).to(DEV)
        want = c.decode(q).cpu().numpy()
        got = kvarn.decode_attention_noalloc(q, c.tiles, c.tile_table, c.n_tiles, c.win_k,
                                             c.win_v, c.win_start, c.win_len, c.lay)
        got = got.cpu().numpy()
        for b in range(2):
            for h in range(32):
                assert rel_l2(got[b, h], want[b, h]) <= ATTN_RTOL


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lay = kvarn.layout(128)
    need = kvarn.decode_workspace_bytes(64, 32, 8, 128, 8192, 128)
    assert need > (16 << 20)
    p = ctypes.c_void_p(256)
    fn = kvarn._L().kvarn_decode_attention_noalloc
    rc = fn(p, p, 1 << 40, p, p, p, p, p, p, 128, 64, 32, 8, 128, 8192, ctypes.c_float(0.088),
            ctypes.byref(lay), p, 0, None)
    assert rc == -5  # KVARN_ERR_WORKSPACE, nothing enqueued
