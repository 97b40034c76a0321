"""Decode under the three launch modes (the launch_flags argument of each
call) gives bit-identical results, eagerly and inside a captured CUDA graph;
and a captured decode step replayed across promotion boundaries (promotion
hoisted out of the graph, as the pages' CUDA-graph decode loop does) matches
the direct path bit for bit at every step, and the fp64 oracle within 1e-4."""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_quantization_token_gb300 import kvarn, synth
from tests.kvarn_helpers import ATTN_RTOL, Cache, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MODES = [0, kvarn.LAUNCH_PDL, kvarn.LAUNCH_PDL | kvarn.LAUNCH_PREFETCH]


def _layers(n_layers=3):
    caches = [Cache("qwen3_8b_decode", 30 + l, [128 * 9 + 70, 128 * 4 + 5], Hkv=8, D=128)
              for l in range(n_layers)]
    qs = [torch.from_numpy(synth.queries("qwen3_8b_decode", 30 + l, (2, 32, 128))).to(DEV)
          for l in range(n_layers)]
    kn = [torch.from_numpy(synth.queries("qwen3_8b_decode", 60 + l, (2, 1, 8, 128))).to(DEV)
          for l in range(n_layers)]
    return caches, qs, kn


def _step(caches, qs, kn, outs, ws, mode):
    # per layer: attend, then append the layer's next token (as a decode loop does)
    for c, q, k, o in zip(caches, qs, kn, outs):
        kvarn.decode_split(q, c.tiles, c.tile_table, c.n_tiles, c.win_k, c.win_v, c.win_start,
                           c.win_len, c.lay, ws, flags=mode)
        kvarn.decode_combine(ws, o, c.Hkv, c.max_tiles, c.cap, flags=mode)
        kvarn.append_window(k, k, c.win_k, c.win_v, c.win_start, c.win_len, flags=mode)


def _run(mode, graph):
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
            _step(caches, qs, kn, outs, ws, mode)
        g.replay()
    else:
        with torch.cuda.stream(stream):
            _step(caches, qs, kn, outs, ws, mode)
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
    c = Cache("qwen3_8b_decode", 40, [128 * 6 + 30], Hkv=8, D=128)
    q = synth.queries("qwen3_8b_decode", 40, (1, 32, 128))
    out = c.decode(torch.from_numpy(q).to(DEV), flags=kvarn.LAUNCH_PDL | kvarn.LAUNCH_PREFETCH)
    out = out.cpu().numpy()
    ref = c.oracle_decode(q)
    for h in range(32):
        assert rel_l2(out[0, h], ref[(0, h)]) < ATTN_RTOL, h


class _DecodeState:
    """Caches of L layers and B sequences with room for the tiles that later
    promotions add: packed pool, per-layer tile tables, FP32 rings of W = 128
    slots, and the host's copy of each sequence's window bookkeeping."""

    L, B, HQ, HKV, D, CAP = 3, 2, 32, 8, 128, 128

    def __init__(self, ctxs, spare_tiles=4, seed=70):
        L, B, HKV, D, CAP = self.L, self.B, self.HKV, self.D, self.CAP
        self.lay = kvarn.layout(D)
        rb = self.rb = self.lay.record_bytes
        self.nt = [c // 128 for c in ctxs]          # windows of ctx % 128 tokens (< W)
        self.wl = [c % 128 for c in ctxs]
        self.max_tiles = max(self.nt) + spare_tiles
        units = L * B * HKV * self.max_tiles
        self.tiles = torch.zeros(units * rb, dtype=torch.uint8, device=DEV)
        tab = np.arange(units, dtype=np.int64).reshape(L, B, HKV, self.max_tiles) * rb
        self.table = torch.from_numpy(tab).to(DEV)
        self.win_k = torch.zeros(L, B, HKV, CAP, D, device=DEV)
        self.win_v = torch.zeros_like(self.win_k)
        for l in range(L):
            for b in range(B):
                k, v = synth.kv_layer("qwen3_8b_decode", seed + 37 * l + 1000 * b, HKV, ctxs[b], D)
                src = np.arange(HKV)[:, None] * ctxs[b] + 128 * np.arange(self.nt[b])[None, :]
                kvarn.compress_tile(torch.from_numpy(k.reshape(-1, D)).to(DEV),
                                    torch.from_numpy(v.reshape(-1, D)).to(DEV),
                                    torch.from_numpy(src.reshape(-1)).to(DEV), self.tiles,
                                    self.table[l, b, :, :self.nt[b]].contiguous().view(-1), self.lay)
                self.win_k[l, b, :, :self.wl[b]] = torch.from_numpy(k[:, 128 * self.nt[b]:]).to(DEV)
                self.win_v[l, b, :, :self.wl[b]] = torch.from_numpy(v[:, 128 * self.nt[b]:]).to(DEV)
        self.win_start = torch.zeros(B, dtype=torch.int32, device=DEV)
        self.win_len = torch.tensor(self.wl, dtype=torch.int32, device=DEV)
        self.n_tiles = torch.tensor(self.nt, dtype=torch.int32, device=DEV)
        self.host_start = [0] * B
        self.ws = torch.zeros(kvarn.decode_workspace_bytes(B, self.HQ, HKV, D, self.max_tiles, CAP),
                              dtype=torch.uint8, device=DEV)
        self.q = torch.empty(L, B, self.HQ, D, device=DEV)
        self.kn = torch.empty(L, B, 1, HKV, D, device=DEV)
        self.out = torch.empty(L, B, self.HQ, D, device=DEV)
        torch.cuda.synchronize()

    def step(self, flags):
        """One decode token through the L layers: attend, append the layer's
        new row (into a slot this step's attention does not read), then one
        window advance of every sequence by that token."""
        for l in range(self.L):
            kvarn.decode_attention(self.q[l], self.tiles, self.table[l], self.n_tiles,
                                   self.win_k[l], self.win_v[l], self.win_start, self.win_len,
                                   self.lay, ws=self.ws, out=self.out[l], flags=flags)
            kvarn.append_window(self.kn[l], self.kn[l], self.win_k[l], self.win_v[l],
                                self.win_start, self.win_len, flags=flags)
        kvarn.window_advance(self.win_start, self.win_len, None, 1, 0, self.CAP, flags=flags)

    def promote_due(self):
        """Outside the step: every sequence whose window reached W = 128 turns
        its oldest 128 rows into the next tile of every layer and KV head."""
        promoted = []
        for b in range(self.B):
            self.wl[b] += 1
            if self.wl[b] < 128:
                continue
            for l in range(self.L):
                src = torch.tensor([(b * self.HKV + h) * self.CAP + self.host_start[b]
                                    for h in range(self.HKV)], dtype=torch.int64, device=DEV)
                dst = self.table[l, b, :, self.nt[b]].contiguous()
                kvarn.compress_tile(self.win_k[l].view(-1, self.D), self.win_v[l].view(-1, self.D),
                                    src, self.tiles, dst, self.lay)
            kvarn.window_advance(self.win_start[b:b + 1], self.win_len[b:b + 1],
                                 self.n_tiles[b:b + 1], 0, 1, self.CAP)
            self.host_start[b] = (self.host_start[b] + 128) % self.CAP
            self.nt[b] += 1
            self.wl[b] -= 128
            promoted.append(b)
        return promoted


def test_graph_replay_matches_direct_path_across_promotions():
    """The captured step (programmatic dependent launch with record prefetch)
    and the same step enqueued directly (plain launches) agree bit for bit on
    every output of every step, before and after each sequence's window
    crosses 128 tokens and is promoted into a tile."""
    ctxs = [128 * 5 + 124, 128 * 3 + 126]
    torch.cuda.synchronize()
    kvarn.device_error(clear=True)
    eager, graphed = _DecodeState(ctxs), _DecodeState(ctxs)
    fast = kvarn.LAUNCH_PDL | kvarn.LAUNCH_PREFETCH
    graphed.kn.zero_()
    graphed.q.zero_()
    graphed.step(fast)  # function attributes and symbol lookups outside capture
    torch.cuda.synchronize()
    # undo that warm-up step on the graphed copy (its appended row lies past the
    # window and is overwritten by the next append)
    graphed.win_len.copy_(eager.win_len)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        graphed.step(fast)
    torch.cuda.synchronize()
    promotions, oracle_checked = [], False
    for s in range(8):
        q = torch.from_numpy(synth.queries("qwen3_8b_decode", 200 + s, (3, 2, 32, 128))).to(DEV)
        kn = torch.from_numpy(synth.queries("qwen3_8b_decode", 300 + s, (3, 2, 1, 8, 128))).to(DEV)
        for st in (eager, graphed):
            st.q.copy_(q)
            st.kn.copy_(kn)
        eager.step(0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(eager.out, graphed.out), f"step {s}: graph replay differs from direct"
        assert torch.isfinite(eager.out).all()
        if promotions and not oracle_checked:  # the first step after a promotion, layer 0
            # the step attended over the cache before its own append: the window
            # without its last row
            pool = eager.tiles.cpu().numpy()
            ref = oracle.decode_attention(
                q[0].cpu().numpy(), pool, eager.table[0].cpu().numpy(), eager.n_tiles.cpu().numpy(),
                eager.win_k[0].cpu().numpy(), eager.win_v[0].cpu().numpy(),
                eager.win_start.cpu().numpy(), eager.win_len.cpu().numpy() - 1, 128 ** -0.5,
                heads=[(b, h) for b in range(2) for h in (0, 11, 31)])
            got = eager.out[0].cpu().numpy()
            for (b, h), r in ref.items():
                assert rel_l2(got[b, h], r) <= ATTN_RTOL, (s, b, h)
            oracle_checked = True
        pe = eager.promote_due()
        pg = graphed.promote_due()
        assert pe == pg
        promotions += [(s, b) for b in pe]
        torch.cuda.synchronize()
        assert torch.equal(eager.n_tiles, graphed.n_tiles)
        assert torch.equal(eager.win_len, graphed.win_len)
    assert {b for _, b in promotions} == {0, 1}, promotions  # both sequences crossed a boundary
    assert oracle_checked
    assert kvarn.device_error() == 0
