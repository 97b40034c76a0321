"""Helpers shared by the GPU parity tests: seeded caches built through the
C ABI, and comparisons of GPU results against the fp64 oracle.

Tolerances (stated for this method): packed codes bit-exact except where the
oracle's pre-rounding value lies within 1e-5 of a rounding boundary (counted
and reported); scales within 1e-6 relative (the offset lo relative to
max(|lo|, delta, RMS of the normalised tile)); attention within 1e-4 relative
L2 of the fp64 oracle evaluated on the GPU's own records.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from kv_cache_quantization_token_gb300 import kvarn, synth

BAND = 1e-5
SCALE_RTOL = 1e-6
ATTN_RTOL = 1e-4
TILE = 128


def band_mask(vpre: np.ndarray) -> np.ndarray:
    frac = vpre - np.floor(vpre)
    return np.abs(frac - 0.5) < BAND


def compare_record(gpu_rec: np.ndarray, ref: dict, D: int, v_bits: int = 2) -> dict:
    """Compare one GPU record with oracle.compress_unit output. Returns counts;
    raises AssertionError when a tolerance is broken."""
    g = oracle.unpack_record(gpu_rec, D, v_bits=v_bits)
    r = oracle.unpack_record(ref["record"], D, v_bits=v_bits)
    stats = {"band_flips": 0, "codes": 0}
    for t in ("k", "v"):
        diff = g[f"{t}_codes"] != r[f"{t}_codes"]
        band = band_mask(ref[f"{t}_vpre"])
        outside = diff & ~band
        assert not outside.any(), (
            f"{t} codes differ outside the rounding band at {np.argwhere(outside)[:5].tolist()}; "
            f"vpre={ref[f'{t}_vpre'][outside][:5]}")
        assert np.all(np.abs(g[f"{t}_codes"].astype(int) - r[f"{t}_codes"]) <= 1)
        stats["band_flips"] += int(diff.sum())
        stats["codes"] += diff.size
    gv = D // min(D, 128)
    pairs = [("k_s", ref["k_s"]), ("k_r", ref["k_r"]), ("k_delta", ref["k_delta"]),
             ("v_s", ref["v_s"]), ("v_r", ref["v_r"]), ("v_delta", ref["v_delta"])]
    worst = 0.0
    for name, want in pairs:
        got = g[name]
        err = np.abs(got - want) / np.maximum(np.abs(want), 1e-30)
        err[(want == 0) & (got == 0)] = 0.0
        worst = max(worst, float(err.max()))
        assert err.max() <= SCALE_RTOL, f"{name} rel err {err.max():.3e}"
    # The offset lo sits in the normalised domain, whose rows have unit std;
    # a constant group (delta = 0) can put lo at a near-zero Walsh coefficient,
    # so lo is compared relative to max(|lo|, delta, RMS of the normalised tile).
    k_norm = ref["k_delta"][None, :] * ref["k_vpre"] + ref["k_lo"][None, :]
    vd = np.repeat(ref["v_delta"].reshape(128, gv), D // gv, axis=1)
    vl = np.repeat(ref["v_lo"].reshape(128, gv), D // gv, axis=1)
    v_norm = vd * ref["v_vpre"] + vl
    for name, want, delta, norm in (("k_lo", ref["k_lo"], ref["k_delta"], k_norm),
                                    ("v_lo", ref["v_lo"], ref["v_delta"], v_norm)):
        got = g[name]
        rms = float(np.sqrt(np.mean(norm ** 2)))
        den = np.maximum(np.maximum(np.abs(want), np.abs(delta)), max(rms, 1e-30))
        err = np.abs(got - want) / den
        err[(want == 0) & (got == 0)] = 0.0
        worst = max(worst, float(err.max()))
        assert err.max() <= SCALE_RTOL, f"{name} rel err {err.max():.3e}"
    stats["scale_rel_err"] = worst
    return stats


def compare_record_f16(gpu_rec: np.ndarray, ref: dict, D: int, v_bits: int = 2) -> dict:
    """Compare a GPU record of the f16-scale layout with
    oracle.compress_unit(..., scale_bits=16). Codes as in compare_record. Each
    stored scale is binary16 rounded from the kernel's fp32 value, the
    oracle's from fp64: they must be equal, except where the fp64 value lies
    within 1e-6 (relative) of the midpoint between two binary16 neighbours,
    where one ulp apart is allowed (counted and returned)."""
    g = oracle.unpack_record(gpu_rec, D, 16, v_bits)
    r = oracle.unpack_record(ref["record"], D, 16, v_bits)
    stats = {"band_flips": 0, "codes": 0, "scale_flips": 0}
    for t in ("k", "v"):
        diff = g[f"{t}_codes"] != r[f"{t}_codes"]
        band = band_mask(ref[f"{t}_vpre"])
        assert not (diff & ~band).any(), f"{t} codes differ outside the rounding band"
        stats["band_flips"] += int(diff.sum())
        stats["codes"] += diff.size
    for name in ("k_delta", "k_lo", "k_s", "k_r", "v_delta", "v_lo", "v_r", "v_s"):
        got, want, exact = g[name], r[name], np.asarray(ref[name], np.float64)
        ne = got != want
        if ne.any():
            gb = got[ne].astype(np.float16).view(np.uint16).astype(np.int32)
            wb = want[ne].astype(np.float16).view(np.uint16).astype(np.int32)
            assert np.all(np.abs(gb - wb) == 1), f"{name}: stored binary16 values more than 1 ulp apart"
            mid = (got[ne] + want[ne]) / 2
            assert np.all(np.abs(exact[ne] - mid) <= 1e-6 * np.abs(mid)), (
                f"{name}: binary16 values differ away from a rounding midpoint")
            stats["scale_flips"] += int(ne.sum())
    return stats


def n_tiles_for(ctx: int, W: int) -> int:
    """Promotion rule: while the window holds >= W tokens, promote 128."""
    return 0 if ctx < W else (ctx - W) // TILE + 1


class Cache:
    """A batch of KVarN caches built on the GPU through the C ABI."""

    def __init__(self, workload, layer, ctxs, Hkv, D, W=128, cap=None, win_start=None, dev="cuda:0",
                 iters=4, scale_bits=32, v_bits=2):
        self.workload, self.layer, self.Hkv, self.D, self.W = workload, layer, Hkv, D, W
        self.dev = torch.device(dev)
        self.B = len(ctxs)
        self.ctxs = list(ctxs)
        self.scale_bits, self.v_bits = scale_bits, v_bits
        self.lay = kvarn.layout(D, iters, scale_bits, v_bits)
        self.rb = self.lay.record_bytes
        self.nt = [n_tiles_for(c, W) for c in ctxs]
        self.max_tiles = max(max(self.nt), 1)
        self.wl = [c - TILE * n for c, n in zip(ctxs, self.nt)]
        self.cap = cap if cap is not None else max(W, TILE * ((max(self.wl) + TILE - 1) // TILE), TILE)
        starts = win_start if win_start is not None else [0] * self.B
        kv = [synth.kv_layer(workload, layer + 1000 * b, Hkv, c, D) for b, c in enumerate(ctxs)]
        self.k = [x[0] for x in kv]
        self.v = [x[1] for x in kv]
        # compress every full tile of every (sequence, head) in one launch
        rows, src0, dst, table = [], [], [], np.zeros((self.B, Hkv, self.max_tiles), np.int64)
        unit, row_base = 0, 0
        for b in range(self.B):
            for h in range(Hkv):
                rows.append((self.k[b][h], self.v[b][h]))
                for i in range(self.nt[b]):
                    src0.append(row_base + TILE * i)
                    dst.append(unit * self.rb)
                    table[b, h, i] = unit * self.rb
                    unit += 1
                row_base += ctxs[b]
        self.n_units = unit
        k_all = np.concatenate([r[0] for r in rows]) if rows else np.zeros((0, D), np.float32)
        v_all = np.concatenate([r[1] for r in rows]) if rows else np.zeros((0, D), np.float32)
        self.tiles = torch.zeros(max(unit, 1) * self.rb, dtype=torch.uint8, device=self.dev)
        if unit:
            kvarn.compress_tile(torch.from_numpy(k_all).to(self.dev),
                                torch.from_numpy(v_all).to(self.dev),
                                torch.tensor(src0, dtype=torch.int64, device=self.dev),
                                self.tiles, torch.tensor(dst, dtype=torch.int64, device=self.dev),
                                self.lay)
        self.tile_table = torch.from_numpy(table).to(self.dev)
        self.n_tiles = torch.tensor(self.nt, dtype=torch.int32, device=self.dev)
        # window: the not-yet-promoted tail of each sequence, written into the ring
        wk = np.zeros((self.B, Hkv, self.cap, D), np.float32)
        wv = np.zeros_like(wk)
        for b in range(self.B):
            for j in range(self.wl[b]):
                slot = (starts[b] + j) % self.cap
                wk[b, :, slot] = self.k[b][:, TILE * self.nt[b] + j]
                wv[b, :, slot] = self.v[b][:, TILE * self.nt[b] + j]
        self.win_k = torch.from_numpy(wk).to(self.dev)
        self.win_v = torch.from_numpy(wv).to(self.dev)
        self.win_start = torch.tensor(starts, dtype=torch.int32, device=self.dev)
        self.win_len = torch.tensor(self.wl, dtype=torch.int32, device=self.dev)
        self.starts = starts

    def decode(self, q, scale=None, **kw):
        return kvarn.decode_attention(q, self.tiles, self.tile_table, self.n_tiles, self.win_k,
                                      self.win_v, self.win_start, self.win_len, self.lay,
                                      softmax_scale=scale, **kw)

    def oracle_decode(self, q: np.ndarray, heads=None, scale=None):
        scale = self.D ** -0.5 if scale is None else scale
        return oracle.decode_attention(q, self.tiles.cpu().numpy(), self.tile_table.cpu().numpy(),
                                       self.nt, self.win_k.cpu().numpy(), self.win_v.cpu().numpy(),
                                       self.starts, self.wl, scale, heads=heads,
                                       scale_bits=self.scale_bits, v_bits=self.v_bits)


def rel_l2(got: np.ndarray, want: np.ndarray) -> float:
    den = np.linalg.norm(want)
    if den == 0:
        return float(np.linalg.norm(got))
    return float(np.linalg.norm(got.astype(np.float64) - want) / den)


PREFILL_RTOL = 1e-4  # tensor-core prefill: fp16 hi + lo operand pairs, fp32 accumulation


class PrefillRun:
    """A prompt streamed through the C ABI in chunks: append -> promote (while
    the window holds >= W tokens) -> chunked-prefill attention. Keeps, for the
    chunks listed in `keep`, a copy of the window and the outputs so the
    oracle can be evaluated on the same state."""

    def __init__(self, workload, layer, n_tokens, Hq, Hkv, D, W=256, chunk=512, keep=None,
                 dev="cuda:0", scale=None, scale_bits=32, cached=False, v_bits=2):
        dev = torch.device(dev)
        self.Hq, self.Hkv, self.D, self.W = Hq, Hkv, D, W
        self.k, self.v = synth.kv_layer(workload, layer, Hkv, n_tokens, D)
        self.q = synth.queries(workload, layer, (n_tokens, Hq, D))
        self.scale_bits, self.v_bits = scale_bits, v_bits
        self.lay = kvarn.layout(D, scale_bits=scale_bits, v_bits=v_bits)
        rb = self.rb = self.lay.record_bytes
        self.cap = cap = TILE * ((W - 1 + chunk + TILE - 1) // TILE)
        max_tiles = n_tokens // TILE + 1
        self.tiles = torch.zeros(Hkv * max_tiles * rb, dtype=torch.uint8, device=dev)
        table = (np.arange(Hkv)[:, None] * max_tiles + np.arange(max_tiles)[None, :]) * rb
        self.table = torch.from_numpy(table.astype(np.int64)).to(dev)
        win_k = torch.zeros(1, Hkv, cap, D, device=dev)
        win_v = torch.zeros_like(win_k)
        start, length, n_tiles = 0, 0, 0
        self.snap = {}
        # cached: one workspace for the whole prompt; each chunk converts only
        # the tiles promoted since the previous chunk
        ws_blocks = max_tiles + cap // TILE
        ws = (torch.empty(kvarn.prefill_workspace_bytes(max_tiles, cap, Hkv, D), dtype=torch.uint8,
                          device=dev) if cached else None)
        prev_tiles = 0
        keep = set(keep if keep is not None else range(0, n_tokens, chunk))
        for pos0 in range(0, n_tokens, chunk):
            C = min(chunk, n_tokens - pos0)
            kn = np.ascontiguousarray(self.k[:, pos0:pos0 + C].transpose(1, 0, 2))[None]
            vn = np.ascontiguousarray(self.v[:, pos0:pos0 + C].transpose(1, 0, 2))[None]
            kvarn.append_window(torch.from_numpy(kn).to(dev), torch.from_numpy(vn).to(dev),
                                win_k, win_v, torch.tensor([start], dtype=torch.int32, device=dev),
                                torch.tensor([length], dtype=torch.int32, device=dev))
            length += C
            while length >= W:
                src = torch.tensor([h * cap + start for h in range(Hkv)], dtype=torch.int64,
                                   device=dev)
                dst = self.table[:, n_tiles].contiguous()
                kvarn.compress_tile(win_k.view(-1, D), win_v.view(-1, D), src, self.tiles, dst,
                                    self.lay)
                n_tiles += 1
                start = (start + TILE) % cap
                length -= TILE
            qc = torch.from_numpy(self.q[pos0:pos0 + C]).to(dev)
            if cached:
                out = kvarn.prefill_attention(qc, pos0, self.tiles, self.table, n_tiles, win_k[0],
                                              win_v[0], start, length, self.lay, softmax_scale=scale,
                                              ws=ws, ws_blocks=ws_blocks, cached_tiles=prev_tiles)
                prev_tiles = n_tiles
            else:
                out = kvarn.prefill_attention(qc, pos0, self.tiles, self.table, n_tiles, win_k[0],
                                              win_v[0], start, length, self.lay, softmax_scale=scale)
            if pos0 in keep:
                self.snap[pos0] = dict(C=C, n_tiles=n_tiles, start=start, length=length,
                                       win_k=win_k[0].cpu().numpy(), win_v=win_v[0].cpu().numpy(),
                                       out=out.cpu().numpy())
        self.n_tiles = n_tiles
        self.scale = D ** -0.5 if scale is None else scale

    def check(self, pos0, rows):
        """rel-L2 per (i, h) of the chunk at pos0 against the oracle; returns the worst."""
        s = self.snap[pos0]
        pool = self.tiles.cpu().numpy()
        ref = oracle.prefill_attention(self.q[pos0:pos0 + s["C"]], pos0, pool,
                                       self.table.cpu().numpy(), s["n_tiles"], s["win_k"],
                                       s["win_v"], s["start"], s["length"], self.scale, rows=rows,
                                       scale_bits=self.scale_bits, v_bits=self.v_bits)
        worst = 0.0
        for (i, h), r in ref.items():
            e = rel_l2(s["out"][i, h], r)
            worst = max(worst, e)
            assert e <= PREFILL_RTOL, f"chunk {pos0} row {i} head {h}: rel-L2 {e:.3e}"
        return worst
