#!/usr/bin/env python
"""KVarN hot-path benchmark on GB300: decode attention over the compressed
cache at 16k context, and bulk tile compression.

Decode step (the timed unit): one new token of a Qwen3-8B-like model (32 query
heads, 8 KV heads, head_dim 128, batch 1) through 36 layers, each layer with
its own 16k-token compressed cache (128 packed tiles per KV head plus the FP32
window): per layer the split-tile decode kernel and the LSE combine, and the
append of the layer's next K/V token into the window (on a forked stream: it
writes a slot no attention of the step reads); one device-side window advance
per step. The step is captured once as a CUDA graph and replayed, its kernels
chained by programmatic dependent launch.
Whenever the window reaches 128 tokens the oldest 128 are promoted (compressed
into a tile) between replays, as the decode loop of the pages does with its
promotion hoisted out of the graph.

After the decode timing the bulk compression of 32k-token 8B-like caches
(256 tiles x 8 KV heads = 2048 tile-heads per launch) is timed on its own.

Prints one JSON line (see the keys at the end of main()).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KVarN decode-attn tokens/s & HBM GB/s at 16k ctx; tile-compress tiles/s"
L2_BYTES = 129 * 1024 * 1024

# Decode workload: Qwen3-8B-like, batch 1, 32q/8kv heads, head_dim 128, 16k context
WORKLOAD, HQ, HKV, D, LAYERS, CTX0, W = "qwen3_8b_decode", 32, 8, 128, 36, 16384, 128
# Compress bulk workload: 32k-token caches of the same model, 8 KV heads
C_TILES, C_HEADS = 256, 8

# DRAM bytes per launch from an ncu capture, keyed by the kernel source they
# were measured on (None until captured; ignored once the source changes).
NCU_TRAFFIC = {
    # one split launch of the decode section (128 tiles x 8 KV heads + a
    # 124-token window, 17,809,408 algorithmic bytes): 17.88 MB read, nothing
    # written back within the launch. The bench's timed launches run at a
    # longer context, so the figure is scaled by their algorithmic bytes.
    "decode_split": {"src_sha": "cbd2a56274edd276", "bytes": 17877248, "algorithmic": 17809408},
    # one 2048-tile-head launch (the one the bench times): 268.51 MB read +
    # 17.58 MB written back within the launch
    "compress": {"src_sha": "c4499b18558919c0", "bytes": 286092032},
}


# launch flags of the timed decode calls: programmatic dependent launch with
# record prefetch (nothing inside a step writes records, tables or tile counts;
# promotions run between steps)
FAST = 3  # KVARN_LAUNCH_PDL | KVARN_LAUNCH_PREFETCH


def src_sha(name: str) -> str:
    with open(os.path.join(ROOT, "kv_cache_quantization_token_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx, self.proc, self.lines = gpu_index, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        return self.summarize(self.lines)

    @staticmethod
    def summarize(lines):
        """Median SM clock, the maximum clock and the throttle reasons seen
        active, from nvidia-smi csv lines in FIELDS order (others skipped)."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
class OracleDecodeSample:
    """The fp64 oracle (as it stands) on a bounded sample of the decode step:
    layer 0's 8 KV heads, each over its first `n_tiles` tiles, every query
    head of the KV head's group, on host threads (the oracle's C code
    releases the GIL). Its inputs are the oracle's own compressed tiles."""

    def __init__(self, n_tiles: int, threads: int = 0):
        import oracle
        from concurrent.futures import ThreadPoolExecutor
        from kv_cache_quantization_token_gb300 import synth
        self.oracle, self.n_tiles = oracle, n_tiles
        self.threads = threads or max(1, min(len(os.sched_getaffinity(0)), HKV))
        self.pool = ThreadPoolExecutor(self.threads)
        rb = oracle.record_bytes(D)
        self.table = (np.arange(n_tiles, dtype=np.int64) * rb)[None, None, :]
        self.q = synth.queries(WORKLOAD, 0, (1, HQ, D))
        n_tok = 128 * n_tiles

        def setup(h):
            k, v = synth.kv_stream(WORKLOAD, 0, h, n_tok, D)
            return np.concatenate([oracle.compress_unit(k[128 * i:128 * i + 128],
                                                        v[128 * i:128 * i + 128])["record"]
                                   for i in range(n_tiles)])
        self.recs = list(self.pool.map(setup, range(HKV)))
        self.sample = (f"layer 0 of {LAYERS}: {HKV} KV heads x {HQ // HKV} query heads over "
                       f"{n_tok} of {CTX0} tokens, scaled to the full step")

    def _head(self, h):
        G = HQ // HKV
        wk = np.zeros((1, 1, 128, D), np.float32)
        return self.oracle.decode_attention(self.q[:, h * G:(h + 1) * G], self.recs[h], self.table,
                                            [self.n_tiles], wk, wk, [0], [0], D ** -0.5,
                                            heads=[(0, g) for g in range(G)])

    def run(self) -> float:
        """Seconds of one sample; tokens/s of the full step = 1 / (that x scale)."""
        t0 = time.perf_counter()
        list(self.pool.map(self._head, range(HKV)))
        return time.perf_counter() - t0

    @property
    def scale(self) -> float:
        return LAYERS * CTX0 / (128.0 * self.n_tiles)


def oracle_compress_baseline(sample: dict) -> dict:
    """The oracle's tile compression timed on host threads (1 and all cores)
    over the first units of the bulk-compress input, and the GPU records of
    the same units compared with the oracle's: codes that differ, of which
    inside the rounding band (|frac(v) - 1/2| < 1e-5 of the oracle's
    pre-rounding value v) and outside it, and the largest relative scale
    difference. The oracle's codes are exact only up to that band."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    k, v, recs, rb = sample["k"], sample["v"], sample["records"], sample["record_bytes"]
    n = k.shape[0] // 128
    unit = lambda u: oracle.compress_unit(k[128 * u:128 * u + 128], v[128 * u:128 * u + 128])
    t0 = time.perf_counter()
    for u in range(4):
        unit(u)
    t1 = (time.perf_counter() - t0) / 4
    cores = max(1, len(os.sched_getaffinity(0)))
    with ThreadPoolExecutor(cores) as pool:
        t0 = time.perf_counter()
        refs = list(pool.map(unit, range(n)))
        tn = (time.perf_counter() - t0) / n
    codes = differ = in_band = outside = 0
    worst = 0.0
    # the offsets lo: how many meet 1e-6 relative to |lo| itself, how many only
    # relative to max(|lo|, delta, RMS of the normalised tile) (the bound the
    # parity tests apply: a constant group can put lo at a near-zero Walsh
    # coefficient), and how many neither
    lo_n = lo_plain = lo_widened_only = lo_out = 0
    lo_worst = 0.0
    gv = D // min(D, 128)
    for u, ref in enumerate(refs):
        got = oracle.unpack_record(recs[u * rb:(u + 1) * rb], D)
        want = oracle.unpack_record(ref["record"], D)
        for t in ("k", "v"):
            d = got[f"{t}_codes"] != want[f"{t}_codes"]
            vpre = ref[f"{t}_vpre"]
            band = np.abs(vpre - np.floor(vpre) - 0.5) < 1e-5
            codes += d.size
            differ += int(d.sum())
            in_band += int((d & band).sum())
            outside += int((d & ~band).sum())
            for f in ("delta", "s", "r"):
                w = np.asarray(ref[f"{t}_{f}"], np.float64)
                g = got[f"{t}_{f}"].astype(np.float64)
                worst = max(worst, float(np.max(np.abs(g - w) / np.maximum(np.abs(w), 1e-30))))
            lw = np.asarray(ref[f"{t}_lo"], np.float64)
            dw = np.asarray(ref[f"{t}_delta"], np.float64)
            if t == "k":
                norm = dw[None, :] * vpre + lw[None, :]
            else:
                norm = (np.repeat(dw.reshape(128, gv), D // gv, axis=1) * vpre
                        + np.repeat(lw.reshape(128, gv), D // gv, axis=1))
            rms = float(np.sqrt(np.mean(norm ** 2)))
            diff = np.abs(got[f"{t}_lo"].astype(np.float64) - lw)
            plain = diff / np.maximum(np.abs(lw), 1e-30)
            wide = diff / np.maximum(np.maximum(np.abs(lw), np.abs(dw)), max(rms, 1e-30))
            plain[diff == 0] = 0.0
            wide[diff == 0] = 0.0
            lo_n += lw.size
            lo_plain += int((plain <= 1e-6).sum())
            lo_widened_only += int(((plain > 1e-6) & (wide <= 1e-6)).sum())
            lo_out += int((wide > 1e-6).sum())
            lo_worst = max(lo_worst, float(wide.max()))
    return {"oracle_tile_heads_per_s_1_core": 1.0 / t1,
            "oracle_tile_heads_per_s_all_cores": 1.0 / tn, "cores": cores,
            "sample": f"{n} tile-heads of the bulk-compress input (head_dim {D}); 4 on one thread",
            "gpu_vs_oracle": {"codes": codes, "differing": differ, "in_rounding_band": in_band,
                              "outside_rounding_band": outside,
                              "scale_rel_err_max": worst,
                              "lo": {"values": lo_n, "within_1e-6_of_lo": lo_plain,
                                     "within_1e-6_only_widened": lo_widened_only,
                                     "outside_1e-6": lo_out, "widened_rel_err_max": lo_worst},
                              "note": "GPU records of the same units, decoded by the oracle; "
                                      "delta, s and r compared relative to the oracle's value; "
                                      "lo relative to |lo|, and to max(|lo|, delta, RMS of "
                                      "the normalised tile)"}}


def oracle_prefill_baseline(rows_every: int = 16) -> dict:
    """The oracle's causal prefill attention timed on host threads over the
    last 512-token chunk of a 2,048-token prefix of the 8B-like prompt (32q/8kv,
    head_dim 128, W=256): every rows_every-th row, all 32 query heads, over
    tiles the oracle compressed itself; scaled by visible (query, key) pairs to
    the whole prefix's attention."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    from kv_cache_quantization_token_gb300 import synth
    n_tok, Wp, Hq, Hkv = 2048, 256, 32, 8
    k, v = synth.kv_layer("qwen3_8b_prefill", 0, Hkv, n_tok, D)
    q = synth.queries("qwen3_8b_prefill", 0, (n_tok, Hq, D))
    nt = (n_tok - Wp) // 128 + 1                       # tiles after the last promotion
    rb = oracle.record_bytes(D)
    cores = max(1, len(os.sched_getaffinity(0)))
    with ThreadPoolExecutor(cores) as pool:
        recs = list(pool.map(lambda hu: oracle.compress_unit(
            k[hu[0], 128 * hu[1]:128 * hu[1] + 128], v[hu[0], 128 * hu[1]:128 * hu[1] + 128])["record"],
            [(h, i) for h in range(Hkv) for i in range(nt)]))
    pool_b = np.concatenate(recs)
    table = (np.arange(Hkv)[:, None] * nt + np.arange(nt)[None, :]).astype(np.int64) * rb
    wl = n_tok - 128 * nt
    cap = 512
    wk = np.zeros((Hkv, cap, D), np.float32)
    wv = np.zeros_like(wk)
    wk[:, :wl] = k[:, 128 * nt:]
    wv[:, :wl] = v[:, 128 * nt:]
    pos0 = n_tok - 512
    rows = list(range(0, 512, rows_every))

    def one(i):
        return oracle.prefill_attention(q[pos0:pos0 + 512], pos0, pool_b, table, nt, wk, wv, 0, wl,
                                        D ** -0.5, rows=[(i, h) for h in range(Hq)])
    out = {}
    for label, workers in (("1_core", 1), ("all_cores", cores)):
        sample_rows = rows[:4] if workers == 1 else rows
        with ThreadPoolExecutor(workers) as pool:
            t0 = time.perf_counter()
            list(pool.map(one, sample_rows))
            sec = time.perf_counter() - t0
        pairs = sum(pos0 + i + 1 for i in sample_rows)
        total = n_tok * (n_tok + 1) // 2
        layer_s = sec * total / pairs
        out[f"prompt_tokens_per_s_one_layer_{label}"] = n_tok / layer_s
    out.update({"cores": cores, "sample": f"rows 0, {rows_every}, ... of positions {pos0}..{n_tok - 1} "
                                          f"(4 rows on one thread), all {Hq} query heads; scaled "
                                          f"by visible (query, key) pairs to the {n_tok}-token prefix"})
    return out


def reduce_timing(elapsed_ms, units_per_rank, world, device=None):
    """Max-over-ranks timing of a replica run (weak scaling: every rank
    processes units_per_rank in its own elapsed_ms). The job's time is the
    slowest rank's and its throughput the units of all ranks over that time;
    every rank gets the same pair. world 1: the rank's own numbers."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
        dist.barrier()
    return elapsed_ms, world * units_per_rank / (elapsed_ms / 1000.0)


def run_reference(args, rank):
    """--impl reference: the oracle timed on the host cores on this arm's metric,
    one bounded sample (every KV head of one layer over one tile) per step."""
    if rank != 0:
        return
    smp = OracleDecodeSample(1)
    for _ in range(args.warmup):
        smp.run()
    secs = [smp.run() for _ in range(args.steps)]
    value = 1.0 / (float(np.mean(secs)) * smp.scale)
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1000.0 * float(np.mean(secs)), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": workload_config(),
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": smp.threads,
                            "kind": "oracle", "sample": smp.sample},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_prefill_bench(dev, stream, lay, peaks, peak_kind, n_tok=15500, chunk=512, Wp=256, reps=3,
                      workload="qwen3_8b_prefill", hq=None, hkv=None, label="Qwen3-8B-like"):
    """One layer of a chunked prompt (by default the 15,500-token 8B-like one,
    32q/8kv, head_dim 128): per chunk append, promote, prefill
    attention (block dequantisation of the tiles promoted since the previous
    chunk and of the window blocks, into one workspace kept for the whole
    prompt, + tcgen05 attention). Reports prompt tokens/s
    of the attention path scaled to 36 layers, and the contraction throughput
    against the dense fp16 tensor peak (the algorithmic Q.K and P.V
    multiply-adds, counted once)."""
    import torch
    from kv_cache_quantization_token_gb300 import kvarn, synth
    HQ_, HKV_ = (hq or HQ), (hkv or HKV)
    D_ = lay.head_dim
    ks, vs = synth.kv_layer(workload, 0, HKV_, n_tok, D_)
    q = torch.from_numpy(synth.queries(workload, 0, (n_tok, HQ_, D_))).to(dev)
    kn_all = torch.from_numpy(np.ascontiguousarray(ks.transpose(1, 0, 2))).to(dev)  # [n][Hkv][D]
    vn_all = torch.from_numpy(np.ascontiguousarray(vs.transpose(1, 0, 2))).to(dev)
    rb = lay.record_bytes
    cap = 128 * ((Wp - 1 + chunk + 127) // 128)
    max_tiles = n_tok // 128 + 1
    tiles = torch.empty(HKV_ * max_tiles * rb, dtype=torch.uint8, device=dev)
    tab = (np.arange(HKV_)[:, None] * max_tiles + np.arange(max_tiles)[None, :]) * rb
    table = torch.from_numpy(tab.astype(np.int64)).to(dev)
    # promotions of one chunk go out as one compress launch: the (source row,
    # destination record) pairs of every due tile and KV head, prepared ahead
    # (the schedule depends only on the prompt length, the chunk size and W)
    prom = {}
    start = length = n_tiles = 0
    for pos0 in range(0, n_tok, chunk):
        length += min(chunk, n_tok - pos0)
        k = (length - Wp) // 128 + 1 if length >= Wp else 0
        if k:
            src = [h * cap + (start + 128 * i) % cap for i in range(k) for h in range(HKV_)]
            dst = [int(tab[h, n_tiles + i]) for i in range(k) for h in range(HKV_)]
            prom[pos0] = (k, torch.tensor(src, dtype=torch.int64, device=dev),
                          torch.tensor(dst, dtype=torch.int64, device=dev))
            start, length, n_tiles = (start + 128 * k) % cap, length - 128 * k, n_tiles + k
    win_k = torch.zeros(1, HKV_, cap, D_, device=dev)
    win_v = torch.zeros_like(win_k)
    ws_start = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_len = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_nt = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty(n_tok, HQ_, D_, device=dev)
    ws_p = torch.empty(kvarn.prefill_workspace_bytes(max_tiles, cap, HKV_, D_), dtype=torch.uint8,
                       device=dev)
    ev = []

    ws_blocks = max_tiles + cap // 128  # one image workspace for the whole prompt

    def prompt(record):
        start = length = n_tiles = 0
        prev_tiles = 0  # tiles whose operand images the workspace already holds
        ws_start.zero_()
        ws_len.zero_()
        ws_nt.zero_()
        for pos0 in range(0, n_tok, chunk):
            C = min(chunk, n_tok - pos0)
            kvarn.append_window(kn_all[pos0:pos0 + C][None], vn_all[pos0:pos0 + C][None],
                                win_k, win_v, ws_start, ws_len)
            length += C
            k = 0
            if pos0 in prom:  # promote: while the window holds >= W tokens, its oldest 128
                k, psrc, pdst = prom[pos0]
                kvarn.compress_tile(win_k.view(-1, D_), win_v.view(-1, D_), psrc, tiles, pdst, lay)
                n_tiles += k
                start = (start + 128 * k) % cap
                length -= 128 * k
            kvarn.window_advance(ws_start, ws_len, ws_nt, C, k, cap)
            if record:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record()
            kvarn.prefill_attention(q[pos0:pos0 + C], pos0, tiles, table, n_tiles, win_k[0],
                                    win_v[0], start, length, lay, ws=ws_p, out=out[pos0:pos0 + C],
                                    ws_blocks=ws_blocks, cached_tiles=prev_tiles)
            prev_tiles = n_tiles
            if record:
                b.record()
                ev.append((a, b))

    def prompt_plain():
        """The same prompt one promotion and one full conversion at a time
        (kvarn_prefill_attention with a per-call workspace): a check of the
        batched promotions and the kept images."""
        o = torch.empty_like(out)
        ws_start.zero_()
        ws_len.zero_()
        ws_nt.zero_()
        start = length = n_tiles = 0
        for pos0 in range(0, n_tok, chunk):
            C = min(chunk, n_tok - pos0)
            kvarn.append_window(kn_all[pos0:pos0 + C][None], vn_all[pos0:pos0 + C][None],
                                win_k, win_v, ws_start, ws_len)
            kvarn.window_advance(ws_start, ws_len, None, C, 0, cap)
            length += C
            while length >= Wp:
                src = torch.tensor([h * cap + start for h in range(HKV_)], dtype=torch.int64, device=dev)
                kvarn.compress_tile(win_k.view(-1, D_), win_v.view(-1, D_), src, tiles,
                                    table[:, n_tiles].contiguous(), lay)
                n_tiles += 1
                start = (start + 128) % cap
                length -= 128
                kvarn.window_advance(ws_start, ws_len, ws_nt, 0, 1, cap)
            kvarn.prefill_attention(q[pos0:pos0 + C], pos0, tiles, table, n_tiles, win_k[0],
                                    win_v[0], start, length, lay, out=o[pos0:pos0 + C])
        return o

    with torch.cuda.stream(stream):
        ref = prompt_plain()
        prompt(False)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), "batched-promotion prefill differs from the plain loop"
        del ref
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(reps):
            prompt(False)
        t1.record()
        prompt(True)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all().item(), "prefill produced non-finite output"
    layer_ms = t0.elapsed_time(t1) / reps
    attn_ms = float(sum(a.elapsed_time(b) for a, b in ev))
    # algorithmic multiply-adds: every visible (query, key) pair, Q.K and P.V
    vis = sum((p + 1) for p in range(n_tok))
    macs = 2.0 * vis * HQ_ * D_
    tflops = 2.0 * macs / (attn_ms * 1e-3) / 1e12
    peak_tf = float(peaks.get("bf16_tflops", 1900.0))
    res = {"workload": f"{label} chunked prefill: {n_tok}-token prompt, {chunk}-token chunks, W={Wp}, "
                       f"{HQ_}q/{HKV_}kv, head_dim {D_}, causal; one layer",
           "layer_ms": layer_ms, "attention_ms": attn_ms,
           "prompt_tokens_per_s_one_layer": n_tok / (layer_ms * 1e-3),
           "algorithmic_macs": macs, "achieved_tflops": tflops,
           "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak_tf, "unit": "TFLOP/s",
                        "frac": tflops / peak_tf, "traffic": None,
                        "kernel": "prefill_kernel_d256" if D_ == 256 else f"prefill_kernel<{D_}>",
                        "peak_source": peak_kind + " (dense bf16 burst; fp16 runs at the bf16 rate)"},
           "mma": "tcgen05 kind::f16, A operand from TMEM; Q', K~, P and V~ each an fp16 hi+lo "
                  "pair (3 MMAs for Q.K, 3 for P.V)"
                  + ("; keys in 64-key sub-blocks" if D_ == 256 else "")}
    if workload == "qwen3_8b_prefill":
        res["prompt_tokens_per_s_36_layers"] = n_tok / (LAYERS * layer_ms * 1e-3)
    return res


def run_prefill_d256(dev, stream, peaks, peak_kind):
    """Chunked prefill with the batched-decode head shape (16q/4kv, head_dim
    256): one layer of an 8,192-token prompt in 512-token chunks, W=256."""
    from kv_cache_quantization_token_gb300 import kvarn
    return run_prefill_bench(dev, stream, kvarn.layout(256), peaks, peak_kind, n_tok=8192,
                             workload="batched_d256_decode", hq=16, hkv=4,
                             label="16q/4kv head_dim-256")


def run_decode_sweeps(dev, lay, peaks, peak_kind):
    """Decode split throughput beyond the headline configuration: the 8B-like
    model at 4k and 32k context, and at 16k on records of the f16-scale layout
    and of the k4v4 variant (36 layers of distinct caches, split launches back to back as in the
    headline roofline); the 0.6B-like model (16q/8kv, 28 layers, 3072 + 77
    tokens); and batched decode with large
    heads (32 ragged sequences with contexts uniform in [8k, 32k], 16q/4kv,
    head_dim 256; one layer's cache is 0.6 GB), timed as back-to-back split
    launches and as decode steps (split + combine) with a concurrent compress
    stream promoting one tile per sequence per step."""
    import torch
    from kv_cache_quantization_token_gb300 import kvarn, synth
    hbm = float(peaks["hbm_gbs"])
    res = {}
    stream = torch.cuda.Stream(device=dev)

    def back_to_back(launch, n_launch, reps=10):
        with torch.cuda.stream(stream):
            launch()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            launch()
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                g.replay()
            b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (reps * n_launch)

    # ---- 8B-like decode at 4k and 32k, and at 16k on f16-scale and k4v4
    # records; and the 0.6B-like model (16q/8kv, 28 layers) at 3072 + 77 tokens
    points = [("qwen3_8b_ctx4096", WORKLOAD, HQ, LAYERS, 4096, 64, 32, 2),
              ("qwen3_8b_ctx32768", WORKLOAD, HQ, LAYERS, 32768, 64, 32, 2),
              ("qwen3_8b_ctx16384_f16_scales", WORKLOAD, HQ, LAYERS, 16384, 64, 16, 2),
              ("qwen3_8b_ctx16384_k4v4", WORKLOAD, HQ, LAYERS, 16384, 64, 32, 4),
              ("qwen3_0p6b_ctx3072", "qwen3_0p6b_decode", 16, 28, 3072, 77, 32, 2)]
    for name, wl_name, hq, n_layers, ctx, w0, sb, vb in points:
        lay_s = lay if (sb, vb) == (32, 2) else kvarn.layout(D, scale_bits=sb, v_bits=vb)
        n0, cap = ctx // 128, 128
        rb = lay_s.record_bytes
        max_tiles = n0 + 1
        tiles = torch.empty(n_layers * HKV * max_tiles * rb, dtype=torch.uint8, device=dev)
        table = torch.empty(n_layers, 1, HKV, max_tiles, dtype=torch.int64, device=dev)
        win_k = torch.zeros(n_layers, 1, HKV, cap, D, device=dev)
        win_v = torch.zeros_like(win_k)
        raw = []
        for r in range(2):  # two distinct layers of values, stored at n_layers distinct addresses
            ks, vs = synth.kv_layer(wl_name, 200 + r, HKV, ctx + w0, D)
            raw.append((torch.from_numpy(ks.reshape(-1, D)).to(dev),
                        torch.from_numpy(vs.reshape(-1, D)).to(dev), ks[:, ctx:], vs[:, ctx:]))
            del ks, vs
        src = torch.from_numpy((np.arange(HKV)[:, None] * (ctx + w0)
                                + 128 * np.arange(n0)[None, :]).reshape(-1).astype(np.int64)).to(dev)
        for l in range(n_layers):
            tab = ((l * HKV) * max_tiles + np.arange(HKV)[:, None] * max_tiles
                   + np.arange(max_tiles)[None, :]) * rb
            table[l, 0] = torch.from_numpy(tab.astype(np.int64))
            kd, vd, kw, vw = raw[l % 2]
            kvarn.compress_tile(kd, vd, src, tiles,
                                torch.from_numpy(tab[:, :n0].reshape(-1).astype(np.int64)).to(dev), lay_s)
            win_k[l, 0, :, :w0] = torch.from_numpy(kw).to(dev)
            win_v[l, 0, :, :w0] = torch.from_numpy(vw).to(dev)
        del raw
        q = torch.from_numpy(synth.queries(wl_name, 3, (n_layers, 1, hq, D))).to(dev)
        ws = torch.empty(kvarn.decode_workspace_bytes(1, hq, HKV, D, max_tiles, cap) + 256,
                         dtype=torch.uint8, device=dev)
        out = torch.empty(n_layers, 1, hq, D, device=dev)
        wst = torch.zeros(1, dtype=torch.int32, device=dev)
        wl = torch.full((1,), w0, dtype=torch.int32, device=dev)
        nt = torch.full((1,), n0, dtype=torch.int32, device=dev)

        def splits():
            for l in range(n_layers):
                kvarn.decode_split(q[l], tiles, table[l], nt, win_k[l], win_v[l], wst, wl, lay_s, ws,
                                   flags=FAST)

        def steps():
            for l in range(n_layers):
                kvarn.decode_split(q[l], tiles, table[l], nt, win_k[l], win_v[l], wst, wl, lay_s, ws,
                                   flags=FAST)
                kvarn.decode_combine(ws, out[l], HKV, max_tiles, cap, flags=FAST)

        split_ms = back_to_back(splits, n_layers)
        layer_ms = back_to_back(steps, n_layers)
        assert torch.isfinite(out).all().item(), "decode produced non-finite output"
        nbytes = HKV * n0 * rb + HKV * w0 * D * 8 + hq * D * 4
        gbs = nbytes / (split_ms * 1e-3) / 1e9
        res[name] = {
            "record_bytes": rb, "q_heads": hq, "kv_heads": HKV, "layers": n_layers,
            "context": ctx + w0,
            "split_back_to_back_ms": split_ms, "split_bytes_per_launch": nbytes,
            "split_gbs": gbs, "split_frac": gbs / hbm,
            "attention_ms_per_layer": layer_ms,
            f"tokens_per_s_{n_layers}_layers": 1.0 / (n_layers * layer_ms * 1e-3)}
        del tiles, table, win_k, win_v, ws

    # ---- batched decode, head_dim 256 ------------------------------------------
    Bb, Hqb, Hkvb, Db, capb = 32, 16, 4, 256, 128
    layb = kvarn.layout(Db)
    rbb = layb.record_bytes
    ctxs = synth.uniform_ints(4242, 8192, 32768, Bb)
    ntl = ctxs // 128
    wlen = ctxs % 128
    max_tiles = int(ntl.max()) + 1
    pool_tiles = 64  # distinct tile values per head, stored at every sequence's slots
    ks, vs = synth.kv_layer("batched_d256_decode", 0, Hkvb, 128 * pool_tiles + capb, Db)
    kd = torch.from_numpy(ks.reshape(-1, Db)).to(dev)
    vd = torch.from_numpy(vs.reshape(-1, Db)).to(dev)
    tiles = torch.empty(Bb * Hkvb * max_tiles * rbb, dtype=torch.uint8, device=dev)
    tab = ((np.arange(Bb)[:, None, None] * Hkvb + np.arange(Hkvb)[None, :, None]) * max_tiles
           + np.arange(max_tiles)[None, None, :]) * rbb
    table = torch.from_numpy(tab.astype(np.int64)).to(dev)
    src_l, dst_l = [], []
    for b in range(Bb):
        for h in range(Hkvb):
            t = np.arange(ntl[b])
            src_l.append(h * (128 * pool_tiles + capb) + 128 * (t % pool_tiles))
            dst_l.append(tab[b, h, :ntl[b]])
    kvarn.compress_tile(kd, vd, torch.from_numpy(np.concatenate(src_l).astype(np.int64)).to(dev),
                        tiles, torch.from_numpy(np.concatenate(dst_l).astype(np.int64)).to(dev), layb)
    win_k = torch.zeros(Bb, Hkvb, capb, Db, device=dev)
    win_v = torch.zeros_like(win_k)
    tail = torch.from_numpy(ks[:, 128 * pool_tiles:]).to(dev)
    tailv = torch.from_numpy(vs[:, 128 * pool_tiles:]).to(dev)
    win_k[:] = tail[None]
    win_v[:] = tailv[None]
    del ks, vs
    q = torch.from_numpy(synth.queries("batched_d256_decode", 0, (Bb, Hqb, Db))).to(dev)
    wst = torch.zeros(Bb, dtype=torch.int32, device=dev)
    wl = torch.from_numpy(wlen.astype(np.int32)).to(dev)
    nt = torch.from_numpy(ntl.astype(np.int32)).to(dev)
    ws = torch.empty(kvarn.decode_workspace_bytes(Bb, Hqb, Hkvb, Db, max_tiles, capb) + 256,
                     dtype=torch.uint8, device=dev)
    out = torch.empty(Bb, Hqb, Db, device=dev)
    # promotion work of one step: one tile per sequence and KV head, into scratch records
    n_prom = Bb * Hkvb
    psrc = torch.from_numpy((np.arange(n_prom) % Hkvb * (128 * pool_tiles + capb)
                             + 128 * (np.arange(n_prom) % pool_tiles)).astype(np.int64)).to(dev)
    pdst = torch.arange(n_prom, dtype=torch.int64, device=dev) * rbb
    ptiles = torch.empty(n_prom * rbb, dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream(device=dev)
    ev_f, ev_j = torch.cuda.Event(), torch.cuda.Event()

    def split1():
        kvarn.decode_split(q, tiles, table, nt, win_k, win_v, wst, wl, layb, ws, flags=FAST)

    def step_conc():
        cur = torch.cuda.current_stream()
        ev_f.record(cur)
        side.wait_event(ev_f)
        with torch.cuda.stream(side):
            kvarn.compress_tile(kd, vd, psrc, ptiles, pdst, layb)
        ev_j.record(side)
        kvarn.decode_split(q, tiles, table, nt, win_k, win_v, wst, wl, layb, ws, flags=FAST)
        kvarn.decode_combine(ws, out, Hkvb, max_tiles, capb, flags=FAST)
        cur.wait_event(ev_j)

    split_ms = back_to_back(lambda: [split1() for _ in range(8)], 8)
    step_ms = back_to_back(step_conc, 1, reps=40)
    assert torch.isfinite(out).all().item(), "decode produced non-finite output"
    nbytes = int(ntl.sum()) * Hkvb * rbb + int(wlen.sum()) * Hkvb * Db * 8 + Bb * Hqb * Db * 4
    gbs = nbytes / (split_ms * 1e-3) / 1e9
    res["batched_d256"] = {
        "workload": f"batch {Bb}, contexts uniform in [8192, 32768] (seeded; sum {int(ctxs.sum())}), "
                    f"{Hqb}q/{Hkvb}kv heads, head_dim {Db}, K4/V2 tiles + FP32 window (W=128); "
                    f"one layer",
        "split_back_to_back_ms": split_ms, "split_bytes_per_launch": nbytes,
        "split_gbs": gbs, "split_frac": gbs / hbm,
        "step_ms_with_concurrent_compress": step_ms,
        "tokens_per_s_per_layer": Bb / (step_ms * 1e-3),
        "concurrent_compress_tile_heads_per_step": n_prom,
        "peak_source": peak_kind}
    return res


def workload_config():
    return {"workload": f"Qwen3-8B-like KVarN decode attention: batch 1, {HQ}q/{HKV}kv heads, "
                        f"head_dim {D}, {LAYERS} layers of distinct caches at "
                        f"{CTX0}+ tokens (K4/V2 tiles + FP32 window, W={W}); "
                        f"plus bulk compress of {C_TILES}x{C_HEADS} tile-heads (32k ctx)",
            "global_batch": 1, "seq_len": CTX0, "layers": LAYERS, "head_dim": D,
            "q_heads": HQ, "kv_heads": HKV, "parallelism": "replicas",
            "l2": "inputs larger than L2: 36 distinct layer caches (>576 MiB) read per step"}


# --------------------------------------------------------------------------
def run_compress_bench(dev, stream, lay, warmup, hbm, peak_kind, tiles=C_TILES, keep=None):
    """One compress launch over tiles x C_HEADS tile-heads of fresh raw K/V
    (256 MiB of input at the defaults, larger than L2), timed with CUDA
    events per launch. With `keep` (a dict), the raw rows and the GPU records
    of the first 32 units are left there for the host-side baseline leg."""
    import torch
    from kv_cache_quantization_token_gb300 import kvarn, synth
    D, rb = lay.head_dim, lay.record_bytes
    n_units = tiles * C_HEADS
    ks, vs = synth.kv_layer(WORKLOAD, 99, C_HEADS, 128 * tiles, D)
    ck = torch.from_numpy(ks.reshape(-1, D)).to(dev)
    cv = torch.from_numpy(vs.reshape(-1, D)).to(dev)
    if keep is not None:
        keep["k"] = ks.reshape(-1, D)[:32 * 128].copy()
        keep["v"] = vs.reshape(-1, D)[:32 * 128].copy()
    del ks, vs
    csrc = torch.arange(n_units, dtype=torch.int64, device=dev) * 128
    cdst = torch.arange(n_units, dtype=torch.int64, device=dev) * rb
    ctiles = torch.empty(n_units * rb, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            kvarn.compress_tile(ck, cv, csrc, ctiles, cdst, lay)
        c_reps = 20
        cev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(c_reps)]
        for a, b in cev:
            a.record()
            kvarn.compress_tile(ck, cv, csrc, ctiles, cdst, lay)
            b.record()
    torch.cuda.synchronize()
    if keep is not None:
        keep["records"] = ctiles[:32 * rb].cpu().numpy()
        keep["record_bytes"] = rb
    comp_ms = float(np.mean([a.elapsed_time(b) for a, b in cev]))
    comp_bytes = n_units * (2 * 128 * D * 4 + rb)
    comp_gbs = comp_bytes / (comp_ms * 1e-3) / 1e9
    trc = NCU_TRAFFIC["compress"]  # captured on the head_dim-128, 2048-tile-head launch
    same_launch = D == 128 and n_units == C_TILES * C_HEADS
    ctraffic = trc["bytes"] if same_launch and trc["src_sha"] == src_sha("compress.cu") else None
    return {"tile_heads_per_launch": n_units, "ms_per_launch": comp_ms,
            "tiles_per_s": n_units / (comp_ms * 1e-3), "gbs": comp_gbs,
            "bytes_per_launch": comp_bytes,
            "roofline": {"bound": "hbm", "achieved": comp_gbs, "peak": hbm,
                         "unit": "GB/s", "frac": comp_gbs / hbm,
                         "traffic": ctraffic, "kernel": f"compress_kernel<{D}>",
                         "peak_source": peak_kind}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="kvarn", choices=["kvarn", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--section", default="all",
                    choices=["all", "decode", "prefill", "prefill-d256", "decode-sweeps", "compress"],
                    help="decode: the headline decode step alone (no secondary measurements); "
                         "the others run one secondary measurement alone and print its JSON "
                         "(for profiling)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    import torch.distributed as dist
    from kv_cache_quantization_token_gb300 import _build, kvarn, synth

    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    lay = kvarn.layout(D)
    if args.section not in ("all", "decode"):
        peaks, peak_kind = measured_peaks()
        if args.section == "prefill":
            st = torch.cuda.Stream(device=dev)
            sec = {"head_dim_128": run_prefill_bench(dev, st, lay, peaks, peak_kind),
                   "head_dim_256": run_prefill_d256(dev, st, peaks, peak_kind)}
        elif args.section == "prefill-d256":
            sec = run_prefill_d256(dev, torch.cuda.Stream(device=dev), peaks, peak_kind)
        elif args.section == "compress":
            sec = run_compress_bench(dev, torch.cuda.Stream(device=dev), lay, args.warmup,
                                     peaks["hbm_gbs"], peak_kind)
        else:
            sec = run_decode_sweeps(dev, lay, peaks, peak_kind)
        if rank == 0:
            print(json.dumps({"section": args.section, "result": sec}), flush=True)
        return
    rb = lay.record_bytes
    B = 1
    cap = 128
    # the window starts part-filled so that it reaches W = 128, and the first
    # promotion falls, right after the first timed step (1 + warmup tokens are
    # appended before the timed region); further ones follow every 128 steps
    w0 = (126 - args.warmup) % 128
    e2e_steps = max(10, args.steps // 5)
    total_steps = 1 + args.warmup + args.steps + e2e_steps
    max_tiles = CTX0 // 128 + (w0 + total_steps) // 128 + 1

    # ---- caches: raw synthetic K/V per layer, compressed on the GPU --------
    tiles = torch.empty(LAYERS * HKV * max_tiles * rb, dtype=torch.uint8, device=dev)
    table = torch.empty(LAYERS, B, HKV, max_tiles, dtype=torch.int64, device=dev)
    win_k = torch.zeros(LAYERS, B, HKV, cap, D, device=dev)
    win_v = torch.zeros_like(win_k)
    n0 = CTX0 // 128
    for l in range(LAYERS):
        ks, vs = synth.kv_layer(WORKLOAD, l, HKV, CTX0 + w0, D)
        base = (l * HKV) * max_tiles
        tab = (base + np.arange(HKV)[:, None] * max_tiles + np.arange(max_tiles)[None, :]) * rb
        table[l, 0] = torch.from_numpy(tab.astype(np.int64))
        kd = torch.from_numpy(ks.reshape(-1, D)).to(dev)
        vd = torch.from_numpy(vs.reshape(-1, D)).to(dev)
        src = (np.arange(HKV)[:, None] * (CTX0 + w0) + 128 * np.arange(n0)[None, :]).reshape(-1)
        kvarn.compress_tile(kd, vd, torch.from_numpy(src.astype(np.int64)).to(dev), tiles,
                            torch.from_numpy(tab[:, :n0].reshape(-1).astype(np.int64)).to(dev), lay)
        win_k[l, 0, :, :w0] = torch.from_numpy(ks[:, CTX0:]).to(dev)
        win_v[l, 0, :, :w0] = torch.from_numpy(vs[:, CTX0:]).to(dev)
        del kd, vd
    win_start = torch.zeros(B, dtype=torch.int32, device=dev)
    win_len = torch.full((B,), w0, dtype=torch.int32, device=dev)
    n_tiles = torch.full((B,), n0, dtype=torch.int32, device=dev)
    q = torch.from_numpy(synth.queries(WORKLOAD, 0, (LAYERS, B, HQ, D))).to(dev)
    kn = torch.from_numpy(synth.queries(WORKLOAD, 1, (LAYERS, B, 1, HKV, D))).to(dev)
    vn = torch.from_numpy(synth.queries(WORKLOAD, 2, (LAYERS, B, 1, HKV, D))).to(dev)
    out = torch.empty(LAYERS, B, HQ, D, device=dev)
    ws = torch.empty(kvarn.decode_workspace_bytes(B, HQ, HKV, D, max_tiles, cap) + 256,
                     dtype=torch.uint8, device=dev)
    # promotion: the oldest 128 window rows of every (layer, head) -> next tile slot
    win_rows_k = win_k.view(-1, D)
    win_rows_v = win_v.view(-1, D)
    torch.cuda.synchronize()

    host = {"start": 0, "len": w0, "n_tiles": n0}
    launches = {"n": 0}

    def promote_if_due():
        if host["len"] < W:
            return
        if host["n_tiles"] >= max_tiles:
            raise RuntimeError("tile slots exhausted")
        src = ((np.arange(LAYERS * HKV) * cap) + host["start"]).astype(np.int64)
        lh = np.arange(LAYERS * HKV)
        dst = (((lh // HKV) * HKV + lh % HKV) * max_tiles + host["n_tiles"]) * rb
        kvarn.compress_tile(win_rows_k, win_rows_v, torch.from_numpy(src).to(dev, non_blocking=True),
                            tiles, torch.from_numpy(dst.astype(np.int64)).to(dev, non_blocking=True),
                            lay)
        kvarn.window_advance(win_start, win_len, n_tiles, 0, 1, cap)
        host["start"] = (host["start"] + 128) % cap
        host["len"] -= 128
        host["n_tiles"] += 1
        launches["n"] += 2

    # ---- capture one decode step ----------------------------------------
    try:
        ev_split = [(torch.cuda.Event(enable_timing=True, external=True),
                     torch.cuda.Event(enable_timing=True, external=True)) for _ in range(LAYERS)]
        timed_in_graph = True
    except TypeError:
        ev_split, timed_in_graph = None, False

    side = torch.cuda.Stream(device=dev)
    ev_fork, ev_join = torch.cuda.Event(), torch.cuda.Event()

    def step_body(record_events):
        # The layers' new K/V rows go into window slot start + len, which no
        # attention of this step reads, so the appends run on a forked stream
        # and join before the window advance (len += 1).
        cur = torch.cuda.current_stream()
        ev_fork.record(cur)
        side.wait_event(ev_fork)
        with torch.cuda.stream(side):
            for l in range(LAYERS):
                kvarn.append_window(kn[l], vn[l], win_k[l], win_v[l], win_start, win_len,
                                    flags=FAST)
        ev_join.record(side)
        for l in range(LAYERS):
            if record_events:
                ev_split[l][0].record()
            kvarn.decode_split(q[l], tiles, table[l], n_tiles, win_k[l], win_v[l], win_start,
                               win_len, lay, ws, flags=FAST)
            if record_events:
                ev_split[l][1].record()
            kvarn.decode_combine(ws, out[l], HKV, max_tiles, cap, flags=FAST)
        cur.wait_event(ev_join)
        kvarn.window_advance(win_start, win_len, None, 1, 0, cap, flags=FAST)

    per_step_launches = 3 * LAYERS + 1
    # kernels of a step chain by programmatic dependent launch; the split kernels
    # stream their records in before waiting on the previous kernel (nothing in
    # the step writes records, tables or tile counts: promotions run between steps)
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        step_body(False)  # warm the function attributes outside capture
        host["len"] += 1
        promote_if_due()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step_body(False)
    if timed_in_graph:  # the same step with events around each split launch
        graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ev, stream=stream):
            step_body(True)
    # the split kernels of all layers back to back (one graph), for their
    # sustained per-launch time
    graph_split = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_split, stream=stream):
        for l in range(LAYERS):
            kvarn.decode_split(q[l], tiles, table[l], n_tiles, win_k[l], win_v[l], win_start,
                               win_len, lay, ws, flags=FAST)

    def run_steps(n):
        for _ in range(n):
            graph.replay()
            host["len"] += 1
            launches["n"] += per_step_launches
            with torch.cuda.stream(stream):
                promote_if_due()

    with torch.cuda.stream(stream):
        run_steps(args.warmup)
    torch.cuda.synchronize()

    # ---- timed region ----------------------------------------------------
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    launches["n"] = 0
    with torch.cuda.stream(stream):
        t_start.record()
        run_steps(args.steps)
        t_end.record()
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    gpu_launches = launches["n"]
    elapsed_ms, tokens_per_s = reduce_timing(t_start.elapsed_time(t_end), B * args.steps, world, dev)
    ms_per_step = elapsed_ms / args.steps

    # split-kernel durations: one more decode step with events around each split
    # launch, then the splits of all layers back to back
    if timed_in_graph:
        with torch.cuda.stream(stream):
            graph_ev.replay()
            host["len"] += 1
            promote_if_due()
        torch.cuda.synchronize()
        split_ms = float(np.mean([a.elapsed_time(b) for a, b in ev_split]))
        split_how = "CUDA events captured around each split launch of one decode step (graph)"
    else:
        with torch.cuda.stream(stream):
            evs = []
            for l in range(LAYERS):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                kvarn.decode_split(q[l], tiles, table[l], n_tiles, win_k[l], win_v[l], win_start,
                                   win_len, lay, ws, flags=FAST)
                b.record()
                evs.append((a, b))
        torch.cuda.synchronize()
        split_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
        split_how = "CUDA events around eager split launches after the timed region"
    reps = 20
    with torch.cuda.stream(stream):
        graph_split.replay()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(reps):
            graph_split.replay()
        s1.record()
    torch.cuda.synchronize()
    split_seq_ms = s0.elapsed_time(s1) / (reps * LAYERS)
    ctx_now = 128 * host["n_tiles"] + host["len"]
    packed = B * HKV * host["n_tiles"] * rb
    window_bytes = B * HKV * host["len"] * D * 4 * 2
    split_bytes = packed + window_bytes + B * HQ * D * 4
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    split_gbs = split_bytes / (split_ms * 1e-3) / 1e9
    seq_gbs = split_bytes / (split_seq_ms * 1e-3) / 1e9
    tr = NCU_TRAFFIC["decode_split"]
    traffic = (round(tr["bytes"] * split_bytes / tr["algorithmic"])
               if tr["src_sha"] == src_sha("decode.cu") else None)

    # ---- e2e: host buffers through the public API ---------------------------
    q_h = q.cpu().pin_memory()
    kn_h, vn_h = kn.cpu().pin_memory(), vn.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = q.numel() * 4 + kn.numel() * 4 + vn.numel() * 4
    d2h = out.numel() * 4
    with torch.cuda.stream(stream):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(e2e_steps):
            q.copy_(q_h, non_blocking=True)
            kn.copy_(kn_h, non_blocking=True)
            vn.copy_(vn_h, non_blocking=True)
            graph.replay()
            host["len"] += 1
            promote_if_due()
            out_h.copy_(out, non_blocking=True)
        e1.record()
    torch.cuda.synchronize()
    _, e2e_tps = reduce_timing(e0.elapsed_time(e1), B * e2e_steps, world, dev)
    assert np.isfinite(out_h.numpy()).all(), "decode produced non-finite output"

    secondary = args.section == "all"
    compress = prefill = prefill_d256 = sweeps = None
    # ---- compress bulk (32k-token 8B-like caches) ------------------------------
    if secondary:
        compress_sample = {}
        compress = run_compress_bench(dev, stream, lay, args.warmup, hbm, peak_kind,
                                      keep=compress_sample)
        # head_dim 256: 1024 tile-heads, the same 256 MiB of input
        try:
            compress["head_dim_256"] = run_compress_bench(dev, stream, kvarn.layout(256),
                                                          args.warmup, hbm, peak_kind,
                                                          tiles=C_TILES // 2)
        except Exception as e:  # a secondary measurement: report, keep the bench line
            print(f"head_dim-256 compress measurement failed: {e!r}", file=sys.stderr)
            compress["head_dim_256"] = {"error": repr(e)}

        # ---- chunked prefill (15,500-token prompt, 512-token chunks, W=256), and
        # an 8,192-token prompt with head_dim-256 heads
        prefill = run_prefill_bench(dev, stream, lay, peaks, peak_kind)
        prefill_d256 = run_prefill_d256(dev, stream, peaks, peak_kind)
        # ---- decode at other contexts and batched large-head decode
        sweeps = run_decode_sweeps(dev, lay, peaks, peak_kind)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and secondary:
        # layer 0's whole 16k-token cache, repeated for about 10 s of host work
        smp = OracleDecodeSample(CTX0 // 128)
        secs, t_all = [], time.perf_counter()
        while len(secs) < 2 or (time.perf_counter() - t_all < 10.0 and len(secs) < 20):
            secs.append(smp.run())
        sec = float(np.mean(secs))
        cpu = {"value": 1.0 / (sec * smp.scale), "unit": "tokens/s", "cores": smp.threads,
               "kind": "oracle", "sample": f"{smp.sample}; mean of {len(secs)} runs",
               "sample_seconds": float(np.sum(secs))}
        # the same oracle on one host thread (a quarter of the context, ~2 s per run)
        one = OracleDecodeSample(CTX0 // 512, threads=1)
        secs1 = [one.run() for _ in range(3)]
        cpu["single_thread"] = {"value": 1.0 / (float(np.mean(secs1)) * one.scale),
                                "unit": "tokens/s", "cores": 1,
                                "sample": f"{one.sample}; mean of 3 runs",
                                "sample_seconds": float(np.sum(secs1))}
        cpu["compress"] = oracle_compress_baseline(compress_sample)
        cpu["prefill_2048_prefix"] = oracle_prefill_baseline()

    if rank == 0:
        res = {
            "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(),
            "decode": {"ctx_end": ctx_now, "split_bytes_per_launch": split_bytes,
                       "split_back_to_back_ms": split_seq_ms, "split_back_to_back_gbs": seq_gbs,
                       "back_to_back_timing": f"CUDA events around {reps} replays of a graph of "
                                              f"the {LAYERS} layers' split launches (programmatic "
                                              f"dependent launch, records prefetched); each "
                                              f"launch reads its own layer's cache from HBM",
                       "split_isolated_ms": split_ms, "split_isolated_gbs": split_gbs,
                       "isolated_timing": split_how + "; includes the launch latency",
                       "step_attention_gbs": LAYERS * split_bytes / (ms_per_step * 1e-3) / 1e9,
                       "step_attention_frac": LAYERS * split_bytes / (ms_per_step * 1e-3) / 1e9 / hbm,
                       "launch_flags": "PDL|PREFETCH"},
            "roofline": {"bound": "hbm", "achieved": seq_gbs, "peak": hbm, "unit": "GB/s",
                         "frac": seq_gbs / hbm, "traffic": traffic,
                         "traffic_source": "ncu DRAM read + write bytes of one split launch at "
                                           "16.5k context (1.004 x its algorithmic bytes), scaled "
                                           "to this launch's algorithmic bytes",
                         "kernel": "decode_split_kernel",
                         "timing": "average launch duration over back-to-back launches (see "
                                   "decode.back_to_back_timing)", "peak_source": peak_kind},
            "compress": compress,
            "prefill": prefill,
            "prefill_d256": prefill_d256,
            "decode_sweeps": sweeps,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_tps, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": gpu_launches,
            "clocks": clock_info,
        }
        print(json.dumps(res), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
