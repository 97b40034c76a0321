"""Seeded synthetic inputs shaped like the KVarN workloads.

This module holds no arithmetic of the method: it only draws random numbers.
Both the CUDA path's tests/benchmark and the CPU oracle consume its arrays.

The pages measure on wikitext-2 with Qwen3-0.6B / Qwen3-8B weights, which are
not available here; these tensors stand in for them with the same shapes and
with value distributions that have the features KVarN targets (channel
outliers in keys, heavy-tailed per-token scales in values):

  family "lognormal" (single tile; Qwen3-0.6B-like decode):
    K = N(0,1) * per-channel exp(N(0,1)), with 4 distinct outlier channels x20
    V = N(0,1) * per-token exp(0.5 * N(0,1))
  family "heavy" (Qwen3-8B-like decode and prefill; batched head_dim-256 decode):
    K as above with round(0.02 * D) outlier channels x20 (3 at D=128, 5 at D=256)
    V = N(0,1) * per-token |t_4| (Student-t, 4 degrees of freedom)
  queries: N(0,1) fp32.

Draws are fp32 (numpy's float32 normal sampler). Seeds: numpy PCG64 with
seed = base + 1000 * index(workload) + 37 * layer + kv_head for K/V streams;
queries use a separate stream keyed the same way plus 500_000.
"""
from __future__ import annotations

import numpy as np

# workload name -> (seed index, value family)
WORKLOADS = {
    "single_tile": (0, "lognormal"),          # one 128-token tile + 17-token window, D=128
    "qwen3_0p6b_decode": (1, "lognormal"),    # 16q/8kv, D=128, 3k context
    "qwen3_8b_decode": (2, "heavy"),          # 32q/8kv, D=128, 4k-32k context
    "qwen3_8b_prefill": (3, "heavy"),         # 15.5k prompt, 512-token chunks, W=256
    "batched_d256_decode": (4, "heavy"),      # 32 ragged sequences, 16q/4kv, D=256
}


def stream_seed(workload: str, layer: int, kv_head: int, base: int = 0) -> int:
    return base + 1000 * WORKLOADS[workload][0] + 37 * layer + kv_head


def kv_stream(workload: str, layer: int, kv_head: int, n_tokens: int, head_dim: int,
              base: int = 0):
    """K and V rows of one KV head, fp32 [n_tokens][head_dim] each."""
    rng = np.random.default_rng(stream_seed(workload, layer, kv_head, base))
    D = head_dim
    fam = WORKLOADS[workload][1]
    n_out = 4 if fam == "lognormal" else int(round(0.02 * D))
    ch_scale = np.exp(rng.standard_normal(D))
    outliers = rng.choice(D, size=n_out, replace=False)
    ch_scale[outliers] *= 20.0
    k = rng.standard_normal((n_tokens, D), dtype=np.float32)
    k *= ch_scale.astype(np.float32)[None, :]
    if fam == "lognormal":
        tok_scale = np.exp(0.5 * rng.standard_normal(n_tokens))
    else:
        tok_scale = np.abs(rng.standard_t(4.0, n_tokens))
    v = rng.standard_normal((n_tokens, D), dtype=np.float32)
    v *= tok_scale.astype(np.float32)[:, None]
    return k, v


def kv_layer(workload: str, layer: int, n_kv_heads: int, n_tokens: int, head_dim: int,
             base: int = 0):
    """K, V of every KV head of a layer: fp32 [n_kv_heads][n_tokens][head_dim]."""
    ks, vs = zip(*(kv_stream(workload, layer, h, n_tokens, head_dim, base)
                   for h in range(n_kv_heads)))
    return np.stack(ks), np.stack(vs)


def queries(workload: str, layer: int, shape, base: int = 0) -> np.ndarray:
    """N(0,1) fp32 queries of any shape (e.g. [B][Hq][D])."""
    rng = np.random.default_rng(500_000 + stream_seed(workload, layer, 0, base))
    return rng.standard_normal(shape).astype(np.float32)


def uniform_ints(seed: int, lo: int, hi: int, n: int) -> np.ndarray:
    """n seeded integers uniform in [lo, hi] (window lengths, ragged contexts)."""
    return np.random.default_rng(seed).integers(lo, hi + 1, size=n)
