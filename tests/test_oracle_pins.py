"""Pins of the fp64 oracle against facts that do not come from the oracle
itself: textbook matrices, closed forms, invariants of the algebra, hand-worked
examples and library routines the oracle does not use.

Each test names the step of the method it pins (SharpInference issue #180,
"Algorithm (per 128-token tile)"; PR #434 commit 82efc4f for packing) and the
plausible mistake it is there to catch.
"""
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.special

from kv_cache_quantization_token_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# ------------------------------------------------------------------ c1: WHT
def test_wht_order4_matches_textbook_matrix(oracle):
    """Issue #180 step 1. H_4 from the Sylvester recursion, typed in the golden
    file by hand; catches sequency/bit-reversed ordering and sign slips."""
    rows = _read_golden("hadamard4.txt")
    H4 = np.array([[float(x) for x in r.split()] for r in rows]) / 2.0
    got = oracle.wht_rows(np.eye(4))  # row i of the result is H e_i = column i
    np.testing.assert_allclose(got.T, H4, atol=1e-15)
    H2 = oracle.wht_rows(np.eye(2)).T
    np.testing.assert_allclose(H2, np.array([[1, 1], [1, -1]]) / np.sqrt(2), atol=1e-15)


@pytest.mark.parametrize("D", [2, 8, 64, 128, 256])
def test_wht_matches_scipy_sylvester(oracle, D):
    """scipy.linalg.hadamard builds the Sylvester matrix; the oracle does not use it."""
    H = scipy.linalg.hadamard(D) / np.sqrt(D)
    np.testing.assert_allclose(oracle.wht_rows(np.eye(D)).T, H, atol=1e-14)


@pytest.mark.parametrize("D", [4, 64, 128, 256])
def test_wht_orthonormal_self_inverse_preserves_dot(oracle, D):
    """H orthonormal and symmetric: H(Hx) = x, |Hx| = |x|, (Hq).(Hk) = q.k."""
    rng = np.random.default_rng(D)
    x = rng.standard_normal((5, D))
    y = oracle.wht_rows(x)
    np.testing.assert_allclose(oracle.wht_rows(y), x, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    hq, hk = oracle.wht_rows(q[None])[0], oracle.wht_rows(k[None])[0]
    assert abs(hq @ hk - q @ k) <= 1e-12 * (np.abs(q) @ np.abs(k))


# ------------------------------------------------------------- c2: Sinkhorn
def _balanced_pm1(T, D, seed):
    """A +-1 matrix whose every row and every column has mean 0 and std 1."""
    rng = np.random.default_rng(seed)
    a = np.where(rng.permutation(T) < T // 2, 1.0, -1.0)
    b = np.where(rng.permutation(D) < D // 2, 1.0, -1.0)
    return np.outer(a, b)


def test_sinkhorn_closed_form_column_scaled_fixed_point(oracle):
    """Issue #180 step 2. Y = Z diag(b) with Z balanced +-1: the first channel
    step gives s = b exactly and every later std is 1, so r = 1 and Yn = Z.
    Catches exp(+alpha) for exp(-alpha), ln(var) for ln(std), and a sample
    (N-1) std, each of which moves s, r or Yn off the closed form."""
    T, D = 128, 64
    Z = _balanced_pm1(T, D, 3)
    b = np.exp(np.random.default_rng(4).standard_normal(D))
    for iters in (1, 4):
        s, r, yn = oracle.sinkhorn(Z * b[None, :], iters)
        np.testing.assert_allclose(s, b, rtol=1e-13)
        np.testing.assert_allclose(r, 1.0, rtol=1e-13)
        np.testing.assert_allclose(yn, Z, atol=1e-13)


def test_sinkhorn_channel_step_comes_first(oracle):
    """Channel step first (issue #180 step 2 names per-channel before per-token):
    then any positive per-channel scaling of Y is absorbed by s exactly and
    leaves r and Yn unchanged at every iteration count. With the token step
    first this only holds in the limit."""
    k, _ = synth.kv_stream("single_tile", 1, 0, 128, 128)
    Y = oracle.wht_rows(k.astype(np.float64))
    b = np.exp(np.random.default_rng(5).standard_normal(128))
    for iters in (1, 2, 4):
        s0, r0, y0 = oracle.sinkhorn(Y, iters)
        s1, r1, y1 = oracle.sinkhorn(Y * b[None, :], iters)
        np.testing.assert_allclose(s1, s0 * b, rtol=1e-12)
        np.testing.assert_allclose(r1, r0, rtol=1e-12)
        np.testing.assert_allclose(y1, y0, atol=1e-12)


@pytest.mark.parametrize("workload,D", [("single_tile", 128), ("qwen3_8b_decode", 128), ("batched_d256_decode", 256), ("qwen3_8b_decode", 64)])
def test_sinkhorn_normalises_rows_and_converges_on_columns(oracle, workload, D):
    """After the last (token) step every token std of Yn is 1; the worst
    channel |ln std| never grows with more rounds and is below 0.05 at n = 4
    on the synthetic workloads' distributions."""
    k, v = synth.kv_stream(workload, 2, 1, 128, D)
    for x in (k, v):
        Y = oracle.wht_rows(x.astype(np.float64))
        prev = np.inf
        for iters in (1, 2, 3, 4, 6):
            s, r, yn = oracle.sinkhorn(Y, iters)
            np.testing.assert_allclose(yn.std(axis=1), 1.0, rtol=1e-12)
            np.testing.assert_allclose(yn, Y / np.outer(r, s), rtol=1e-12)
            worst = np.abs(np.log(yn.std(axis=0))).max()
            assert worst <= prev * (1 + 1e-9)
            prev = worst
            if iters == 4:
                assert worst < 0.05


def test_sinkhorn_global_scale_moves_only_s(oracle):
    """Y -> cY: s -> c s, r and Yn unchanged (the channel step sees c first)."""
    _, v = synth.kv_stream("qwen3_8b_decode", 0, 3, 128, 128)
    Y = oracle.wht_rows(v.astype(np.float64))
    s0, r0, y0 = oracle.sinkhorn(Y, 4)
    s1, r1, y1 = oracle.sinkhorn(3.7 * Y, 4)
    np.testing.assert_allclose(s1, 3.7 * s0, rtol=1e-12)
    np.testing.assert_allclose(r1, r0, rtol=1e-12)
    np.testing.assert_allclose(y1, y0, atol=1e-12)


def test_sinkhorn_skips_degenerate_groups(oracle):
    """Skip rule (a reading; the pages are silent): an all-zero tensor keeps
    s = r = 1; a constant channel is skipped although fp64 rounding leaves a
    std of ~1e-17 (an absolute 1e-30 guard would take ln of it)."""
    s, r, yn = oracle.sinkhorn(np.zeros((128, 64)), 4)
    assert np.all(s == 1.0) and np.all(r == 1.0) and np.all(yn == 0.0)
    rng = np.random.default_rng(9)
    Y = rng.standard_normal((128, 64))
    Y[:, 5] = 0.1  # constant channel: in the first Sinkhorn step its std is pure rounding
    Y[:, 9] = 0.0  # zero channel: skipped in every round
    s, r, yn = oracle.sinkhorn(Y, 1)
    assert s[5] == 1.0 and s[9] == 1.0
    # after a token step the constant channel is divided by varying r_t, so
    # later rounds update it like any other channel
    s, r, yn = oracle.sinkhorn(Y, 4)
    assert s[9] == 1.0 and np.all(yn[:, 9] == 0.0)
    assert s[5] != 1.0
    assert np.all(np.isfinite(yn))


# ------------------------------------------------------------------- c3: RTN
def test_rtn_hand_worked_cases(oracle):
    """Issue #180 step 3, asymmetric RTN with ties rounding half up. Each golden
    line: bits, values ; expected codes, worked by hand from
    code = floor((y - min) / ((max - min) / (2^bits - 1)) + 1/2)."""
    for line in _read_golden("rtn_cases.txt"):
        lhs, rhs = line.split(";")
        bits, *vals = lhs.split()
        want = [int(c) for c in rhs.split()]
        d, lo, codes, _ = oracle.rtn_group(np.array([float(x) for x in vals]), int(bits))
        assert list(codes) == want, line


@pytest.mark.parametrize("bits", [2, 4])
def test_rtn_error_bound_and_extremes(oracle, bits):
    """|y - (delta code + lo)| <= delta/2; argmin -> 0; argmax -> 2^b - 1."""
    rng = np.random.default_rng(bits)
    for _ in range(20):
        y = rng.standard_normal(128) * np.exp(rng.standard_normal())
        d, lo, codes, vpre = oracle.rtn_group(y, bits)
        assert codes.max() <= (1 << bits) - 1
        assert codes[np.argmin(y)] == 0 and codes[np.argmax(y)] == (1 << bits) - 1
        err = np.abs(y - (d * codes + lo))
        assert np.all(err <= d / 2 * (1 + 1e-12))
        np.testing.assert_allclose(vpre, (y - lo) / d, rtol=1e-15, atol=1e-15)


def test_rtn_constant_group_gives_zero_codes(oracle):
    d, lo, codes, _ = oracle.rtn_group(np.full(128, -1.25), 4)
    assert d == 0.0 and lo == -1.25 and np.all(codes == 0)


# --------------------------------------------------------------- c4: packing
@pytest.mark.parametrize("D,size", [(64, 9216), (128, 16384), (256, 31744)])
def test_record_size(oracle, D, size):
    """K 4 bit + V 2 bit + fp32 scales: 112 D + 1024 + 1024 Gv bytes."""
    assert oracle.record_bytes(D) == size


@pytest.mark.parametrize("D", [64, 128, 256])
def test_pack_unpack_roundtrip(oracle, D):
    rng = np.random.default_rng(D + 1)
    gv = D // min(D, 128)
    f32 = lambda n: rng.standard_normal(n).astype(np.float32).astype(np.float64)
    args = dict(k_codes=rng.integers(0, 16, (128, D)).astype(np.uint8),
                v_codes=rng.integers(0, 4, (128, D)).astype(np.uint8),
                k_delta=f32(D), k_lo=f32(D), k_s=f32(D), k_r=f32(128),
                v_delta=f32(128 * gv), v_lo=f32(128 * gv), v_r=f32(128), v_s=f32(D))
    rec = oracle.pack_record(D, **args)
    back = oracle.unpack_record(rec, D)
    for name, val in args.items():
        np.testing.assert_array_equal(back[name], val, err_msg=name)


def test_pack_bit_order_hand_built(oracle):
    """Channel-major K: token 2i in the low nibble of byte i of channel row c;
    token-major V: channel 4j+k in bits 2k..2k+1 of byte j of token row t."""
    D = 64
    kc = np.zeros((128, D), np.uint8)
    vc = np.zeros((128, D), np.uint8)
    kc[1, 0] = 0xA          # token 1, channel 0 -> high nibble of byte 0
    kc[2, 3] = 0x5          # token 2, channel 3 -> low nibble of byte 3*64 + 1
    vc[0, 1] = 2            # token 0, channel 1 -> bits 2..3 of V byte 0
    vc[5, 63] = 3           # token 5, channel 63 -> bits 6..7 of byte 5*16 + 15
    z = np.zeros
    rec = oracle.pack_record(D, kc, vc, z(D), z(D), z(D), z(128), z(128), z(128), z(128), z(D))
    assert rec[0] == 0xA0 and rec[3 * 64 + 1] == 0x05
    voff = 64 * D
    assert rec[voff] == 0x08 and rec[voff + 5 * 16 + 15] == 0xC0
    assert np.count_nonzero(rec) == 4


# --------------------------------------------------------- c5: reconstruction
@pytest.mark.parametrize("workload,D", [("single_tile", 128), ("qwen3_8b_decode", 128), ("batched_d256_decode", 256), ("qwen3_8b_decode", 64)])
def test_compress_dequant_distortion_bound(oracle, workload, D):
    """Per element of the rotated tile |Yn r s - recon| <= r s delta / 2, so by
    orthonormality each unrotated row error is at most the norm of those
    bounds. Pins compress and dequant against each other: a swapped factor,
    a wrong group index or a missing inverse rotation breaks it."""
    k, v = synth.kv_stream(workload, 0, 0, 128, D)
    o = oracle.compress_unit(k, v)
    kh, vh = oracle.dequant_record(o["record"], D)
    gv = D // min(D, 128)
    f = lambda a: a.astype(np.float32).astype(np.float64)  # stored scales are fp32
    kbound = f(o["k_r"])[:, None] * f(o["k_s"])[None, :] * f(o["k_delta"])[None, :] / 2
    vd = np.repeat(f(o["v_delta"]).reshape(128, gv), D // gv, axis=1)
    vbound = f(o["v_r"])[:, None] * f(o["v_s"])[None, :] * vd / 2
    for x, xh, bnd in ((k, kh, kbound), (v, vh, vbound)):
        err = np.linalg.norm(xh - x.astype(np.float64), axis=1)
        assert np.all(err <= np.linalg.norm(bnd, axis=1) * (1 + 1e-5) + 1e-6)


def test_fold_identity(oracle):
    """Issue #180 step 4, scales folded at read time: for a key row of a tile,
    q . (H K~_t) = r_t (sum_c q'_c s_c delta_c code_tc + sum_c q'_c s_c lo_c)
    with q' = H q. The explicit dequantisation is on the left."""
    D = 128
    k, v = synth.kv_stream("qwen3_8b_decode", 0, 0, 128, D)
    rec = oracle.compress_unit(k, v)["record"]
    kh, _ = oracle.dequant_record(rec, D)
    u = oracle.unpack_record(rec, D)
    q = np.random.default_rng(0).standard_normal(D)
    qr = oracle.wht_rows(q[None])[0]
    folded = u["k_r"] * ((u["k_codes"] * (qr * u["k_s"] * u["k_delta"])[None, :]).sum(1)
                         + (qr * u["k_s"] * u["k_lo"]).sum())
    np.testing.assert_allclose(kh @ q, folded, rtol=1e-11, atol=1e-11)


def test_compress_invariant_to_global_scale(oracle):
    """X -> cX (c > 0) leaves every code unchanged and moves only s."""
    k, v = synth.kv_stream("qwen3_8b_decode", 3, 0, 128, 128)
    a = oracle.compress_unit(k, v)
    b = oracle.compress_unit(k * np.float32(4.0), v * np.float32(0.25))
    ua, ub = oracle.unpack_record(a["record"], 128), oracle.unpack_record(b["record"], 128)
    np.testing.assert_array_equal(ua["k_codes"], ub["k_codes"])
    np.testing.assert_array_equal(ua["v_codes"], ub["v_codes"])
    np.testing.assert_allclose(b["k_s"], 4.0 * a["k_s"], rtol=1e-12)
    np.testing.assert_allclose(b["v_s"], 0.25 * a["v_s"], rtol=1e-12)


def test_zero_tile(oracle):
    z = np.zeros((128, 128), np.float32)
    o = oracle.compress_unit(z, z)
    kh, vh = oracle.dequant_record(o["record"], 128)
    assert np.all(kh == 0) and np.all(vh == 0)
    u = oracle.unpack_record(o["record"], 128)
    assert np.all(u["k_s"] == 1) and np.all(u["v_r"] == 1) and np.all(u["k_delta"] == 0)


# ------------------------------------------------------- c6: state machine
@pytest.mark.parametrize("W", [128, 256])
def test_rechunking_gives_identical_tiles(oracle, W):
    """PR #434 commit 99c3773 and issue #433 item 1: tiles do not depend on the
    chunking. Chunk sizes 1, 17 and 512 over 700 tokens."""
    Hkv, D, n = 2, 64, 700
    ks, vs = synth.kv_layer("single_tile", 0, Hkv, n, D)
    k_tok, v_tok = ks.transpose(1, 0, 2), vs.transpose(1, 0, 2)
    results = []
    for chunk in (1, 17, 512):
        sm = oracle.CacheStateMachine(Hkv, D, W=W)
        for i0 in range(0, n, chunk):
            sm.append(k_tok[i0:i0 + chunk], v_tok[i0:i0 + chunk])
            if chunk == 1:
                lo = 0 if W == 128 else (128 if sm.n_tokens >= W else 0)
                assert lo <= sm.win_len < W
        results.append(sm)
    for sm in results[1:]:
        assert sm.n_tiles == results[0].n_tiles == (n - W) // 128 + 1
        for t in range(sm.n_tiles):
            for h in range(Hkv):
                assert np.array_equal(sm.records[t][h], results[0].records[t][h])
        np.testing.assert_array_equal(sm.window(1)[0], results[0].window(1)[0])


# ------------------------------------------------------- c7/c8: attention
def test_attend_reduces_to_textbook_softmax(oracle):
    """With no tiles, decode is plain softmax attention (scipy.special.softmax)."""
    rng = np.random.default_rng(11)
    q, K, V = rng.standard_normal(64), rng.standard_normal((40, 64)), rng.standard_normal((40, 64))
    p = scipy.special.softmax(0.125 * (K @ q))
    np.testing.assert_allclose(oracle.attend(q, K, V, 0.125), p @ V, rtol=1e-12, atol=1e-14)


def test_attend_special_cases(oracle):
    rng = np.random.default_rng(12)
    K, V = rng.standard_normal((30, 32)), rng.standard_normal((30, 32))
    np.testing.assert_allclose(oracle.attend(np.zeros(32), K, V, 1.0), V.mean(0), atol=1e-13)
    np.testing.assert_allclose(oracle.attend(rng.standard_normal(32), K[:1], V[:1], 0.3), V[0],
                               atol=1e-15)
    assert np.all(oracle.attend(np.ones(32), K[:0], V[:0], 1.0) == 0.0)
    q = 1000.0 * K[7] / np.linalg.norm(K[7])
    np.testing.assert_allclose(oracle.attend(q, K, V, 1.0), V[7], atol=1e-9)


def test_decode_independent_of_tile_order(oracle):
    """Permuting the order of tiles in the table leaves the output unchanged."""
    D, n_t = 64, 3
    k, v = synth.kv_stream("single_tile", 0, 0, 128 * n_t + 5, D)
    pool = np.concatenate([oracle.compress_unit(k[128 * i:128 * i + 128],
                                                v[128 * i:128 * i + 128])["record"]
                           for i in range(n_t)])
    rb = oracle.record_bytes(D)
    win_k = np.zeros((1, 1, 128, D), np.float32)
    win_v = np.zeros((1, 1, 128, D), np.float32)
    win_k[0, 0, :5], win_v[0, 0, :5] = k[-5:], v[-5:]
    q = synth.queries("single_tile", 0, (1, 1, D))
    outs = []
    for perm in ([0, 1, 2], [2, 0, 1]):
        table = (np.array(perm, np.int64) * rb)[None, None, :]
        outs.append(oracle.decode_attention(q, pool, table, [n_t], win_k, win_v, [0], [5],
                                            1 / 8)[(0, 0)])
    np.testing.assert_allclose(outs[0], outs[1], rtol=1e-12, atol=1e-14)


def test_prefill_chunk_of_one_equals_decode(oracle):
    """c8: causal prefill restricted to a single query is decode (c7) at that
    step; query i of a chunk sees exactly pos0 + i + 1 tokens."""
    Hkv, Hq, D, n = 1, 2, 64, 300
    ks, vs = synth.kv_layer("qwen3_8b_decode", 0, Hkv, n, D)
    qs = synth.queries("qwen3_8b_decode", 0, (n, Hq, D))
    sm = oracle.CacheStateMachine(Hkv, D, W=128)
    rb = oracle.record_bytes(D)
    full_chunk = None
    for pos in range(n):
        sm.append(ks[:, pos:pos + 1].transpose(1, 0, 2), vs[:, pos:pos + 1].transpose(1, 0, 2))
        if pos in (0, 127, 128, 255, 299):
            pool = np.concatenate([r[0] for r in sm.records]) if sm.records else np.zeros(rb, np.uint8)
            table = (np.arange(max(sm.n_tiles, 1), dtype=np.int64) * rb)[None, :]
            wk, wv = sm.window(0)
            win_k = np.zeros((1, 256, D), np.float32)
            win_v = np.zeros((1, 256, D), np.float32)
            win_k[0, :len(wk)], win_v[0, :len(wv)] = wk, wv
            dec = oracle.decode_attention(qs[pos][None], pool, table[None], [sm.n_tiles],
                                          win_k[None], win_v[None], [0], [sm.win_len], 1 / 8)
            pre = oracle.prefill_attention(qs[pos:pos + 1], pos, pool, table, sm.n_tiles, win_k,
                                           win_v, 0, sm.win_len, 1 / 8)
            for h in range(Hq):
                np.testing.assert_allclose(pre[(0, h)], dec[(0, h)], rtol=1e-13, atol=1e-15)


def test_prefill_window_only_is_causal_softmax(oracle):
    """c8 with no tiles: each chunk row i is textbook softmax attention
    (scipy) over the raw window tokens at positions <= pos0 + i, the window a
    ring that wraps (token w at slot (start + w) mod capacity). Pins the
    causal bound (pos0 + i + 1 keys, not pos0 + i) and the ring order."""
    rng = np.random.default_rng(21)
    Hkv, Hq, D, cap, L, start = 1, 2, 64, 64, 50, 40
    keys = rng.standard_normal((L, D)).astype(np.float32)
    vals = rng.standard_normal((L, D)).astype(np.float32)
    win_k = np.zeros((Hkv, cap, D), np.float32)
    win_v = np.zeros((Hkv, cap, D), np.float32)
    for w in range(L):
        win_k[0, (start + w) % cap], win_v[0, (start + w) % cap] = keys[w], vals[w]
    C, pos0, scale = 20, 30, 0.2
    q = rng.standard_normal((C, Hq, D)).astype(np.float32)
    out = oracle.prefill_attention(q, pos0, np.zeros(oracle.record_bytes(D), np.uint8),
                                   np.zeros((Hkv, 1), np.int64), 0, win_k, win_v, start, L, scale)
    K, V = keys.astype(np.float64), vals.astype(np.float64)
    for i in range(C):
        vis = pos0 + i + 1
        for h in range(Hq):
            p = scipy.special.softmax(scale * (K[:vis] @ q[i, h].astype(np.float64)))
            np.testing.assert_allclose(out[(i, h)], p @ V[:vis], rtol=1e-12, atol=1e-14)


def test_decode_gqa_groups_are_contiguous(oracle):
    """GQA reading: query head h reads KV head h // G (contiguous groups, not
    h mod Hkv). Window-only caches that differ per KV head and per sequence;
    every (sequence, query head) against textbook softmax over its own KV
    head's tokens."""
    rng = np.random.default_rng(23)
    B, Hkv, G, D, cap, L = 2, 3, 2, 64, 32, 9
    Hq = Hkv * G
    win_k = rng.standard_normal((B, Hkv, cap, D)).astype(np.float32)
    win_v = rng.standard_normal((B, Hkv, cap, D)).astype(np.float32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    out = oracle.decode_attention(q, np.zeros(oracle.record_bytes(D), np.uint8),
                                  np.zeros((B, Hkv, 1), np.int64), [0] * B, win_k, win_v,
                                  [3] * B, [L] * B, 0.3)
    for b in range(B):
        for h in range(Hq):
            K = win_k[b, h // G, 3:3 + L].astype(np.float64)
            V = win_v[b, h // G, 3:3 + L].astype(np.float64)
            p = scipy.special.softmax(0.3 * (K @ q[b, h].astype(np.float64)))
            np.testing.assert_allclose(out[(b, h)], p @ V, rtol=1e-12, atol=1e-14)


# ------------------------------------------- c4 variant: f16-scale layout
def test_f16_rounding_matches_numpy(oracle):
    """The oracle's binary16 encoder (written from the format's definition)
    against numpy's float16 conversion, an independent implementation of the
    same IEEE rounding: random magnitudes over the whole range, exact ties
    between neighbours (ties go to the even fraction), subnormals, the
    overflow threshold 65520, and every one of the 65536 bit patterns decoded."""
    rng = np.random.default_rng(16)
    mags = np.ldexp(rng.random(4000) + 0.5, rng.integers(-30, 18, 4000))
    vals = np.concatenate([mags, -mags])
    h = np.arange(0, 0x7C00, 37, dtype=np.uint16).view(np.float16).astype(np.float64)
    ties = (h[:-1] + np.nextafter(h[:-1].astype(np.float16), np.float16(np.inf)).astype(np.float64)) / 2
    edge = np.array([0.0, -0.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -25, 2.0 ** -14, 65504.0,
                     65519.999, 65520.0, 1e9, -1e9, np.inf, -np.inf])
    with np.errstate(over="ignore"):
        for v in np.concatenate([vals, ties, edge]):
            want = int(np.array(v).astype(np.float16).view(np.uint16))
            assert oracle.f16_bits(v) == want, (v, hex(oracle.f16_bits(v)), hex(want))
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = allbits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_value(int(b)) for b in allbits])
    fin = ~np.isnan(ref)
    np.testing.assert_array_equal(got[fin], ref[fin])
    assert np.isnan(got[~fin]).all()


@pytest.mark.parametrize("D,size", [(64, 7680), (128, 14336), (256, 28160)])
def test_f16_record_size(oracle, D, size):
    """Codes as in the fp32 layout (96 D bytes), every scale field 2 bytes:
    96 D + 2 (4 D + 256 + 256 Gv); all multiples of 128."""
    assert oracle.record_bytes(D, 16) == size and size % 128 == 0


@pytest.mark.parametrize("D", [64, 128, 256])
def test_f16_pack_unpack_roundtrip(oracle, D):
    rng = np.random.default_rng(D + 16)
    gv = D // min(D, 128)
    f16 = lambda n: rng.standard_normal(n).astype(np.float16).astype(np.float64)
    args = dict(k_codes=rng.integers(0, 16, (128, D)).astype(np.uint8),
                v_codes=rng.integers(0, 4, (128, D)).astype(np.uint8),
                k_delta=f16(D), k_lo=f16(D), k_s=f16(D), k_r=f16(128),
                v_delta=f16(128 * gv), v_lo=f16(128 * gv), v_r=f16(128), v_s=f16(D))
    rec = oracle.pack_record(D, scale_bits=16, **args)
    back = oracle.unpack_record(rec, D, scale_bits=16)
    for name, val in args.items():
        np.testing.assert_array_equal(back[name], val, err_msg=name)
    # the scale fields sit right after the codes, low byte first
    assert int(rec[96 * D]) | (int(rec[96 * D + 1]) << 8) == oracle.f16_bits(args["k_delta"][0])


@pytest.mark.parametrize("workload,D", [("qwen3_8b_decode", 128), ("batched_d256_decode", 256)])
def test_f16_layout_keeps_codes_and_rounds_scales(oracle, workload, D):
    """The f16-scale record holds the fp32 layout's codes and every scale
    rounded once from fp64 to binary16; dequantisation uses the stored
    values (checked against the same algebra with the rounded scales and
    scipy's Sylvester matrix)."""
    from scipy.linalg import hadamard
    k, v = synth.kv_stream(workload, 0, 1, 128, D)
    a = oracle.compress_unit(k, v)
    b = oracle.compress_unit(k, v, scale_bits=16)
    ua = oracle.unpack_record(a["record"], D)
    ub = oracle.unpack_record(b["record"], D, scale_bits=16)
    for t in ("k_codes", "v_codes"):
        np.testing.assert_array_equal(ua[t], ub[t])
    for name in ("k_delta", "k_lo", "k_s", "k_r", "v_delta", "v_lo", "v_r", "v_s"):
        want = np.asarray(b[name], np.float64).astype(np.float16).astype(np.float64)
        np.testing.assert_array_equal(ub[name], want, err_msg=name)
    kk, vv = oracle.dequant_record(b["record"], D, scale_bits=16)
    H = hadamard(D) / np.sqrt(D)
    gv = D // min(D, 128)
    gidx = np.arange(D) // min(D, 128)
    kt = ub["k_r"][:, None] * ub["k_s"][None, :] * (ub["k_delta"][None, :] * ub["k_codes"] + ub["k_lo"][None, :])
    vd = ub["v_delta"].reshape(128, gv)[:, gidx]
    vl = ub["v_lo"].reshape(128, gv)[:, gidx]
    vt = ub["v_r"][:, None] * ub["v_s"][None, :] * (vd * ub["v_codes"] + vl)
    np.testing.assert_allclose(kk, kt @ H, rtol=0, atol=1e-12 * np.abs(kt).max())
    np.testing.assert_allclose(vv, vt @ H, rtol=0, atol=1e-12 * np.abs(vt).max())


# ------------------------------------------- c4 variant: 4-bit values (k4v4)
@pytest.mark.parametrize("D,size", [(64, 11264), (128, 20480), (256, 39936)])
def test_v4_record_size(oracle, D, size):
    """4-bit V codes take D/2 bytes per token: 128 D code bytes in all."""
    assert oracle.record_bytes(D, v_bits=4) == size
    assert oracle.record_bytes(D, v_bits=4) - oracle.record_bytes(D) == 32 * D


def test_v4_pack_bit_order_hand_built(oracle):
    """Token-major V as in the k4v2 layout, two channels per byte: channel
    2j + k of token t in bits 4k..4k+3 of byte j of token row t."""
    D = 64
    kc = np.zeros((128, D), np.uint8)
    vc = np.zeros((128, D), np.uint8)
    vc[0, 1] = 0xB          # token 0, channel 1 -> high nibble of V byte 0
    vc[3, 62] = 0x6         # token 3, channel 62 -> low nibble of byte 3*32 + 31
    z = np.zeros
    rec = oracle.pack_record(D, kc, vc, z(D), z(D), z(D), z(128), z(128), z(128), z(128), z(D),
                             v_bits=4)
    voff = 64 * D
    assert rec[voff] == 0xB0 and rec[voff + 3 * 32 + 31] == 0x06
    assert np.count_nonzero(rec) == 2


@pytest.mark.parametrize("D", [64, 128, 256])
def test_v4_pack_unpack_roundtrip(oracle, D):
    rng = np.random.default_rng(D + 4)
    gv = D // min(D, 128)
    f32 = lambda n: rng.standard_normal(n).astype(np.float32).astype(np.float64)
    args = dict(k_codes=rng.integers(0, 16, (128, D)).astype(np.uint8),
                v_codes=rng.integers(0, 16, (128, D)).astype(np.uint8),
                k_delta=f32(D), k_lo=f32(D), k_s=f32(D), k_r=f32(128),
                v_delta=f32(128 * gv), v_lo=f32(128 * gv), v_r=f32(128), v_s=f32(D))
    rec = oracle.pack_record(D, v_bits=4, **args)
    back = oracle.unpack_record(rec, D, v_bits=4)
    for name, val in args.items():
        np.testing.assert_array_equal(back[name], val, err_msg=name)


@pytest.mark.parametrize("workload,D", [("qwen3_8b_decode", 128), ("batched_d256_decode", 256)])
def test_v4_compress_keeps_keys_and_bounds_value_error(oracle, workload, D):
    """The k4v4 record: the K half is the k4v2 record's (codes and scales);
    V is quantised to 16 levels per token group, so every rotated, normalised
    V element is within delta/2 of its reconstruction, the group extremes take
    codes 0 and 15, and the V step is (max - min)/15."""
    k, v = synth.kv_stream(workload, 2, 0, 128, D)
    a = oracle.compress_unit(k, v)
    b = oracle.compress_unit(k, v, v_bits=4)
    ua = oracle.unpack_record(a["record"], D)
    ub = oracle.unpack_record(b["record"], D, v_bits=4)
    for name in ("k_codes", "k_delta", "k_lo", "k_s", "k_r", "v_s", "v_r"):
        np.testing.assert_array_equal(ua[name], ub[name], err_msg=name)
    gv = D // min(D, 128)
    gw = D // gv
    vpre, vc = b["v_vpre"], ub["v_codes"].astype(np.int64)
    assert vc.max() <= 15 and vc.min() >= 0
    y = b["v_delta"].reshape(128, gv).repeat(gw, 1) * vpre + b["v_lo"].reshape(128, gv).repeat(gw, 1)
    recon = b["v_delta"].reshape(128, gv).repeat(gw, 1) * vc + b["v_lo"].reshape(128, gv).repeat(gw, 1)
    half = b["v_delta"].reshape(128, gv).repeat(gw, 1) / 2
    assert np.all(np.abs(y - recon) <= half * (1 + 1e-12) + 1e-300)
    for t in range(0, 128, 17):
        for g in range(gv):
            seg = vpre[t, g * gw:(g + 1) * gw]
            codes = vc[t, g * gw:(g + 1) * gw]
            assert codes[np.argmin(seg)] == 0 and codes[np.argmax(seg)] == 15
    # and the stored V offset and step are the group minimum and range / 15
    yv = y.reshape(128, gv, gw)
    np.testing.assert_allclose(b["v_lo"].reshape(128, gv), yv.min(-1), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b["v_delta"].reshape(128, gv), (yv.max(-1) - yv.min(-1)) / 15,
                               rtol=1e-12, atol=1e-12)


def test_v4_dequant_distortion_bound(oracle):
    """Unrotated V rows of a k4v4 record are within the norm of the per-element
    bounds r s delta / 2 of the exact rows (orthonormal H), and tighter than
    the k4v2 record's on the same tile."""
    D = 128
    k, v = synth.kv_stream("qwen3_8b_decode", 3, 0, 128, D)
    b = oracle.compress_unit(k, v, v_bits=4)
    _, vv = oracle.dequant_record(b["record"], D, v_bits=4)
    _, v2 = oracle.dequant_record(oracle.compress_unit(k, v)["record"], D)
    bound = np.sqrt(((b["v_r"][:, None] * b["v_s"][None, :] * b["v_delta"][:, None] / 2) ** 2).sum(1))
    err = np.linalg.norm(vv - v.astype(np.float64), axis=1)
    assert np.all(err <= bound * (1 + 1e-9))
    assert np.linalg.norm(vv - v) < np.linalg.norm(v2 - v)


# ------------------------------------------- c4 variant: 3-bit values (k4v3)
@pytest.mark.parametrize("D", [64, 128, 256])
def test_v3_record_size(oracle, D):
    """Token rows of 3 D / 8 bytes: 16 D bytes more than the k4v2 record."""
    assert oracle.record_bytes(D, v_bits=3) - oracle.record_bytes(D) == 16 * D
    assert oracle.record_bytes(128, v_bits=3) == 18432


def test_v3_pack_bit_order_hand_built(oracle):
    """Each token's V codes are a little-endian bit stream, channel c at bits
    3c..3c+2: code 5 = 0b101 at channel 2 of token 0 sets stream bits 6 and 8
    (bit 6 of byte 0, bit 0 of byte 1: a code straddling two bytes); code 6 =
    0b110 at the last channel of token 3 sets the top two bits of that row's
    last byte."""
    D = 128
    z = lambda n: np.zeros(n)
    vc = np.zeros((128, D), np.uint8)
    vc[0, 2] = 5
    vc[3, D - 1] = 6
    rec = oracle.pack_record(D, np.zeros((128, D), np.uint8), vc, z(D), z(D), z(D), z(128),
                             z(128), z(128), z(128), z(D), v_bits=3)
    voff = 64 * D
    row = 3 * D // 8
    assert rec[voff] == 0x40 and rec[voff + 1] == 0x01
    assert rec[voff + 3 * row + row - 1] == 0xC0
    assert np.count_nonzero(rec) == 3


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("scale_bits", [32, 16])
def test_v3_pack_unpack_roundtrip(oracle, D, scale_bits):
    rng = np.random.default_rng(D + 3 + scale_bits)
    gv = D // min(D, 128)
    f32 = lambda n: rng.standard_normal(n).astype(np.float16).astype(np.float64)
    args = dict(k_codes=rng.integers(0, 16, (128, D)).astype(np.uint8),
                v_codes=rng.integers(0, 8, (128, D)).astype(np.uint8),
                k_delta=f32(D), k_lo=f32(D), k_s=f32(D), k_r=f32(128),
                v_delta=f32(128 * gv), v_lo=f32(128 * gv), v_r=f32(128), v_s=f32(D))
    rec = oracle.pack_record(D, scale_bits=scale_bits, v_bits=3, **args)
    assert rec.size == oracle.record_bytes(D, scale_bits, 3)
    back = oracle.unpack_record(rec, D, scale_bits, v_bits=3)
    for name, val in args.items():
        np.testing.assert_array_equal(back[name], val, err_msg=name)


@pytest.mark.parametrize("workload,D", [("qwen3_8b_decode", 128), ("batched_d256_decode", 256)])
def test_v3_compress_keeps_keys_and_bounds_value_error(oracle, workload, D):
    """The k4v3 record: the K half is the k4v2 record's; V is quantised to 8
    levels per token group (step (max - min)/7), every normalised V element
    is within delta/2 of its reconstruction, and the group extremes take
    codes 0 and 7."""
    k, v = synth.kv_stream(workload, 4, 0, 128, D)
    a = oracle.compress_unit(k, v)
    b = oracle.compress_unit(k, v, v_bits=3)
    ua = oracle.unpack_record(a["record"], D)
    ub = oracle.unpack_record(b["record"], D, v_bits=3)
    for name in ("k_codes", "k_delta", "k_lo", "k_s", "k_r", "v_s", "v_r"):
        np.testing.assert_array_equal(ua[name], ub[name], err_msg=name)
    gv = D // min(D, 128)
    gw = D // gv
    vpre, vc = b["v_vpre"], ub["v_codes"].astype(np.int64)
    assert vc.max() <= 7 and vc.min() >= 0
    dl = b["v_delta"].reshape(128, gv).repeat(gw, 1)
    lo = b["v_lo"].reshape(128, gv).repeat(gw, 1)
    y, recon = dl * vpre + lo, dl * vc + lo
    assert np.all(np.abs(y - recon) <= dl / 2 * (1 + 1e-12) + 1e-300)
    for t in range(0, 128, 13):
        for g in range(gv):
            seg, codes = vpre[t, g * gw:(g + 1) * gw], vc[t, g * gw:(g + 1) * gw]
            assert codes[np.argmin(seg)] == 0 and codes[np.argmax(seg)] == 7
    yv = y.reshape(128, gv, gw)
    np.testing.assert_allclose(b["v_delta"].reshape(128, gv), (yv.max(-1) - yv.min(-1)) / 7,
                               rtol=1e-12, atol=1e-12)


def test_v3_distortion_between_v2_and_v4(oracle):
    """Unrotated V rows of a k4v3 record are within the norm of r s delta / 2
    of the exact rows, and their error lies between the k4v2 and k4v4
    records' on the same tile."""
    D = 128
    k, v = synth.kv_stream("qwen3_8b_decode", 5, 0, 128, D)
    err = {}
    for vb in (2, 3, 4):
        b = oracle.compress_unit(k, v, v_bits=vb)
        _, vv = oracle.dequant_record(b["record"], D, v_bits=vb)
        e = np.linalg.norm(vv - v.astype(np.float64), axis=1)
        if vb == 3:
            bound = np.sqrt(((b["v_r"][:, None] * b["v_s"][None, :] * b["v_delta"][:, None] / 2)
                             ** 2).sum(1))
            assert np.all(e <= bound * (1 + 1e-9))
        err[vb] = np.linalg.norm(e)
    assert err[4] < err[3] < err[2]


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("scale_bits", [32, 16])
@pytest.mark.parametrize("v_bits", [2, 3, 4])
def test_dequant_is_the_scaled_affine_code_rotated_back(oracle, D, scale_bits, v_bits):
    """Issue #180, "Algorithm (per 128-token tile)": a stored row is rebuilt as
    r_t s_c (delta code + lo) in the rotated space, keys with per-channel
    (delta, lo), values with per-token (delta, lo) for each 128-channel group,
    then rotated back by the orthonormal Sylvester-Hadamard matrix (scipy).
    Written here from the record's unpacked fields, at every value width and
    both scale widths."""
    k, v = synth.kv_stream("batched_d256_decode" if D == 256 else "qwen3_8b_decode", 3, 1, 128, D)
    rec = oracle.compress_unit(k, v, scale_bits=scale_bits, v_bits=v_bits)["record"]
    u = oracle.unpack_record(rec, D, scale_bits, v_bits)
    kh, vh = oracle.dequant_record(rec, D, scale_bits, v_bits)
    H = scipy.linalg.hadamard(D) / np.sqrt(D)
    kc, vc = u["k_codes"].astype(np.float64), u["v_codes"].astype(np.float64)
    k_rot = u["k_r"][:, None] * u["k_s"][None, :] * (u["k_delta"][None, :] * kc + u["k_lo"][None, :])
    gv = D // 128
    g = np.arange(D) // 128
    vd = u["v_delta"].reshape(128, gv)[:, g]
    vl = u["v_lo"].reshape(128, gv)[:, g]
    v_rot = u["v_r"][:, None] * u["v_s"][None, :] * (vd * vc + vl)
    assert vc.max() <= 2 ** v_bits - 1 and kc.max() <= 15
    np.testing.assert_allclose(kh, k_rot @ H, rtol=1e-10, atol=1e-12 * np.abs(kh).max())
    np.testing.assert_allclose(vh, v_rot @ H, rtol=1e-10, atol=1e-12 * np.abs(vh).max())


def test_prefill_window_token_sits_after_the_tiles(oracle):
    """c8 positions with tiles and a window: tile k holds positions
    [128k, 128k + 128), window token j position 128 n_tiles + j (PR #434,
    commit 6040076: the window stages the newest tokens). Perturbing window
    token j leaves every query row at an earlier position bit-identical,
    including rows inside the tiles. With a zero query (equal weights over the
    visible tokens) a row at position p >= 128 n_tiles + j moves by exactly
    the value's change divided by p + 1."""
    Hkv, Hq, D, n = 1, 2, 64, 424
    ks, vs = synth.kv_layer("qwen3_8b_decode", 1, Hkv, n, D)
    sm = oracle.CacheStateMachine(Hkv, D, W=128)
    for pos in range(n):
        sm.append(ks[:, pos:pos + 1].transpose(1, 0, 2), vs[:, pos:pos + 1].transpose(1, 0, 2))
    assert sm.n_tiles == 3 and sm.win_len == 40
    rb = oracle.record_bytes(D)
    pool = np.concatenate([r[0] for r in sm.records])
    table = (np.arange(sm.n_tiles, dtype=np.int64) * rb)[None, :]
    wk, wv = sm.window(0)
    win_k = np.zeros((1, 64, D), np.float32)
    win_v = np.zeros((1, 64, D), np.float32)
    win_k[0, :40], win_v[0, :40] = wk, wv
    pos0, C = 300, n - 300
    q = synth.queries("qwen3_8b_decode", 1, (C, Hq, D))
    q[:, 0] = 0.0  # head 0: equal weights
    base = oracle.prefill_attention(q, pos0, pool, table, sm.n_tiles, win_k, win_v, 0, 40, 1 / 8)
    j = 10
    pk, pv = win_k.copy(), win_v.copy()
    pk[0, j] += 3.0
    pv[0, j] -= 5.0
    moved = oracle.prefill_attention(q, pos0, pool, table, sm.n_tiles, pk, pv, 0, 40, 1 / 8)
    p_j = 128 * sm.n_tiles + j
    dv = pv[0, j].astype(np.float64) - win_v[0, j].astype(np.float64)
    for (i, h), o in base.items():
        p = pos0 + i
        if p < p_j:
            np.testing.assert_array_equal(moved[(i, h)], o)
        elif h == 0:
            np.testing.assert_allclose(moved[(i, h)] - o, dv / (p + 1), rtol=1e-9, atol=1e-13)


def test_decode_batch_rows_are_independent(oracle):
    """c7 over a batch: each sequence reads only its own table row, tile count,
    window ring, start and length. Two sequences with different tile counts,
    windows and ring starts give, head by head, the result of decoding each
    sequence alone."""
    Hkv, G, D, cap = 2, 2, 64, 256
    Hq = Hkv * G
    rb = oracle.record_bytes(D)
    seqs = []
    for b, (n, start) in enumerate([(128 * 3 + 37, 200), (128 + 5, 17)]):
        ks, vs = synth.kv_layer("qwen3_8b_decode", 5 + b, Hkv, n, D)
        sm = oracle.CacheStateMachine(Hkv, D, W=128)
        sm.append(ks.transpose(1, 0, 2), vs.transpose(1, 0, 2))
        win_k = np.zeros((Hkv, cap, D), np.float32)
        win_v = np.zeros((Hkv, cap, D), np.float32)
        for h in range(Hkv):
            wk, wv = sm.window(h)
            for w in range(sm.win_len):
                win_k[h, (start + w) % cap], win_v[h, (start + w) % cap] = wk[w], wv[w]
        seqs.append((sm, win_k, win_v, start))
    max_tiles = max(s[0].n_tiles for s in seqs)
    # one pool: sequence b's tile t of KV head h at record ((b * Hkv + h) * max_tiles + t)
    pool = np.zeros(2 * Hkv * max_tiles * rb, np.uint8)
    table = np.zeros((2, Hkv, max_tiles), np.int64)
    for b, (sm, _, _, _) in enumerate(seqs):
        for t in range(sm.n_tiles):
            for h in range(Hkv):
                off = ((b * Hkv + h) * max_tiles + t) * rb
                pool[off:off + rb] = sm.records[t][h]
                table[b, h, t] = off
    q = synth.queries("qwen3_8b_decode", 9, (2, Hq, D))
    both = oracle.decode_attention(q, pool, table, [s[0].n_tiles for s in seqs],
                                   np.stack([s[1] for s in seqs]), np.stack([s[2] for s in seqs]),
                                   [s[3] for s in seqs], [s[0].win_len for s in seqs], 1 / 8)
    for b, (sm, win_k, win_v, start) in enumerate(seqs):
        alone = oracle.decode_attention(q[b:b + 1], pool, table[b:b + 1], [sm.n_tiles],
                                        win_k[None], win_v[None], [start], [sm.win_len], 1 / 8)
        for h in range(Hq):
            np.testing.assert_array_equal(both[(b, h)], alone[(0, h)])
