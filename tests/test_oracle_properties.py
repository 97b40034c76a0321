"""Property-based pins of the oracle (hypothesis; skipped where it is not
installed): random inputs checked against the definitions the pages fix --
the RTN error bound and range (SharpInference issue #180, step 3), the
token-std normalisation Sinkhorn ends with and its factorised form (step 2),
the orthonormal self-inverse Walsh-Hadamard rotation (step 1), and the
record pack / unpack round trip of every layout variant."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402

SETTINGS = settings(max_examples=40, deadline=None, derandomize=True)


@SETTINGS
@given(st.integers(0, 2**31 - 1), st.integers(1, 300), st.sampled_from([2, 4]),
       st.floats(1e-3, 1e3), st.booleans())
def test_rtn_bound_and_range(seed, n, bits, spread, repeat):
    rng = np.random.default_rng(seed)
    y = rng.standard_normal(n) * spread + rng.standard_normal() * spread
    if repeat:  # ties and duplicates: a few distinct values only
        y = np.round(y / spread * 2) * spread / 2
    delta, lo, codes, vpre = oracle.rtn_group(y, bits)
    top = (1 << bits) - 1
    assert codes.min() >= 0 and codes.max() <= top
    assert lo == y.min()
    if delta == 0:
        assert np.all(codes == 0) and np.all(y == lo)
    else:
        assert delta == pytest.approx((y.max() - y.min()) / top, rel=1e-15)
        err = np.abs(y - (delta * codes + lo))
        assert np.all(err <= delta / 2 * (1 + 1e-12))
        assert codes[np.argmin(y)] == 0 and codes[np.argmax(y)] == top


@SETTINGS
@given(st.integers(0, 2**31 - 1), st.sampled_from([8, 16, 32, 128]),
       st.sampled_from([8, 16, 64, 128]), st.integers(1, 6))
def test_sinkhorn_factorisation_and_unit_token_std(seed, T, D, iters):
    rng = np.random.default_rng(seed)
    Y = rng.standard_normal((T, D)) * np.exp(rng.standard_normal(D))[None, :] \
        * np.exp(0.5 * rng.standard_normal(T))[:, None]
    s, r, yn = oracle.sinkhorn(Y, iters)
    assert np.all(s > 0) and np.all(r > 0)
    np.testing.assert_allclose(yn, Y / (r[:, None] * s[None, :]), rtol=1e-12, atol=0)
    np.testing.assert_allclose(yn.std(axis=1), 1.0, rtol=1e-12)  # the last step is a token step


@SETTINGS
@given(st.integers(0, 2**31 - 1), st.sampled_from([64, 128, 256]), st.integers(1, 5))
def test_wht_orthonormal_and_self_inverse(seed, D, rows):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, D)).astype(np.float32)
    y = oracle.wht_rows(x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x.astype(np.float64), axis=1),
                               rtol=1e-12)
    np.testing.assert_allclose(oracle.wht_rows(y.astype(np.float32)), x, rtol=0, atol=1e-5)


@SETTINGS
@given(st.integers(0, 2**31 - 1), st.sampled_from([64, 128, 256]), st.sampled_from([32, 16]),
       st.sampled_from([2, 3, 4]))
def test_record_round_trip_every_layout(seed, D, scale_bits, v_bits):
    rng = np.random.default_rng(seed)
    T, gv = 128, D // min(D, 128)
    kc = rng.integers(0, 16, (T, D)).astype(np.uint8)
    vc = rng.integers(0, 1 << v_bits, (T, D)).astype(np.uint8)
    sc = {n: rng.standard_normal(m) for n, m in
          (("k_delta", D), ("k_lo", D), ("k_s", D), ("k_r", T), ("v_delta", T * gv),
           ("v_lo", T * gv), ("v_r", T), ("v_s", D))}
    rec = oracle.pack_record(D, kc, vc, *[sc[n] for n in ("k_delta", "k_lo", "k_s", "k_r",
                                                           "v_delta", "v_lo", "v_r", "v_s")],
                             scale_bits=scale_bits, v_bits=v_bits)
    assert rec.size == oracle.record_bytes(D, scale_bits, v_bits)
    u = oracle.unpack_record(rec, D, scale_bits, v_bits)
    np.testing.assert_array_equal(u["k_codes"], kc)
    np.testing.assert_array_equal(u["v_codes"], vc)
    for n, a in sc.items():
        want = (a.astype(np.float32) if scale_bits == 32 else a.astype(np.float16)).astype(np.float64)
        np.testing.assert_array_equal(u[n], want, err_msg=n)


@settings(max_examples=15, deadline=None, derandomize=True)
@given(st.lists(st.integers(1, 200), min_size=1, max_size=12), st.sampled_from([128, 256]))
def test_tiles_independent_of_chunking(chunks, W):
    """Any sequence of chunk sizes promotes the same tiles as token-at-a-time
    appends (PR #434: tiles do not depend on the chunking), and the window
    keeps its invariant: fewer than W tokens, at least W - 128 once a tile
    was promoted."""
    Hkv, D = 1, 64
    n = sum(chunks)
    ks, vs = synth_kv(n, D)
    ref = oracle.CacheStateMachine(Hkv, D, W=W)
    for i in range(n):
        ref.append(ks[i:i + 1], vs[i:i + 1])
    sm = oracle.CacheStateMachine(Hkv, D, W=W)
    i0 = 0
    for c in chunks:
        sm.append(ks[i0:i0 + c], vs[i0:i0 + c])
        i0 += c
        assert sm.win_len < W
        if sm.n_tiles:
            assert sm.win_len >= W - 128
    assert sm.n_tiles == ref.n_tiles == ((n - W) // 128 + 1 if n >= W else 0)
    for t in range(sm.n_tiles):
        np.testing.assert_array_equal(sm.records[t][0], ref.records[t][0])


def synth_kv(n, D):
    from kv_cache_quantization_token_gb300 import synth
    k, v = synth.kv_layer("single_tile", 3, 1, n, D)
    return k.transpose(1, 0, 2).copy(), v.transpose(1, 0, 2).copy()
