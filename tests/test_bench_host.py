"""Host-side helpers of bench.py that need no GPU."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_clock_summary():
    lines = [
        "2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "2040, 2070, 1350.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbage line",
        "[N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2055, 2070, 1200.0, 0x0000000000000008, Active, Not Active, Not Active, Not Active",
    ]
    got = bench.ClockSampler.summarize(lines)
    assert got == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0,
                   "reasons": ["hw_slowdown", "sw_power_cap"], "samples": 3}
    assert bench.ClockSampler.summarize([]) is None


def test_traffic_table_names_existing_sources():
    """Each recorded ncu traffic figure is tied to a kernel source file that exists."""
    for name, src in (("decode_split", "decode.cu"), ("compress", "compress.cu")):
        entry = bench.NCU_TRAFFIC[name]
        assert len(entry["src_sha"]) == 16 and entry["bytes"] > 0
        assert len(bench.src_sha(src)) == 16


def test_compress_parity_sample_counts():
    """The bench's compress parity sample, fed the oracle's own records as the
    device's: no code differs, scales agree to fp32 storage, every offset lo
    meets 1e-6 relative to |lo| itself; a perturbed lo is counted as outside."""
    import numpy as np
    import oracle
    from kv_cache_quantization_token_gb300 import synth
    D = bench.D
    ks, vs = synth.kv_layer("qwen3_8b_decode", 0, 1, 128 * 4, D)
    k, v = np.ascontiguousarray(ks[0]), np.ascontiguousarray(vs[0])
    refs = [oracle.compress_unit(k[128 * u:128 * u + 128], v[128 * u:128 * u + 128]) for u in range(4)]
    recs = np.frombuffer(b"".join(bytes(r["record"]) for r in refs), np.uint8).copy()
    rb = recs.size // 4
    got = bench.oracle_compress_baseline({"k": k, "v": v, "records": recs, "record_bytes": rb})
    cmp_ = got["gpu_vs_oracle"]
    assert cmp_["codes"] == 4 * 2 * 128 * D and cmp_["differing"] == 0
    assert cmp_["scale_rel_err_max"] < 1e-6
    lo = cmp_["lo"]
    assert lo["values"] == 4 * (D + 128 * (D // min(D, 128)))
    assert lo["within_1e-6_of_lo"] == lo["values"] and lo["outside_1e-6"] == 0
    # one K offset of unit 0 moved by 1e-3 of the tile's scale: counted
    # outside the bound, and nothing else changes
    f = oracle.unpack_record(recs[:rb], D)
    f["k_lo"][0] += 1e-3 * max(abs(f["k_lo"][0]), abs(f["k_delta"][0]), 1.0)
    recs[:rb] = oracle.pack_record(D, f["k_codes"], f["v_codes"], f["k_delta"], f["k_lo"], f["k_s"],
                                   f["k_r"], f["v_delta"], f["v_lo"], f["v_r"], f["v_s"])
    got2 = bench.oracle_compress_baseline({"k": k, "v": v, "records": recs, "record_bytes": rb})
    lo2 = got2["gpu_vs_oracle"]["lo"]
    assert lo2["outside_1e-6"] == 1 and lo2["within_1e-6_only_widened"] == 0
    assert got2["gpu_vs_oracle"]["differing"] == 0
