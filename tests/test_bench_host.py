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
