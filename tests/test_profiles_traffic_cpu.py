"""bench.py's DRAM-traffic constants against the committed ncu summaries (CPU).

`roofline.traffic` of each bench line is scaled from ncu DRAM counters that
profiles/ records for the current kernels; the constants in bench.py and the
tables in profiles/ must be the same numbers, so a kernel change that
refreshes one and not the other fails here."""
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402

UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}


def kernel_tables(name):
    """[(heading, read_bytes, write_bytes)] of every metric table in a profile."""
    text = open(os.path.join(ROOT, "profiles", name)).read()
    out = []
    for block in re.split(r"\n### ", text)[1:]:
        head = block.splitlines()[0].strip()
        vals = {}
        for m in re.finditer(r"\| dram__bytes_(read|write)\.sum \| ([0-9.]+) (\w+) \|", block):
            vals[m.group(1)] = float(m.group(2)) * UNITS[m.group(3)]
        if vals:
            out.append((head, round(vals.get("read", 0)), round(vals.get("write", 0))))
    return out


def test_olmoe_decode_traffic_matches_profile():
    t = kernel_tables("decode_stream_kernel_olmoe_decode.md")
    head, rd, wr = t[0]  # the full capture (the second table is the warm-cache one)
    assert head.startswith("decode_stream_kernel")
    assert bench.DECODE_DRAM_RATIO["olmoe_decode"] == pytest.approx((rd + wr) / 26_738_688, rel=1e-9)


def test_large_fanout_decode_traffic_matches_profile():
    t = dict((h.split(":")[0], (r, w)) for h, r, w in kernel_tables("decode_stream_kernel_large_fanout_b1_b16.md"))
    rd, wr = t["T = 1"]
    assert bench.DECODE_DRAM_RATIO["large_fanout_b1"] == pytest.approx((rd + wr) / 16_711_680, rel=1e-9)
    rd, wr = t["T = 16"]
    assert bench.DECODE_DRAM_RATIO["large_fanout_b16"] == pytest.approx((rd + wr) / 145_391_616, rel=1e-9)


def test_batch256_grouped_traffic_matches_profile():
    t = kernel_tables("grouped_path_large_fanout_b256.md")
    names = [h for h, _, _ in t]
    assert len(t) == 6 and any("route" in n for n in names) and any("combine" in n for n in names), names
    total = sum(r + w for _, r, w in t)
    assert bench.DECODE_DRAM_RATIO["large_fanout_b256"] == pytest.approx(total / 630_030_336, rel=1e-9)


def test_prefill_gemm_traffic_matches_profile():
    t = kernel_tables("prefill_olmoe_grouped_and_shared_kernels.md")
    gemms = [(h, r, w) for h, r, w in t if h.startswith("grouped_gemm_kernel")]
    assert [h for h, _, _ in gemms[:2]] == ["grouped_gemm_kernel<2>", "grouped_gemm_kernel<1>"]
    assert bench.PREFILL_GEMM_DRAM_BYTES == sum(r + w for _, r, w in gemms[:2])
