"""The partial-residency benchmark line in both modes, at a few steps: it runs,
its bookkeeping is consistent, and the time model's fields are present
(needs a GB300)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("mode,slots,prefetch", [("zerocopy", 30, 0), ("copy", 30, 0), ("copy", 30, 4)])
def test_partial_bench_line(mode, slots, prefetch):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "olmoe_partial",
                          "--mode", mode, "--slots", str(slots), "--prefetch", str(prefetch),
                          "--steps", "24", "--warmup", "3"],
                         capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["config"]["mode"] == mode and line["config"]["slots"] == slots
    assert line["value"] > 0 and line["steps"] == 24
    res, tm = line["residency"], line["time_model"]
    assert 0.0 < res["hit_rate"] < 1.0
    # 16 layers x 8 distinct experts per token: hits + misses per token = 128.
    assert 0.0 < res["misses_per_token"] < 128.0
    assert tm["t_calc_us"] > 0 and tm["bandwidth_gbs"] > 0 and tm["predicted_tok_s"] > 0
    assert line["gpu_launches"] > 0
    if prefetch:
        assert line["config"]["prefetch_spares"] == prefetch
        assert res["prefetch_copies_per_token"] > 0
