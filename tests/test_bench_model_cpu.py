"""Host arithmetic of the benchmark and the workload generator (CPU only):
the partial-residency line's time model against the oracle's definition, and
the Zipf popularity the decode workloads are drawn with."""
import math
import os
import sys

import numpy as np

from int4_routed_expert_moe_gb300 import synth
from oracle import moe_oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_time_model_line_matches_the_oracle_model():
    # Runs made from the model itself: t_calc = 0.9 ms, 80 GB/s; the fit on
    # the two extremes must recover both and predict the middle run exactly.
    t_calc, bw, Ktm, K = 0.9e-3, 80e9, 256, 1536
    b_low, b_main = 2.7e8, 8.66e7

    def run(steps, bytes_per_token):
        t = moe_oracle.time_model(t_calc, bytes_per_token, bw)
        return {"ms": t * steps * 1e3, "bytes_out": bytes_per_token * steps}

    full, low, main = run(Ktm, 0.0), run(Ktm, b_low), run(K, b_main)
    main["ms"] *= 1.05  # the measured run is 5 % slower than the model
    tm = bench.time_model_line(full, low, main, K, Ktm, 64, 0)
    fit_tc, fit_bw = moe_oracle.fit_time_model([0.0, b_low], [t_calc, moe_oracle.time_model(t_calc, b_low, bw)])
    assert math.isclose(tm["t_calc_us"], fit_tc * 1e6, rel_tol=1e-6)
    assert math.isclose(tm["bandwidth_gbs"], fit_bw / 1e9, rel_tol=1e-6)
    want = 1.0 / moe_oracle.time_model(t_calc, b_main, bw)
    assert math.isclose(tm["predicted_tok_s"], want, rel_tol=1e-4)
    assert math.isclose(tm["pred_over_meas"], 1.05, rel_tol=1e-3)
    assert tm["endpoints_tok_s"] == {"64": round(1 / t_calc, 2), "0": round(1 / (t_calc + b_low / bw), 2)}


def test_zipf_logits_pick_ranks_with_the_stated_popularity():
    # Gumbel-top-k: the first choice is a draw with P(rank r) = r^-a / sum_r r^-a.
    E, alpha, T = 16, 1.0, 40000
    lg = synth.logits_zipf(11, 0, 0, T, E, alpha)
    ranks = synth.zipf_ranks(11, 0, E)
    assert sorted(ranks.tolist()) == list(range(1, E + 1))
    first = np.argmax(lg, axis=1)
    freq = np.bincount(ranks[first] - 1, minlength=E) / T
    p = np.arange(1, E + 1, dtype=np.float64) ** -alpha
    p /= p.sum()
    sigma = np.sqrt(p * (1 - p) / T)
    assert np.all(np.abs(freq - p) < 5 * sigma), (freq, p)


def test_uniform_zipf_exponent_gives_uniform_choices():
    E, T = 8, 40000
    lg = synth.logits_zipf(12, 1, 0, T, E, 0.0)
    freq = np.bincount(np.argmax(lg, axis=1), minlength=E) / T
    sigma = math.sqrt((1 / E) * (1 - 1 / E) / T)
    assert np.all(np.abs(freq - 1 / E) < 5 * sigma), freq
