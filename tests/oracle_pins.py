"""Pins of the CPU oracle: facts fixed by the pages or by mathematics.

Each ``pin_*`` takes the oracle module (so a planted mistake can be fed in)
and raises AssertionError when the oracle disagrees. None re-types the
oracle's formulas: they use hand-derived values, closed forms for special
inputs, brute force, invariants, or a textbook routine a special case reduces
to. Used by test_oracle_pins.py (real oracle) and by the planted-mistake test
(mutated copies of it).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

from int4_routed_expert_moe_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _silu(v):
    return v / (1.0 + math.exp(-v))


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _num(v):
    return float(v) if not isinstance(v, str) else float(v.replace("inf", "inf"))


# ---- storage ---------------------------------------------------------------
def pin_nibble_order(orc):
    # byte 0x21: element 0 = low nibble 1, element 1 = high nibble 2.
    got = orc.unpack_codes(np.array([[0x21, 0xF0], [0x0F, 0x80]], dtype=np.uint8))
    assert got.tolist() == [[1, 2, 0, 15], [15, 0, 0, 8]], got.tolist()


# Hand case: H=4, I=2, g=2 (two groups along H for gate/up, one along I for down).
HAND = dict(
    q_gate=[[1, 2, 3, 4], [0, 15, 8, 8]],
    s_gate=[[0.5, 0.25], [1.0, 0.125]],
    z_gate=[[0, 2], [8, 8]],
    q_up=[[8, 8, 8, 9], [10, 6, 8, 8]],
    s_up=[[0.5, 0.5], [0.5, 0.5]],
    z_up=[[8, 8], [8, 8]],
    q_down=[[9, 7], [8, 8], [12, 8], [0, 15]],
    s_down=[[1.0], [1.0], [0.25], [0.5]],
    z_down=[[8], [8], [8], [8]],
    x=[1.0, -1.0, 2.0, 0.5],
)
# Dequantised by hand: (q - z) * s per element.
HAND_WG = [[0.5, 1.0, 0.25, 0.5], [-8.0, 7.0, 0.0, 0.0]]
HAND_WU = [[0.0, 0.0, 0.0, 0.5], [1.0, -1.0, 0.0, 0.0]]
HAND_WD = [[1.0, -1.0], [0.0, 0.0], [1.0, 0.0], [-4.0, 3.5]]


def hand_expert():
    f16 = lambda a: np.array(a, dtype=np.float16)
    return {
        "qp_gate": synth.pack_codes(HAND["q_gate"]), "s_gate": f16(HAND["s_gate"]), "z_gate": f16(HAND["z_gate"]),
        "qp_up": synth.pack_codes(HAND["q_up"]), "s_up": f16(HAND["s_up"]), "z_up": f16(HAND["z_up"]),
        "qp_down": synth.pack_codes(HAND["q_down"]), "s_down": f16(HAND["s_down"]), "z_down": f16(HAND["z_down"]),
    }


def pin_dequant_hand(orc):
    e = hand_expert()
    wg, wu, wd = orc.dequantize_expert(e, 2)
    assert np.array_equal(wg, np.array(HAND_WG)), wg
    assert np.array_equal(wu, np.array(HAND_WU)), wu
    assert np.array_equal(wd, np.array(HAND_WD)), wd


def pin_expert_ffn_hand(orc):
    # g = W_g x = [0.25, -15]; u = W_u x = [0.25, 2]; h = silu(g) * u;
    # y = W_d h = [h0 - h1, 0, h0, -4 h0 + 3.5 h1].
    e = hand_expert()
    wg, wu, wd = orc.dequantize_expert(e, 2)
    y = orc.expert_ffn(np.array(HAND["x"]), wg, wu, wd)
    h0 = _silu(0.25) * 0.25
    h1 = _silu(-15.0) * 2.0
    want = [h0 - h1, 0.0, h0, -4.0 * h0 + 3.5 * h1]
    assert np.allclose(y, want, rtol=1e-13, atol=1e-15), (y, want)


def pin_expert_ffn_constant_codes(orc):
    # Every code of a matrix equal to c, one scale s and zero z: every weight
    # is a = (c - z) s, so g_n = a_g S, u_n = a_u S with S = sum(x), h_n the
    # same for all n, and y_m = a_d * I * h. Non-integer z, negative g.
    H, I, g = 256, 128, 64
    r = np.random.default_rng(5)
    x = r.standard_normal(H).astype(np.float16)
    cases = [(3, 7, 12, 8.0, 8.0, 8.0), (12, 2, 5, 4.5, 9.25, 0.0)]
    for cg, cu, cd, zg, zu, zd in cases:
        sg, su, sd = 0.0078125, 0.00390625, 0.005859375
        arrs = {
            "qp_gate": synth.pack_codes(np.full((I, H), cg)), "s_gate": np.full((I, H // g), sg, np.float16), "z_gate": np.full((I, H // g), zg, np.float16),
            "qp_up": synth.pack_codes(np.full((I, H), cu)), "s_up": np.full((I, H // g), su, np.float16), "z_up": np.full((I, H // g), zu, np.float16),
            "qp_down": synth.pack_codes(np.full((H, I), cd)), "s_down": np.full((H, I // g), sd, np.float16), "z_down": np.full((H, I // g), zd, np.float16),
        }
        wg, wu, wd = orc.dequantize_expert(arrs, g)
        y = orc.expert_ffn(x, wg, wu, wd)
        S = float(np.sum(x.astype(np.float64)))
        ag, au, ad = (cg - zg) * sg, (cu - zu) * su, (cd - zd) * sd
        h = _silu(ag * S) * (au * S)
        want = ad * I * h
        assert np.allclose(y, want, rtol=1e-12, atol=1e-300), (y[:3], want)


def pin_group_axis(orc):
    # Constant codes c, zero z, a different scale per group along the row:
    # g_n = (c - z) * sum_G s_G * sum_{c in G} x_c. Distinguishes c // g from
    # c % g and rows from columns.
    H, I, g = 8, 2, 2
    x = np.array([1.0, 2.0, -1.0, 0.5, 3.0, -2.0, 0.25, 1.0])
    s_row = np.array([0.5, 0.25, 2.0, 1.0])
    c, z = 11, 8
    arr_q = synth.pack_codes(np.full((I, H), c))
    s = np.stack([s_row, s_row[::-1]]).astype(np.float16)
    z_ = np.full((I, H // g), z, np.float16)
    w = orc.dequantize(arr_q, s, z_, g)
    gsum = [x[0] + x[1], x[2] + x[3], x[4] + x[5], x[6] + x[7]]
    want0 = (c - z) * sum(s_row[i] * gsum[i] for i in range(4))
    want1 = (c - z) * sum(s_row[::-1][i] * gsum[i] for i in range(4))
    got = w @ x
    assert np.allclose(got, [want0, want1], rtol=1e-14), (got, want0, want1)


def pin_block_bytes(orc):
    # 3*H*I/2 code bytes + 3*(H*I/g) groups * (FP16 scale + FP16 zero).
    assert orc.expert_block_bytes(256, 128, 64) == 55296
    assert orc.expert_block_bytes(2048, 1024, 128) == 3342336
    assert orc.expert_block_bytes(2048, 512, 128) == 1671168


# ---- routing -----------------------------------------------------------------
def pin_route_golden(orc):
    cases = _load("route_cases.json")
    for c in cases["cases"]:
        lg = np.array([[_num(v) for v in row] for row in c["logits"]], dtype=np.float32)
        ids, w = orc.route(lg, c["k"], c["renorm"])
        assert ids.tolist() == c["ids"], (c["name"], ids.tolist())
        assert np.allclose(w, c["weights"], rtol=1e-7, atol=1e-12), (c["name"], w)
    for c in cases["errors"]:
        lg = np.array([[_num(v) for v in row] for row in c["logits"]], dtype=np.float32)
        try:
            orc.route(lg, c["k"], False)
        except ValueError:
            continue
        raise AssertionError(f"{c['name']}: no error")


def pin_route_dense_softmax(orc):
    # k = E with renormalisation: the weights are the dense softmax in the
    # selection order (scipy's softmax is the textbook routine).
    from scipy.special import softmax
    r = np.random.default_rng(11)
    lg = r.standard_normal((5, 16)).astype(np.float32)
    ids, w = orc.route(lg, 16, True)
    for t in range(5):
        ref = softmax(lg[t].astype(np.float64))
        assert np.allclose(w[t], ref[ids[t]], rtol=1e-12), t
        assert sorted(ids[t].tolist()) == list(range(16))


def pin_route_invariants(orc):
    r = np.random.default_rng(12)
    lg = r.standard_normal((40, 64)).astype(np.float32)
    lg[3, 10] = lg[3, 40]  # an exact tie
    for renorm in (False, True):
        ids, w = orc.route(lg, 8, renorm)
        for t in range(40):
            chosen = list(ids[t])
            rest = [e for e in range(64) if e not in chosen]
            # every chosen expert beats every other by (logit desc, index asc)
            worst = min((-float(lg[t, e]), e) for e in rest)
            assert all((-float(lg[t, e]), e) < worst for e in chosen)
            assert all((-float(lg[t, a]), a) < (-float(lg[t, b]), b)
                       for a, b in zip(chosen, chosen[1:]))
            # weight ratios are exp of logit differences
            for a in range(1, 8):
                want = math.exp(float(lg[t, chosen[a]]) - float(lg[t, chosen[0]]))
                assert abs(w[t, a] / w[t, 0] - want) < 1e-12 * max(1.0, want)
            s = float(np.sum(w[t]))
            assert (abs(s - 1.0) < 1e-12) if renorm else (0.0 < s <= 1.0 + 1e-12)


def pin_coverage(orc):
    # lucashiago etapa 3: with each token choosing a uniform random k-subset,
    # the mean number of distinct experts n tokens touch is E(1-(1-k/E)^n).
    E, k, n, trials = 64, 8, 6, 400
    r = np.random.default_rng(13)
    touched = []
    for _ in range(trials):
        lg = r.uniform(0.0, 1.0, (n, E)).astype(np.float32)
        ids, _ = orc.route(lg, k, False)
        touched.append(len(set(ids.reshape(-1).tolist())))
    mean = float(np.mean(touched))
    se = float(np.std(touched)) / math.sqrt(trials)
    want = E * (1 - (1 - k / E) ** n)
    assert abs(mean - want) < 4 * se + 1e-9, (mean, want, se)
    assert abs(orc.expected_touched(E, k, n) - want) < 1e-12


# ---- layer -------------------------------------------------------------------
def pin_layer_dense_bruteforce(orc):
    wl = synth.WORKLOADS["tiny_layer"]
    H, I, E, k, g = wl["H"], wl["I"], wl["E"], wl["k"], wl["g"]
    for zero, renorm in (("eight", True), ("int", False), ("frac", True)):
        experts = {e: synth.expert_arrays(77, 0, e, H, I, g, zero=zero) for e in range(E)}
        x = synth.activations(77, 0, 4, H)
        lg = synth.logits_normal(77, 0, 4, E)
        routed = orc.moe_layer(x, lg, experts, k, renorm, g)["y"]
        dense = orc.moe_layer_dense(x, lg, experts, E, k, renorm, g)
        assert np.allclose(routed, dense, rtol=1e-12, atol=1e-15), zero


def pin_shared_ffn_torch(orc):
    # The FP16 non-routed FFN reduces to torch's silu and matmul in float64.
    import torch
    r = np.random.default_rng(14)
    x = r.standard_normal((3, 32)).astype(np.float16)
    wg = (r.standard_normal((48, 32)) / 6).astype(np.float16)
    wu = (r.standard_normal((48, 32)) / 6).astype(np.float16)
    wd = (r.standard_normal((32, 48)) / 7).astype(np.float16)
    got = orc.shared_ffn(x, wg, wu, wd)
    t = lambda a: torch.from_numpy(a.astype(np.float64))
    ref = (torch.nn.functional.silu(t(x) @ t(wg).T) * (t(x) @ t(wu).T)) @ t(wd).T
    assert np.allclose(got, ref.numpy(), rtol=1e-12, atol=1e-14)


def pin_token_sort(orc):
    r = np.random.default_rng(15)
    T, k, E = 37, 4, 9
    ids = np.stack([r.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    off, ptok, pj = orc.token_sort(ids, E)
    hist = np.bincount(ids.reshape(-1), minlength=E)
    assert off[0] == 0 and off[-1] == T * k
    assert np.array_equal(np.diff(off), hist)
    seen = set()
    for e in range(E):
        pairs = [(int(ptok[p]), int(pj[p])) for p in range(off[e], off[e + 1])]
        assert all(ids[t, j] == e for t, j in pairs)
        assert pairs == sorted(pairs)  # stable: token order, then slot j
        seen.update(pairs)
    assert len(seen) == T * k


# ---- residency ---------------------------------------------------------------
def pin_residency_hand(orc):
    c = _load("residency_hand_trace.json")
    out = orc.residency_sim(c["steps"], c["E"], c["C"], c["S"], c["decay"])
    assert [list(t) for t in out["trace"]] == c["trace"], out["trace"]
    assert out["counts"] == c["counts_after"]
    assert out["slot_of"] == c["slot_of_after"]
    assert (out["hits"], out["misses"], out["evictions"]) == (c["hits"], c["misses"], c["evictions"])


def pin_residency_degenerate(orc):
    # C = E: after the canonical placement nothing ever misses.
    r = np.random.default_rng(16)
    steps = [r.choice(12, 3, replace=False).tolist() for _ in range(50)]
    out = orc.residency_sim(steps, 12, 12, 0, 0.9)
    assert out["misses"] == 0 and out["trace"] == []
    # decay = 1: plain access counts (LFU) with lowest-id ties. With one
    # expert needed per step and C = 1 the resident expert is always the
    # one needed, so every step after a change of id misses exactly once.
    steps = [[3], [3], [1], [1], [1], [3]]
    out = orc.residency_sim(steps, 4, 1, 0, 1.0)
    assert [(t[0], t[1], t[3]) for t in out["trace"]] == [(0, 3, 0), (2, 1, 3), (5, 3, 1)]
    # decay = 1, C = 2: victim = lowest count, ties to the lower id.
    steps = [[2], [2], [3], [0]]
    out = orc.residency_sim(steps, 4, 2, 0, 1.0)
    # t0: counts [0,0,1,0] evict 0 (tie 0,1 -> 0); t1 hit; t2: evict 1 (count 0)
    # t3: counts [1,0,2,1], need 0, candidates {2:2, 3:1} -> evict 3.
    assert [(t[0], t[1], t[3]) for t in out["trace"]] == [(0, 2, 0), (2, 3, 1), (3, 0, 3)]
    # spares: the miss takes the lowest free slot; the victim's slot frees up.
    out = orc.residency_sim([[2], [3]], 4, 2, 1, 0.5)
    assert out["trace"][0] == (0, 2, 2, 0) and out["trace"][1][2] == 0


def pin_hit_ceiling(orc):
    # lucashiago etapa 4: no policy beats the sum of the C largest access
    # probabilities. Single draws (k = 1) with Zipf popularity; and uniform
    # use collapses every policy to C/E.
    E, C, steps = 32, 8, 6000
    r = np.random.default_rng(17)
    p = 1.0 / np.arange(1, E + 1)
    p /= p.sum()
    draws = r.choice(E, size=steps, p=p)
    out = orc.residency_sim([[int(d)] for d in draws], E, C, 0, 0.9)
    rate = out["hits"] / steps
    ceil = orc.hit_ceiling(p, C)
    assert rate <= ceil + 3 * math.sqrt(ceil * (1 - ceil) / steps)
    assert rate > 0.5 * ceil  # the decayed count is far from useless here
    draws = r.integers(0, E, size=steps)
    out = orc.residency_sim([[int(d)] for d in draws], E, C, 0, 0.9)
    rate = out["hits"] / steps
    assert abs(rate - C / E) < 4 * math.sqrt((C / E) * (1 - C / E) / steps)


# ---- cost of non-resident weights --------------------------------------------
def pin_time_model_campaign(orc):
    # The printed residency campaign (claims.json, experiment residency39):
    # per configuration, response time and host-to-device traffic over 36
    # measured responses. Fitted on the two extreme configurations of one
    # model and executor, the model t = t_calc + bytes_out / bandwidth must
    # predict the configurations between them to within 3 %, and a fit on all
    # of them must leave no residual above 2 %.
    d = _load("residency39_campaign.json")
    n_resp = d["contract"]["measuredResponsesPerConfiguration"]
    fams = {}
    for r in d["results"]:
        if r["measuredRequestH2dGiB"] > 0:  # the fully resident rows run another executor
            fams.setdefault((r["model"], r["executor"]), []).append(r)
    assert len(fams) == 3
    for rows in fams.values():
        b = [r["measuredRequestH2dGiB"] * 2.0 ** 30 / n_resp for r in rows]
        t = [r["responseSeconds"] for r in rows]
        lo, hi = b.index(min(b)), b.index(max(b))
        tc, bw = orc.fit_time_model([b[lo], b[hi]], [t[lo], t[hi]])
        assert 3.0 < tc < min(t) and 4e9 < bw < 1e10, (tc, bw)  # seconds, bytes/s
        for bi, ti in zip(b, t):
            assert abs(orc.time_model(tc, bi, bw) / ti - 1.0) < 0.03, (bi, ti)
        tc, bw = orc.fit_time_model(b, t)
        for bi, ti in zip(b, t):
            assert abs(orc.time_model(tc, bi, bw) / ti - 1.0) < 0.02, (bi, ti)
    # No traffic costs nothing beyond the computation.
    assert orc.time_model(0.25, 0.0, 1e9) == 0.25


def pin_expected_outside_bruteforce(orc):
    # Exact mean over every routing of n tokens, each a k-subset of E experts
    # (all equally likely), of the distinct touched experts outside the
    # resident set {0..C-1}.
    import itertools
    for E, C, k, n in ((5, 2, 2, 2), (6, 3, 1, 3), (4, 1, 3, 2)):
        subsets = list(itertools.combinations(range(E), k))
        total = count = 0
        for choice in itertools.product(subsets, repeat=n):
            touched = set().union(*choice)
            total += sum(1 for e in touched if e >= C)
            count += 1
        assert abs(orc.expected_outside(E, C, k, n) - total / count) < 1e-12, (E, C, k, n)


def pin_residency_prefetch_hand(orc):
    # Hand-derived trace (tests/golden/residency_prefetch_trace.json): a
    # staged miss keeps its spare slot, unused staged copies go back to the
    # free slots, prefetch stops when no slot is free.
    c = _load("residency_prefetch_trace.json")
    lay = orc.ResidencyLayer(c["E"], c["C"], c["S"], c["decay"], c["policy"])
    trace, staged = [], []
    step = 0
    for op in c["ops"]:
        if op["op"] == "prefetch":
            staged.append(len(lay.prefetch(op["ids"])))
        else:
            for (e, slot, victim) in lay.step(op["ids"]):
                trace.append([step, e, slot, victim])
            step += 1
    assert staged == [op["staged"] for op in c["ops"] if op["op"] == "prefetch"], staged
    assert trace == c["trace"], trace
    assert list(lay.slot_of) == c["slot_of_after"]
    assert [float(v) for v in lay.counts] == c["counts_after"]
    assert (lay.hits, lay.misses, lay.evictions, lay.prefetched, lay.prefetch_copies) == (
        c["hits"], c["misses"], c["evictions"], c["prefetched"], c["prefetch_copies"])


ALL_PINS = [
    pin_nibble_order, pin_dequant_hand, pin_expert_ffn_hand,
    pin_expert_ffn_constant_codes, pin_group_axis, pin_block_bytes,
    pin_route_golden, pin_route_dense_softmax, pin_route_invariants,
    pin_coverage, pin_layer_dense_bruteforce, pin_shared_ffn_torch,
    pin_token_sort, pin_residency_hand, pin_residency_degenerate,
    pin_hit_ceiling, pin_time_model_campaign, pin_expected_outside_bruteforce,
    pin_residency_prefetch_hand,
]
