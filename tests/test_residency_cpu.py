"""Residency manager decisions (host logic, dry-run mode: no GPU) against the
oracle's policy model: bit-exact traces, counts, slot tables and statistics."""
import json
import os

import numpy as np
import pytest

from int4_routed_expert_moe_gb300 import synth
from oracle import moe_oracle
from tests._lib import ROOT, binding

moe = binding()


def dry(E, C, S, decay, L=1, max_ids=8):
    cfg = dict(layers=L, experts=E, slots=C, spares=S, max_ids_per_step=max_ids, dry_run=1,
               block_bytes=4096, decay=decay)
    return moe.moe_residency_create(cfg, None, None, None)


def test_hand_trace_matches_golden():
    c = json.load(open(os.path.join(ROOT, "tests", "golden", "residency_hand_trace.json")))
    h = dry(c["E"], c["C"], c["S"], c["decay"], max_ids=1)
    try:
        for ids in c["steps"]:
            moe.moe_residency_prepare(h, 0, ids)
        tr = [[s, e, sl, v] for (s, l, e, sl, v) in moe.moe_residency_trace(h)]
        assert tr == c["trace"]
        assert moe.moe_residency_counts(h, 0, c["E"]).tolist() == c["counts_after"]
        assert moe.moe_residency_slot_table(h, 0, c["E"]).tolist() == c["slot_of_after"]
        st = moe.moe_residency_get_stats(h, 0)
        assert (st["hits"], st["misses"], st["evictions"]) == (c["hits"], c["misses"], c["evictions"])
        assert st["h2d_bytes"] == 0  # dry run copies nothing
    finally:
        moe.moe_residency_destroy(h)


@pytest.mark.parametrize("E,C,S,k,T,decay,alpha", [
    (64, 30, 0, 8, 1, 0.9, 1.0),     # the OLMoE partial-residency shape
    (64, 30, 2, 8, 1, 0.9, 1.0),     # with spare slots
    (64, 40, 0, 8, 4, 0.9, 1.0),     # batched decode
    (32, 12, 0, 4, 2, 1.0, 0.5),     # decay 1: plain counts
    (64, 16, 1, 8, 1, 0.5, 0.0),     # uniform popularity
])
def test_policy_matches_oracle(E, C, S, k, T, decay, alpha):
    L, steps = 2, 300
    h = dry(E, C, S, decay, L=L, max_ids=T * k)
    try:
        per_layer = {l: [] for l in range(L)}
        for step in range(steps):
            for l in range(L):
                lg = synth.logits_zipf(9, l, step, T, E, alpha)
                ids, _ = moe_oracle.route(lg, k, False)
                flat = ids.reshape(-1).tolist()
                per_layer[l].append(flat)
                moe.moe_residency_prepare(h, l, flat)
        trace = moe.moe_residency_trace(h)
        for l in range(L):
            ref = moe_oracle.residency_sim(per_layer[l], E, C, S, decay)
            got = [(s, e, sl, v) for (s, ll, e, sl, v) in trace if ll == l]
            assert got == [tuple(t) for t in ref["trace"]]
            assert moe.moe_residency_counts(h, l, E).tolist() == ref["counts"]  # bit-exact
            assert moe.moe_residency_slot_table(h, l, E).tolist() == ref["slot_of"]
            st = moe.moe_residency_get_stats(h, l)
            assert (st["hits"], st["misses"], st["evictions"]) == (ref["hits"], ref["misses"], ref["evictions"])
            assert st["steps"] == steps
    finally:
        moe.moe_residency_destroy(h)


def test_capacity_is_checked_at_init():
    cfg = dict(layers=1, experts=64, slots=6, spares=0, max_ids_per_step=8, dry_run=1,
               block_bytes=4096, decay=0.9)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_residency_create(cfg, None, None, None)
    assert ei.value.status == moe.MOE_ERR_CAPACITY
    cfg.update(slots=65)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_residency_create(cfg, None, None, None)
    assert ei.value.status == moe.MOE_ERR_CAPACITY
    cfg.update(slots=8, decay=0.0)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_residency_create(cfg, None, None, None)
    assert ei.value.status == moe.MOE_ERR_ARG


def test_rejected_steps_change_nothing():
    h = dry(16, 4, 0, 0.9, max_ids=4)
    try:
        moe.moe_residency_prepare(h, 0, [5, 6])
        before = (moe.moe_residency_counts(h, 0, 16).tolist(), moe.moe_residency_slot_table(h, 0, 16).tolist(),
                  moe.moe_residency_get_stats(h, 0), moe.moe_residency_trace(h))
        # More ids than max_ids_per_step, ids out of range: rejected whole.
        for ids, status in (([1, 2, 3, 7, 9], moe.MOE_ERR_ARG), ([1, 16], moe.MOE_ERR_ARG),
                            ([-1], moe.MOE_ERR_ARG), (list(range(9)), moe.MOE_ERR_ARG)):
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_residency_prepare(h, 0, ids)
            assert ei.value.status == status
        after = (moe.moe_residency_counts(h, 0, 16).tolist(), moe.moe_residency_slot_table(h, 0, 16).tolist(),
                 moe.moe_residency_get_stats(h, 0), moe.moe_residency_trace(h))
        assert before == after
        with pytest.raises(moe.MoeError):
            moe.moe_residency_prepare(h, 1, [0])  # layer out of range
    finally:
        moe.moe_residency_destroy(h)


def test_injected_failure_with_spares_keeps_previous_generation():
    # Copies land in spare slots only, so a failure leaves every published
    # expert intact: counts, slot table and statistics keep their values.
    h = dry(16, 4, 4, 0.9, max_ids=4)
    try:
        moe.moe_residency_prepare(h, 0, [0, 1])
        before = (moe.moe_residency_counts(h, 0, 16).tolist(), moe.moe_residency_slot_table(h, 0, 16).tolist(),
                  moe.moe_residency_get_stats(h, 0))
        moe.moe_residency_inject_copy_failure(h, 2)
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_residency_prepare(h, 0, [8, 9, 10, 11])
        assert ei.value.status == moe.MOE_ERR_INJECTED
        after = (moe.moe_residency_counts(h, 0, 16).tolist(), moe.moe_residency_slot_table(h, 0, 16).tolist(),
                 moe.moe_residency_get_stats(h, 0))
        assert before == after
        # The hook fires once; the retried step then succeeds as if fresh.
        moe.moe_residency_prepare(h, 0, [8, 9, 10, 11])
        ref = moe_oracle.residency_sim([[0, 1], [8, 9, 10, 11]], 16, 4, 4, 0.9)
        assert moe.moe_residency_slot_table(h, 0, 16).tolist() == ref["slot_of"]
    finally:
        moe.moe_residency_destroy(h)


def test_injected_failure_in_place_marks_overwritten_victims_absent():
    # No spares: the first two copies of the failed step reuse victims' slots
    # in place; those victims can no longer be served and become absent. The
    # rest of the previous generation and the counts are kept.
    h = dry(16, 4, 0, 0.9, max_ids=4)
    try:
        before_table = moe.moe_residency_slot_table(h, 0, 16).tolist()  # experts 0..3 in slots 0..3
        before_counts = moe.moe_residency_counts(h, 0, 16).tolist()
        moe.moe_residency_inject_copy_failure(h, 2)
        with pytest.raises(moe.MoeError):
            moe.moe_residency_prepare(h, 0, [8, 9, 10])
        table = moe.moe_residency_slot_table(h, 0, 16).tolist()
        # misses 8, 9 would have evicted 0 and 1 (lowest (count, id)); their slots were overwritten
        assert table[0] == -1 and table[1] == -1
        assert table[2:4] == before_table[2:4] and all(v == -1 for v in table[4:])
        assert moe.moe_residency_counts(h, 0, 16).tolist() == before_counts
        assert moe.moe_residency_get_stats(h, 0)["steps"] == 0
        # The freed slots are used first by the next step.
        moe.moe_residency_prepare(h, 0, [8, 9, 10])
        t = moe.moe_residency_slot_table(h, 0, 16)
        assert sorted(t[t >= 0].tolist()) == [0, 1, 2, 3]
        assert t[8] >= 0 and t[9] >= 0 and t[10] >= 0
    finally:
        moe.moe_residency_destroy(h)


# ---- victim policies: LRU and profile-pinned --------------------------------
def dry_policy(E, C, S, decay, policy, pinned=0, profile=None, L=1, max_ids=8):
    cfg = dict(layers=L, experts=E, slots=C, spares=S, max_ids_per_step=max_ids, dry_run=1,
               block_bytes=4096, decay=decay, policy=policy, pinned=pinned, profile=profile)
    return moe.moe_residency_create(cfg, None, None, None)


def test_policy_hand_traces_match_golden():
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "residency_policy_traces.json")))
    for c in g["cases"]:
        prof = None if c["profile"] is None else np.asarray(c["profile"])
        h = dry_policy(c["E"], c["C"], c["S"], c["decay"], c["policy"], c["pinned"], prof, max_ids=c["max_ids"])
        try:
            for ids in c["steps"]:
                moe.moe_residency_prepare(h, 0, ids)
            tr = [[s, e, sl, v] for (s, l, e, sl, v) in moe.moe_residency_trace(h)]
            assert tr == c["trace"], c["name"]
            assert moe.moe_residency_slot_table(h, 0, c["E"]).tolist() == c["slot_of_after"], c["name"]
            st = moe.moe_residency_get_stats(h, 0)
            assert (st["hits"], st["misses"], st["evictions"]) == (c["hits"], c["misses"], c["evictions"])
        finally:
            moe.moe_residency_destroy(h)
        # The oracle's model gives the same trace by hand.
        ref = moe_oracle.residency_sim(c["steps"], c["E"], c["C"], c["S"], c["decay"], c["policy"],
                                       c["profile"], c["pinned"])
        assert [list(t) for t in ref["trace"]] == c["trace"]
        if "decay_trace" in c:
            d = moe_oracle.residency_sim(c["steps"], c["E"], c["C"], c["S"], c["decay"], "decay")
            assert [list(t) for t in d["trace"]] == c["decay_trace"]


@pytest.mark.parametrize("policy,E,C,S,k,T,alpha,pinned", [
    ("lru", 64, 30, 0, 8, 1, 1.0, 0),
    ("lru", 64, 30, 2, 8, 1, 1.0, 0),
    ("lru", 32, 12, 0, 4, 2, 0.5, 0),
    ("pinned", 64, 30, 0, 8, 1, 1.0, 22),
    ("pinned", 64, 40, 1, 8, 4, 1.0, 8),
    ("pinned", 64, 16, 0, 8, 1, 0.0, 8),
])
def test_policy_variants_match_oracle(policy, E, C, S, k, T, alpha, pinned):
    L, steps = 2, 300
    prof = np.stack([1.0 / synth.zipf_ranks(9, l, E) ** max(alpha, 1e-9) for l in range(L)])
    h = dry_policy(E, C, S, 0.9, policy, pinned, prof if policy == "pinned" else None, L=L, max_ids=T * k)
    try:
        per_layer = {l: [] for l in range(L)}
        for step in range(steps):
            for l in range(L):
                lg = synth.logits_zipf(9, l, step, T, E, alpha)
                ids, _ = moe_oracle.route(lg, k, False)
                flat = ids.reshape(-1).tolist()
                per_layer[l].append(flat)
                moe.moe_residency_prepare(h, l, flat)
        trace = moe.moe_residency_trace(h)
        for l in range(L):
            ref = moe_oracle.residency_sim(per_layer[l], E, C, S, 0.9, policy, prof[l], pinned)
            got = [(s, e, sl, v) for (s, ll, e, sl, v) in trace if ll == l]
            assert got == [tuple(t) for t in ref["trace"]]
            st = moe.moe_residency_get_stats(h, l)
            assert (st["hits"], st["misses"], st["evictions"]) == (ref["hits"], ref["misses"], ref["evictions"])
            assert moe.moe_residency_slot_table(h, l, E).tolist() == ref["slot_of"]
            if policy == "pinned":
                top = np.argsort(-prof[l], kind="stable")[:pinned]
                assert all(v not in set(top.tolist()) for (_, _, _, v) in got)
                assert all(ref["slot_of"][e] >= 0 for e in top)
    finally:
        moe.moe_residency_destroy(h)


def test_pinned_capacity_and_arguments():
    with pytest.raises(moe.MoeError):  # 25 pinned leave 5 < 8 slots for a step's misses
        dry_policy(64, 30, 0, 0.9, "pinned", 25, np.ones((1, 64)))
    with pytest.raises(moe.MoeError):  # the pinned policy needs a profile
        dry_policy(64, 30, 0, 0.9, "pinned", 4, None)
    with pytest.raises(moe.MoeError):  # unknown policy
        dry_policy(64, 30, 0, 0.9, 7)


@pytest.mark.parametrize("alpha", [1.0, 0.0])
def test_policy_hit_rates_against_the_ceiling(alpha):
    # Stationary popularity: over a long run no policy beats the best fixed
    # set (the sum of the C largest inclusion frequencies, measured on the
    # same stream); with the true profile, pinning is within a few points of
    # it on Zipf popularity; with uniform popularity every policy sits at
    # about C/E.
    E, C, k, steps, pinned = 64, 30, 8, 3000, 22
    stream = []
    for s in range(steps):
        ids, _ = moe_oracle.route(synth.logits_zipf(13, 0, s, 1, E, alpha), k, False)
        stream.append(ids.reshape(-1).tolist())
    freq = np.zeros(E)
    for ids in stream:
        freq[ids] += 1
    p = freq / steps
    ceiling = moe_oracle.hit_ceiling(p, C) / k  # hit fraction of the accesses
    prof = 1.0 / synth.zipf_ranks(13, 0, E) ** max(alpha, 1e-9)
    rates = {}
    for policy in ("decay", "lru", "pinned"):
        r = moe_oracle.residency_sim(stream, E, C, 0, 0.9, policy, prof, pinned)
        rates[policy] = r["hits"] / (r["hits"] + r["misses"])
    for policy, rate in rates.items():
        assert rate <= ceiling + 0.01, (policy, rate, ceiling)
    if alpha > 0:
        assert rates["pinned"] >= ceiling - 0.08, (rates, ceiling)
        assert rates["pinned"] >= rates["lru"] - 0.01, rates
    else:
        for rate in rates.values():
            assert abs(rate - C / E) < 0.05, (rates, C / E)


# ---- prefetch of predicted misses into spare slots ---------------------------
def _run_ops(ops, lib_h=None, orc=None):
    out = []
    for op in ops:
        if op["op"] == "step":
            if lib_h is not None:
                moe.moe_residency_prepare(lib_h, 0, op["ids"])
            if orc is not None:
                orc.step(op["ids"])
        else:
            n_lib = moe.moe_residency_prefetch(lib_h, 0, op["ids"]) if lib_h is not None else None
            n_orc = len(orc.prefetch(op["ids"])) if orc is not None else None
            out.append((n_lib, n_orc))
    return out


def test_prefetch_hand_trace_matches_golden():
    c = json.load(open(os.path.join(ROOT, "tests", "golden", "residency_prefetch_trace.json")))
    h = dry_policy(c["E"], c["C"], c["S"], c["decay"], c["policy"], max_ids=2)
    try:
        staged = _run_ops(c["ops"], lib_h=h)
        assert [n for n, _ in staged] == [op["staged"] for op in c["ops"] if op["op"] == "prefetch"]
        tr = [[s, e, sl, v] for (s, l, e, sl, v) in moe.moe_residency_trace(h)]
        assert tr == c["trace"]
        assert moe.moe_residency_slot_table(h, 0, c["E"]).tolist() == c["slot_of_after"]
        assert moe.moe_residency_counts(h, 0, c["E"]).tolist() == c["counts_after"]
        st = moe.moe_residency_get_stats(h, 0)
        assert (st["hits"], st["misses"], st["evictions"], st["prefetched"], st["prefetch_copies"]) == (
            c["hits"], c["misses"], c["evictions"], c["prefetched"], c["prefetch_copies"])
    finally:
        moe.moe_residency_destroy(h)


@pytest.mark.parametrize("policy,E,C,S,k,alpha", [
    ("decay", 64, 30, 4, 8, 1.0),
    ("lru", 64, 30, 2, 8, 1.0),
    ("pinned", 64, 30, 3, 8, 1.0),
    ("decay", 32, 12, 6, 4, 0.0),
])
def test_prefetch_policies_match_oracle(policy, E, C, S, k, alpha):
    # Each step is preceded by a prefetch of the S non-resident experts with
    # the highest decayed counts (ties: lower id) -- a popularity predictor.
    steps = 250
    ranks = synth.zipf_ranks(5, 0, E)
    profile = 1.0 / ranks.astype(np.float64) ** max(alpha, 1e-9)
    pinned = C - k if policy == "pinned" else 0
    h = dry_policy(E, C, S, 0.9, policy, pinned=pinned, profile=profile if policy == "pinned" else None,
                   max_ids=k)
    orc = moe_oracle.ResidencyLayer(E, C, S, 0.9, policy, profile, pinned)
    try:
        for step in range(steps):
            counts = moe.moe_residency_counts(h, 0, E)
            table = moe.moe_residency_slot_table(h, 0, E)
            cand = sorted((e for e in range(E) if table[e] < 0), key=lambda e: (-counts[e], e))[:S]
            n_lib = moe.moe_residency_prefetch(h, 0, cand)
            assert n_lib == len(orc.prefetch(cand))
            lg = synth.logits_zipf(5, 0, step, 1, E, alpha)
            ids, _ = moe_oracle.route(lg, k, False)
            moe.moe_residency_prepare(h, 0, ids.reshape(-1).tolist())
            orc.step(ids.reshape(-1).tolist())
        assert moe.moe_residency_slot_table(h, 0, E).tolist() == orc.slot_of
        st = moe.moe_residency_get_stats(h, 0)
        assert (st["hits"], st["misses"], st["evictions"], st["prefetched"], st["prefetch_copies"]) == (
            orc.hits, orc.misses, orc.evictions, orc.prefetched, orc.prefetch_copies)
        trace = [(s, e, sl, v) for (s, l, e, sl, v) in moe.moe_residency_trace(h)]
        assert len(trace) == orc.misses
        if alpha > 0:
            assert orc.prefetched > 0  # the predictor serves some misses
    finally:
        moe.moe_residency_destroy(h)


def test_prefetch_arguments_and_limits():
    h = dry_policy(8, 3, 0, 0.9, "decay", max_ids=2)  # no spare slots
    try:
        assert moe.moe_residency_prefetch(h, 0, [5, 6]) == 0
        with pytest.raises(moe.MoeError):
            moe.moe_residency_prefetch(h, 0, [9])
        with pytest.raises(moe.MoeError):
            moe.moe_residency_prefetch(h, 1, [5])
    finally:
        moe.moe_residency_destroy(h)
    h = dry_policy(8, 3, 2, 0.9, "decay", max_ids=2)
    try:
        # Resident and repeated ids are skipped; out-of-range ids stage nothing.
        with pytest.raises(moe.MoeError):
            moe.moe_residency_prefetch(h, 0, [5, 99])
        assert moe.moe_residency_get_stats(h, 0)["prefetch_copies"] == 0
        assert moe.moe_residency_prefetch(h, 0, [0, 5, 5, 6, 7]) == 2
        # A rejected step (capacity) keeps the staged copies for the next one.
        with pytest.raises(moe.MoeError):
            moe.moe_residency_prepare(h, 0, [1, 2, 3, 4])
        moe.moe_residency_prepare(h, 0, [6])
        st = moe.moe_residency_get_stats(h, 0)
        assert (st["misses"], st["prefetched"]) == (1, 1)
        # 5 was not needed: its spare slot is free again for the next prefetch.
        assert moe.moe_residency_prefetch(h, 0, [5, 7]) == 2
    finally:
        moe.moe_residency_destroy(h)


def test_prefetch_injected_failure_stages_nothing_more():
    h = dry_policy(8, 3, 2, 0.9, "decay", max_ids=2)
    try:
        moe.moe_residency_inject_copy_failure(h, 1)  # the second copy from now fails
        with pytest.raises(moe.MoeError):
            moe.moe_residency_prefetch(h, 0, [5, 6])
        # The first copy was staged, the second not; the next step uses the first.
        moe.moe_residency_prepare(h, 0, [5, 6])
        st = moe.moe_residency_get_stats(h, 0)
        assert (st["prefetch_copies"], st["prefetched"], st["misses"]) == (1, 1, 2)
    finally:
        moe.moe_residency_destroy(h)
