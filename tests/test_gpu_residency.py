"""Residency manager with real copies (needs a GB300): H2D copies from a
pinned, immutable source into the slot pool, slot-table publish, and the
routed layer computed from the managed pool, step after step."""
import hashlib

import numpy as np
import pytest
import torch

from int4_routed_expert_moe_gb300 import synth
from oracle import moe_oracle
from tests._lib import binding
from tests.gpu_util import tol_ok

pytestmark = pytest.mark.gpu

SHAPE = (256, 128, 64)
L, E, K = 2, 16, 2


def _setup(moe, C, S, seed):
    H, I, g = SHAPE
    bb = moe.moe_expert_block_bytes(SHAPE)
    src = torch.empty((L, E, bb), dtype=torch.uint8).pin_memory()
    arrays = {}
    for l in range(L):
        for e in range(E):
            arrays[(l, e)] = synth.expert_arrays(seed, l, e, H, I, g)
            moe.moe_pack_expert(SHAPE, arrays[(l, e)], out=src[l, e].numpy())
    dev = torch.device("cuda")
    pool = torch.zeros((L, C + S, bb), dtype=torch.uint8, device=dev)
    slot_of = torch.full((L, E), -9, dtype=torch.int32, device=dev)
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    cfg = dict(layers=L, experts=E, slots=C, spares=S, max_ids_per_step=4 * K, block_bytes=bb, decay=0.9)
    h = moe.moe_residency_create(cfg, src, pool, slot_of, compute, copy)
    return h, src, pool, slot_of, arrays, bb


@pytest.mark.parametrize("C,S", [(8, 0), (8, 2)])
def test_residency_copies_publish_and_forward(C, S):
    moe = binding()
    H, I, g = SHAPE
    T = 4
    h, src, pool, slot_of, arrays, bb = _setup(moe, C, S, 71)
    digest = hashlib.sha256(src.numpy().tobytes()).hexdigest()
    dev = torch.device("cuda")
    ws = torch.zeros(moe.moe_forward_workspace_bytes(SHAPE, T, K, E, moe.MOE_PATH_GEMV),
                     dtype=torch.uint8, device=dev)
    ids_steps = {l: [] for l in range(L)}
    try:
        for step in range(12):
            for l in range(L):
                lg = synth.logits_zipf(71, l, step, T, E, 1.0)
                ids_d = torch.empty((T, K), dtype=torch.int32, device=dev)
                w_d = torch.empty((T, K), dtype=torch.float32, device=dev)
                moe.moe_route(torch.from_numpy(lg).to(dev), K, True, ids_d, w_d)
                ids_h = ids_d.cpu().numpy()  # the step's ids reach the host
                ids_steps[l].append(ids_h.reshape(-1).tolist())
                moe.moe_residency_prepare(h, l, ids_h)
                x16 = synth.activations(71, step * L + l, T, H)
                y = torch.empty((T, H), dtype=torch.float16, device=dev)
                moe.moe_expert_forward(SHAPE, torch.from_numpy(x16).to(dev), ids_d, w_d, E, pool[l],
                                       slot_of[l], C + S, None, y, ws, moe.MOE_PATH_GEMV)
                ref = moe_oracle.moe_layer(x16, lg, lambda e, l=l: arrays[(l, e)], K, True, g)
                ok, err, bound = tol_ok(y.float().cpu().numpy(), ref["y"])
                assert ok, (step, l, err, bound)
                assert moe.moe_workspace_flags(ws) == 0
        torch.cuda.synchronize()
        trace = moe.moe_residency_trace(h)
        for l in range(L):
            host_table = moe.moe_residency_slot_table(h, l, E)
            assert np.array_equal(slot_of[l].cpu().numpy(), host_table)  # published = decided
            for e in range(E):
                s = host_table[e]
                if s >= 0:  # the slot holds exactly the source block
                    assert torch.equal(pool[l, s].cpu(), src[l, e])
            ref = moe_oracle.residency_sim(ids_steps[l], E, C, S, 0.9)
            assert [(s_, e, sl, v) for (s_, ll, e, sl, v) in trace if ll == l] == [tuple(t) for t in ref["trace"]]
            st = moe.moe_residency_get_stats(h, l)
            assert st["h2d_bytes"] == st["misses"] * bb and st["copies"] == st["misses"]
        assert hashlib.sha256(src.numpy().tobytes()).hexdigest() == digest  # source never written
    finally:
        moe.moe_residency_destroy(h)


def test_residency_injected_failure_keeps_serving_valid_experts():
    moe = binding()
    H, I, g = SHAPE
    C, S, T = 8, 2, 1
    h, src, pool, slot_of, arrays, bb = _setup(moe, C, S, 72)
    dev = torch.device("cuda")
    try:
        before = slot_of[0].cpu().numpy().copy()
        moe.moe_residency_inject_copy_failure(h, 1)
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_residency_prepare(h, 0, [10, 11])
        assert ei.value.status == moe.MOE_ERR_INJECTED
        torch.cuda.synchronize()
        assert np.array_equal(slot_of[0].cpu().numpy(), before)  # previous generation kept
        moe.moe_residency_prepare(h, 0, [10, 11])  # retried step succeeds
        torch.cuda.synchronize()
        table = slot_of[0].cpu().numpy()
        assert table[10] >= 0 and table[11] >= 0
        assert torch.equal(pool[0, table[10]].cpu(), src[0, 10])
        assert torch.equal(pool[0, table[11]].cpu(), src[0, 11])
    finally:
        moe.moe_residency_destroy(h)


def test_residency_rejects_pageable_source():
    moe = binding()
    bb = moe.moe_expert_block_bytes(SHAPE)
    dev = torch.device("cuda")
    cfg = dict(layers=1, experts=E, slots=6, spares=0, max_ids_per_step=2, block_bytes=bb, decay=0.9)
    with pytest.raises(ValueError):
        moe.moe_residency_create(cfg, torch.empty((1, E, bb), dtype=torch.uint8), torch.empty((1, 6, bb), dtype=torch.uint8, device=dev),
                                 torch.empty((1, E), dtype=torch.int32, device=dev))


def test_residency_prefetch_copies_and_forward():
    # After each layer's experts are enqueued, the next layer's predicted
    # misses (the S non-resident experts with the highest decayed counts) are
    # prefetched into spare slots on the copy stream; the next prepare() takes
    # the needed ones without a copy. Outputs, slot contents, decisions and
    # copy counts are checked against the oracle.
    moe = binding()
    H, I, g = SHAPE
    C, S, T = 8, 3, 2
    h, src, pool, slot_of, arrays, bb = _setup(moe, C, S, 73)
    dev = torch.device("cuda")
    ws = [torch.zeros(moe.moe_forward_workspace_bytes(SHAPE, T, K, E, moe.MOE_PATH_GEMV), dtype=torch.uint8,
                      device=dev) for _ in range(L)]
    orc = {l: moe_oracle.ResidencyLayer(E, C, S, 0.9) for l in range(L)}
    pending = []

    def predict_and_prefetch(l):
        counts = moe.moe_residency_counts(h, l, E)
        table = moe.moe_residency_slot_table(h, l, E)
        cand = sorted((e for e in range(E) if table[e] < 0), key=lambda e: (-counts[e], e))[:S]
        assert moe.moe_residency_prefetch(h, l, cand) == len(orc[l].prefetch(cand))

    try:
        for step in range(16):
            for l in range(L):
                lg = synth.logits_zipf(73, l, step, T, E, 1.2)
                ids_d = torch.empty((T, K), dtype=torch.int32, device=dev)
                w_d = torch.empty((T, K), dtype=torch.float32, device=dev)
                moe.moe_route(torch.from_numpy(lg).to(dev), K, True, ids_d, w_d)
                ids_h = ids_d.cpu().numpy()
                moe.moe_residency_prepare(h, l, ids_h)
                orc[l].step(ids_h.reshape(-1).tolist())
                x16 = synth.activations(73, step * L + l, T, H)
                y = torch.empty((T, H), dtype=torch.float16, device=dev)
                moe.moe_expert_forward(SHAPE, torch.from_numpy(x16).to(dev), ids_d, w_d, E, pool[l],
                                       slot_of[l], C + S, None, y, ws[l], moe.MOE_PATH_GEMV)
                pending.append((y, moe_oracle.moe_layer(x16, lg, lambda e, l=l: arrays[(l, e)], K, True, g)["y"]))
                predict_and_prefetch((l + 1) % L)  # overlaps this layer's experts
        torch.cuda.synchronize()
        for y, ref in pending:
            ok, err, bound = tol_ok(y.float().cpu().numpy(), ref)
            assert ok, (err, bound)
        assert all(moe.moe_workspace_flags(w) == 0 for w in ws)
        total_prefetched = 0
        for l in range(L):
            table = moe.moe_residency_slot_table(h, l, E)
            assert np.array_equal(slot_of[l].cpu().numpy(), table)
            assert table.tolist() == orc[l].slot_of
            for e in range(E):
                if table[e] >= 0:
                    assert torch.equal(pool[l, table[e]].cpu(), src[l, e])
            st = moe.moe_residency_get_stats(h, l)
            o = orc[l]
            assert (st["hits"], st["misses"], st["prefetched"], st["prefetch_copies"]) == (
                o.hits, o.misses, o.prefetched, o.prefetch_copies)
            assert st["copies"] == st["misses"] - st["prefetched"] + st["prefetch_copies"]
            assert st["h2d_bytes"] == st["copies"] * bb
            total_prefetched += st["prefetched"]
        assert total_prefetched > 0
    finally:
        moe.moe_residency_destroy(h)
