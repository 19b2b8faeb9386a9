"""Routed expert FFN whose absent experts are read in place from pinned host
memory over the CPU-GPU link, vs the CPU oracle and vs the same kernels with
every expert resident (needs a GB300)."""
import numpy as np
import pytest
import torch

from int4_routed_expert_moe_gb300 import synth
from oracle import moe_oracle
from tests._lib import binding
from tests.gpu_util import LayerPool, tol_ok

pytestmark = pytest.mark.gpu

moe = binding() if torch.cuda.is_available() else None
UNFUSED = 3


def _inputs(lp, seed, T, k, renorm=False):
    H, I, g = lp.shape
    dev = torch.device("cuda")
    x16 = synth.activations(seed, 1, T, H)
    lg = synth.logits_normal(seed, 3, T, lp.E)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    moe.moe_route(torch.from_numpy(lg).to(dev), k, renorm, ids, w)
    return x16, lg, torch.from_numpy(x16).to(dev), ids, w


def _zero_copy(lp, resident, x, ids, w, y_shared=None):
    """Pool holding only `resident` experts (slots in that order), the rest
    read from a pinned host copy of all E blocks."""
    dev = torch.device("cuda")
    E, bb = lp.E, lp.block_bytes
    host = lp.pool.cpu().pin_memory()
    n_slots = max(1, len(resident))
    pool = torch.zeros((n_slots, bb), dtype=torch.uint8, device=dev)
    slot_of = torch.full((E,), -1, dtype=torch.int32, device=dev)
    for s, e in enumerate(resident):
        pool[s] = lp.pool[e]
        slot_of[e] = s
    T, k = ids.shape
    H = lp.shape[0]
    y = torch.empty((T, H), dtype=torch.float16, device=dev)
    ws = torch.zeros(moe.moe_forward_workspace_bytes(lp.shape, T, k, E, UNFUSED), dtype=torch.uint8, device=dev)
    moe.moe_expert_forward_zero_copy(lp.shape, x, ids, w, E, pool, slot_of, n_slots, host, y_shared, y, ws)
    torch.cuda.synchronize()
    return y, moe.moe_workspace_flags(ws)


def _all_resident(lp, x, ids, w, y_shared=None):
    T, k = ids.shape
    dev = torch.device("cuda")
    y = torch.empty((T, lp.shape[0]), dtype=torch.float16, device=dev)
    ws = torch.zeros(moe.moe_forward_workspace_bytes(lp.shape, T, k, lp.E, UNFUSED), dtype=torch.uint8,
                     device=dev)
    moe.moe_expert_forward(lp.shape, x, ids, w, lp.E, lp.pool, lp.slot_of, lp.E, y_shared, y, ws, UNFUSED)
    return y


@pytest.mark.parametrize("shape,E,k,T,resident", [
    ((2048, 1024, 128), 16, 8, 4, list(range(8))),     # half the experts over the link
    ((2048, 1024, 128), 16, 8, 4, []),                 # every expert over the link
    ((1088, 320, 32), 6, 3, 5, [5, 0, 3]),             # ragged shape, scattered slots
])
def test_zero_copy_matches_oracle_and_resident(shape, E, k, T, resident):
    lp = LayerPool(moe, 61, 0, shape, E, zero="int")
    x16, lg, x, ids, w = _inputs(lp, 61, T, k)
    y, flags = _zero_copy(lp, resident, x, ids, w)
    assert flags == 0
    got = y.float().cpu().numpy()
    # Same kernels, same arithmetic: only the address the blocks come from differs.
    assert np.array_equal(got, _all_resident(lp, x, ids, w).float().cpu().numpy())
    ref = moe_oracle.moe_layer(x16, lg, lp.arrays, k, False, shape[2])
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    ok, err, bound = tol_ok(got, ref["y"])
    assert ok, (err, bound)


def test_zero_copy_layer_inside_a_larger_allocation():
    # The host source of layer 1 of a [3][E][block] pinned allocation: the
    # device reads must land on that layer, not on the allocation's start.
    lp = LayerPool(moe, 65, 0, (512, 256, 64), 6, zero="int")
    dev = torch.device("cuda")
    x16, lg, x, ids, w = _inputs(lp, 65, 3, 2)
    host = torch.zeros((3, 6, lp.block_bytes), dtype=torch.uint8).pin_memory()
    host[1].copy_(lp.pool.cpu())
    pool = torch.zeros((1, lp.block_bytes), dtype=torch.uint8, device=dev)
    slot_of = torch.full((6,), -1, dtype=torch.int32, device=dev)
    y = torch.empty((3, 512), dtype=torch.float16, device=dev)
    ws = torch.zeros(moe.moe_forward_workspace_bytes(lp.shape, 3, 2, 6, UNFUSED), dtype=torch.uint8, device=dev)
    moe.moe_expert_forward_zero_copy(lp.shape, x, ids, w, 6, pool, slot_of, 1, host[1], None, y, ws)
    torch.cuda.synchronize()
    assert moe.moe_workspace_flags(ws) == 0
    ref = moe_oracle.moe_layer(x16, lg, lp.arrays, 2, False, 64)
    ok, err, bound = tol_ok(y.float().cpu().numpy(), ref["y"])
    assert ok, (err, bound)


def test_zero_copy_with_shared_output():
    lp = LayerPool(moe, 62, 0, (512, 256, 64), 8)
    x16, lg, x, ids, w = _inputs(lp, 62, 3, 2, renorm=True)
    ysh16 = synth.activations(62, 2, 3, 512)
    ysh = torch.from_numpy(ysh16).cuda()
    y, flags = _zero_copy(lp, [1, 2], x, ids, w, y_shared=ysh)
    assert flags == 0
    ref = moe_oracle.moe_layer(x16, lg, lp.arrays, 2, True, 64, y_shared=ysh16)
    ok, err, bound = tol_ok(y.float().cpu().numpy(), ref["y"])
    assert ok, (err, bound)


def test_zero_copy_bad_slot_still_flagged():
    lp = LayerPool(moe, 63, 0, (512, 256, 64), 4)
    dev = torch.device("cuda")
    x16, lg, x, ids, w = _inputs(lp, 63, 2, 2)
    host = lp.pool.cpu().pin_memory()
    slot_of = torch.tensor([0, 1, 2, 9], dtype=torch.int32, device=dev)  # slot 9 >= n_slots
    y = torch.empty((2, 512), dtype=torch.float16, device=dev)
    ws = torch.zeros(moe.moe_forward_workspace_bytes(lp.shape, 2, 2, 4, UNFUSED), dtype=torch.uint8, device=dev)
    ids_all3 = torch.full((2, 2), 3, dtype=torch.int32, device=dev)
    ids_all3[:, 1] = -1
    moe.moe_expert_forward_zero_copy(lp.shape, x, ids_all3, w, 4, lp.pool, slot_of, 4, host, None, y, ws)
    torch.cuda.synchronize()
    assert moe.moe_workspace_flags(ws) & 1
    assert torch.all(y == 0)


def test_zero_copy_rejects_pageable_source():
    lp = LayerPool(moe, 64, 0, (512, 256, 64), 4)
    dev = torch.device("cuda")
    x16, lg, x, ids, w = _inputs(lp, 64, 2, 2)
    pageable = lp.pool.cpu()
    slot_of = torch.full((4,), -1, dtype=torch.int32, device=dev)
    y = torch.empty((2, 512), dtype=torch.float16, device=dev)
    ws = torch.zeros(moe.moe_forward_workspace_bytes(lp.shape, 2, 2, 4, UNFUSED), dtype=torch.uint8, device=dev)
    with pytest.raises(moe.MoeError):
        moe.moe_expert_forward_zero_copy(lp.shape, x, ids, w, 4, lp.pool, slot_of, 4, pageable, None, y, ws)
