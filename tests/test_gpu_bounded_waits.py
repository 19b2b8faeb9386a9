"""The streamed decode kernel's bounded waits (needs a GB300).

Every wait of the kernel gives up after about a second: the block sets bit 2
of the workspace error word, stops waiting, lets its own copies land and
exits, and the last block out still zeroes the counters. The tests make one
wait run out without any fault: the grid barrier's counter, which every
block releases into between the gate/up and the down items, starts far
below zero, so the count the waiters expect never comes. The call must come
back with bit 2 set, the counters zeroed, and the next call on the same
workspace must be correct. (The single-token schedule of up to 16 picks has
no counter: its blocks poll each other's marked h words, which every block
writes itself, so nothing outside the kernel can withhold them; its polls
end on the same bound and abort path, read in the code. One token with 17
picks takes the grid-barrier schedule and is tested here.)
"""
import numpy as np
import pytest
import torch

from int4_routed_expert_moe_gb300 import synth
from oracle import moe_oracle
from tests._lib import binding
from tests.gpu_util import LayerPool, tol_ok

pytestmark = pytest.mark.gpu

moe = binding() if torch.cuda.is_available() else None

SHAPE = (2048, 1024, 128)  # the OLMoE expert shape
E = 64
CNT_BASE = 64  # workspace word of the grid barrier's counter


@pytest.fixture(scope="module")
def pool():
    return LayerPool(moe, 80, 0, SHAPE, E)


def _call(lp, x, lg, ws, T, K):
    dev = torch.device("cuda")
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    y = torch.empty((T, SHAPE[0]), dtype=torch.float16, device=dev)
    moe.moe_layer_forward(SHAPE, x, lg, K, False, ids, w, lp.pool, lp.slot_of, E, None, y, ws, moe.MOE_PATH_GEMV)
    return y


@pytest.mark.parametrize("T,K", [(4, 8), (1, 17)])
def test_decode_wait_expires_and_workspace_recovers(pool, T, K):
    dev = torch.device("cuda")
    x16 = synth.activations(pool.seed, 5, T, SHAPE[0])
    lg16 = synth.logits_normal(pool.seed, 6, T, E)
    x, lg = torch.from_numpy(x16).to(dev), torch.from_numpy(lg16).to(dev)
    ws = torch.zeros(moe.moe_forward_workspace_bytes(SHAPE, T, K, E, moe.MOE_PATH_GEMV), dtype=torch.uint8,
                     device=dev)
    words = ws.view(torch.int32)
    n = 1
    words[CNT_BASE:CNT_BASE + n] = -(1 << 30)  # a release count nobody reaches
    _call(pool, x, lg, ws, T, K)
    torch.cuda.synchronize()
    flags = moe.moe_workspace_flags(ws)
    assert flags & 4, flags  # a wait ran out and says so
    assert int(words[1]) == 0 and bool(torch.all(words[CNT_BASE:CNT_BASE + n] == 0))
    moe.moe_workspace_clear_flags(ws)
    y = _call(pool, x, lg, ws, T, K)
    assert moe.moe_workspace_flags(ws) == 0
    ref = moe_oracle.moe_layer(x16, lg16, pool.arrays, K, False, SHAPE[2])
    ok, err, bound = tol_ok(y.float().cpu().numpy(), ref["y"])
    assert ok, (T, err, bound)
