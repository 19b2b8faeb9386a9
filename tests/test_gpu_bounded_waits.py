"""The streamed decode kernel's bounded waits (needs a GB300).

Every wait of the kernel gives up after about a second: the block sets bit 2
of the workspace error word, stops waiting, lets its own copies land and
exits, and the last block out still zeroes the counters. The tests make one
wait run out without any fault: a counter that every block releases into
starts far below zero, so the count the waiters expect never comes -- the
grid barrier's counter of the several-token schedule (4 tokens, and one
token with 17 picks, which takes that schedule), and the per-unit counters
that one token's exchange warps poll before copying h. The call must come
back with bit 2 set, the counters zeroed, and the next call on the same
workspace must be correct.
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
CNT_BASE = 64  # workspace word of the kernel's first counter


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


@pytest.mark.parametrize("T,K,counters", [(4, 8, 1), (1, 17, 1), (1, 8, 8)])
def test_decode_wait_expires_and_workspace_recovers(pool, T, K, counters):
    dev = torch.device("cuda")
    x16 = synth.activations(pool.seed, 5, T, SHAPE[0])
    lg16 = synth.logits_normal(pool.seed, 6, T, E)
    x, lg = torch.from_numpy(x16).to(dev), torch.from_numpy(lg16).to(dev)
    ws = torch.zeros(moe.moe_forward_workspace_bytes(SHAPE, T, K, E, moe.MOE_PATH_GEMV), dtype=torch.uint8,
                     device=dev)
    words = ws.view(torch.int32)
    n = counters  # the grid barrier's counter, or one counter per unit (one token, <= 16 picks)
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
