"""Shared (non-routed) FP16 SwiGLU FFN on the tensor cores vs the CPU oracle,
through the C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

from int4_routed_expert_moe_gb300 import synth
from oracle import moe_oracle
from tests._lib import binding
from tests.gpu_util import tol_ok

pytestmark = pytest.mark.gpu

moe = binding() if torch.cuda.is_available() else None


def _run(T, H, Is, seed):
    dev = torch.device("cuda")
    w = synth.shared_weights(seed, H, Is)
    x = synth.activations(seed, 1, T, H)
    tw = {k: torch.from_numpy(v).to(dev) for k, v in w.items()}
    y = torch.empty((T, H), dtype=torch.float16, device=dev)
    ws = torch.zeros(moe.moe_shared_workspace_bytes(T, H, Is), dtype=torch.uint8, device=dev)
    moe.moe_shared_forward(torch.from_numpy(x).to(dev), tw["wg"], tw["wu"], tw["wd"], y, ws)
    assert moe.moe_workspace_flags(ws) == 0
    return x, w, y.float().cpu().numpy()


@pytest.mark.parametrize("T,H,Is", [
    (4, 256, 128),      # one tile
    (130, 512, 320),    # ragged tokens (two token tiles) and Is not a multiple of 128
    (1, 64, 64),        # smallest shape: one K step, one row block with 64 live rows
    (300, 1024, 2048),  # several tiles in every direction
])
def test_shared_matches_oracle(T, H, Is):
    x, w, y = _run(T, H, Is, 51)
    ref = moe_oracle.shared_ffn(x, w["wg"], w["wu"], w["wd"])
    ok, err, bound = tol_ok(y, ref)
    assert ok, (err, bound)


def test_shared_config_shape_sampled():
    # The prefill configuration's shared FFN: 2048 tokens, H 2048, Is 4096.
    T, H, Is = 2048, 2048, 4096
    x, w, y = _run(T, H, Is, 52)
    rows = [0, 1, 127, 128, 1000, 2047]
    ref = moe_oracle.shared_ffn(x[rows], w["wg"], w["wu"], w["wd"])
    ok, err, bound = tol_ok(y[rows], ref)
    assert ok, (err, bound)


def test_shared_deterministic():
    _, _, a = _run(130, 512, 320, 53)
    _, _, b = _run(130, 512, 320, 53)
    assert np.array_equal(a, b)


def test_shared_rejects_bad_shapes():
    dev = torch.device("cuda")
    x = torch.zeros((4, 100), dtype=torch.float16, device=dev)
    wg = torch.zeros((64, 100), dtype=torch.float16, device=dev)
    wd = torch.zeros((100, 64), dtype=torch.float16, device=dev)
    y = torch.empty((4, 100), dtype=torch.float16, device=dev)
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    with pytest.raises(moe.MoeError):
        moe.moe_shared_forward(x, wg, wg, wd, y, ws)


def test_shared_largest_hidden():
    # H = 8192: 128 K steps in the gate/up GEMM, 64 output row blocks in the down GEMM.
    x, w, y = _run(40, 8192, 256, 54)
    ref = moe_oracle.shared_ffn(x, w["wg"], w["wu"], w["wd"])
    ok, err, bound = tol_ok(y, ref)
    assert ok, (err, bound)


def test_shared_empty_batch():
    dev = torch.device("cuda")
    x = torch.empty((0, 256), dtype=torch.float16, device=dev)
    wg = torch.zeros((128, 256), dtype=torch.float16, device=dev)
    wd = torch.zeros((256, 128), dtype=torch.float16, device=dev)
    y = torch.empty((0, 256), dtype=torch.float16, device=dev)
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    moe.moe_shared_forward(x, wg, wg, wd, y, ws)
    torch.cuda.synchronize()
