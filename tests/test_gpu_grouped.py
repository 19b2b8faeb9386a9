"""Grouped tensor-core path (token sort, tcgen05 gate/up and down GEMMs,
combine) vs the CPU oracle, through the C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

from int4_routed_expert_moe_gb300 import synth
from oracle import moe_oracle
from tests._lib import binding
from tests.gpu_util import LayerPool, run_layer, tol_ok

pytestmark = pytest.mark.gpu

moe = binding() if torch.cuda.is_available() else None
GROUPED = 2


def _logits(kind, seed, T, E):
    if kind == "zipf":
        return synth.logits_zipf(seed, 0, 3, T, E, 1.1)
    if kind == "uniform":
        return synth.logits_uniform(seed, 3, T, E)
    return synth.logits_normal(seed, 3, T, E)


def _case(shape, E, k, renorm, T, seed, zero="eight", shared=False, kind="normal", path=GROUPED,
          sample=None):
    H, I, g = shape
    lp = LayerPool(moe, seed, 0, shape, E, zero=zero)
    x = synth.activations(seed, 1, T, H)
    lg = _logits(kind, seed, T, E)
    ysh = synth.activations(seed, 2, T, H) if shared else None
    y, ids, w, flags = run_layer(moe, lp, x, lg, k, renorm, path, y_shared=ysh)
    assert flags == 0
    rows = np.arange(T) if sample is None else np.asarray(sample)
    ref = moe_oracle.moe_layer(x[rows], lg[rows], lp.arrays, k, renorm, g,
                               y_shared=None if ysh is None else ysh[rows])
    assert np.array_equal(ids[rows], ref["ids"])
    ok, err, bound = tol_ok(y[rows], ref["y"])
    assert ok, (err, bound)
    return y


@pytest.mark.parametrize("zero", ["eight", "int", "frac"])
@pytest.mark.parametrize("shared", [False, True])
def test_grouped_tiny_layer(zero, shared):
    _case((256, 128, 64), 8, 2, True, 4, 41, zero=zero, shared=shared)


@pytest.mark.parametrize("shape,E,k,T", [
    ((512, 256, 128), 16, 4, 64),    # 256 pairs, ~16 per expert, two gate/up row blocks
    ((320, 192, 64), 4, 2, 150),     # H and I not multiples of 128 (partial row blocks), odd group count
    ((256, 128, 32), 2, 1, 300),     # g = 32 (two groups per K step); ~150 pairs per expert: two tiles
    ((1024, 512, 128), 8, 2, 513),   # tiles of 128 and ragged tails
    ((128, 256, 64), 8, 2, 100),     # 2 gate/up K steps per item: some expand warps own no step of an item
    ((192, 128, 64), 4, 2, 90),      # 3 gate/up K steps, 2 down K steps per item
    ((2048, 1408, 128), 8, 4, 96),   # Qwen-like expert shape: 11 row blocks of 128, down K of 22 steps
])
def test_grouped_shapes(shape, E, k, T):
    _case(shape, E, k, False, T, 42, zero="int")


def test_grouped_olmoe_prefill_layer_sampled():
    # One OLMoE-shaped prefill layer: 512 tokens, uniform logits, 4096 pairs
    # over 64 experts; the oracle checks a sample of tokens.
    _case((2048, 1024, 128), 64, 8, False, 512, 43, kind="uniform",
          sample=[0, 1, 77, 255, 256, 400, 510, 511])


def test_grouped_matches_gemv_path():
    shape, E, k, T = (2048, 1024, 128), 64, 8, 16
    lp = LayerPool(moe, 44, 0, shape, E)
    x = synth.activations(44, 1, T, 2048)
    lg = synth.logits_normal(44, 3, T, E)
    ya, ida, _, fa = run_layer(moe, lp, x, lg, k, False, GROUPED)
    yb, idb, _, fb = run_layer(moe, lp, x, lg, k, False, 1)
    assert fa == 0 and fb == 0 and np.array_equal(ida, idb)
    ok, err, bound = tol_ok(ya, yb, rel=3e-3)
    assert ok, (err, bound)


def test_grouped_deterministic():
    a = _case((512, 256, 128), 16, 4, False, 64, 45)
    b = _case((512, 256, 128), 16, 4, False, 64, 45)
    assert np.array_equal(a, b)


def test_grouped_auto_path_above_gemv_limit():
    # 40 tokens x 8 choices = 320 pairs > 256: MOE_PATH_AUTO takes the grouped path.
    _case((512, 256, 128), 16, 8, False, 40, 46, path=0)


def test_grouped_absent_expert_and_bad_token():
    shape, E, k, T = (256, 128, 64), 8, 2, 6
    lp = LayerPool(moe, 47, 0, shape, E)
    lp.slot_of[3] = -1
    x = synth.activations(47, 1, T, 256)
    lg = np.zeros((T, E), np.float32)
    lg[:, 3] = 5.0
    lg[:, 1] = 4.0
    lg[2, 0] = np.nan  # token 2: no routing
    y, ids, w, flags = run_layer(moe, lp, x, lg, k, True, GROUPED)
    assert flags & 1
    assert ids[2].tolist() == [-1, -1] and np.all(y[2] == 0)
    wg, wu, wd = moe_oracle.dequantize_expert(lp.arrays(1), 64)
    for t in [0, 1, 3, 4, 5]:
        j1 = list(ids[t]).index(1)
        want = w[t, j1] * moe_oracle.expert_ffn(x[t], wg, wu, wd)
        ok, err, bound = tol_ok(y[t], want)
        assert ok, (t, err, bound)


def test_grouped_workspace_reuse():
    # Two different batches on one workspace: no state leaks between calls.
    shape, E, k = (512, 256, 128), 16, 4
    lp = LayerPool(moe, 48, 0, shape, E)
    dev = torch.device("cuda")
    ws = torch.zeros(moe.moe_forward_workspace_bytes(shape, 100, k, E, GROUPED), dtype=torch.uint8, device=dev)
    for rep, T in enumerate((100, 37)):
        x = synth.activations(48, rep, T, 512)
        lg = synth.logits_normal(48, rep, T, E)
        ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        w = torch.empty((T, k), dtype=torch.float32, device=dev)
        moe.moe_route(torch.from_numpy(lg).to(dev), k, False, ids, w)
        y = torch.empty((T, 512), dtype=torch.float16, device=dev)
        moe.moe_expert_forward(shape, torch.from_numpy(x).to(dev), ids, w, E, lp.pool, lp.slot_of, E, None, y,
                               ws, GROUPED)
        assert moe.moe_workspace_flags(ws) == 0
        ref = moe_oracle.moe_layer(x, lg, lp.arrays, k, False, 128)
        ok, err, bound = tol_ok(y.float().cpu().numpy(), ref["y"])
        assert ok, (rep, err, bound)


@pytest.mark.parametrize("shape,E,k,T", [
    ((8192, 128, 128), 2, 1, 48),   # largest hidden: 128 K steps of the gate/up GEMM
    ((256, 8192, 64), 2, 1, 40),    # largest intermediate: 64 row blocks, 128 K steps of the down GEMM
])
def test_grouped_maximum_sizes(shape, E, k, T):
    _case(shape, E, k, False, T, 49, zero="int")


def test_grouped_empty_batch():
    shape, E, k = (256, 128, 64), 8, 2
    lp = LayerPool(moe, 50, 0, shape, E)
    dev = torch.device("cuda")
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    x = torch.empty((0, 256), dtype=torch.float16, device=dev)
    ids = torch.empty((0, k), dtype=torch.int32, device=dev)
    w = torch.empty((0, k), dtype=torch.float32, device=dev)
    y = torch.empty((0, 256), dtype=torch.float16, device=dev)
    moe.moe_expert_forward(shape, x, ids, w, E, lp.pool, lp.slot_of, E, None, y, ws, GROUPED)
    torch.cuda.synchronize()
    assert moe.moe_workspace_flags(ws) == 0
