"""moe_layer_forward_noalloc against moe_layer_forward (needs a GB300).

The no-allocation entry point serves callers that cannot allocate device
memory (under a host framework that owns all allocations, or with a fixed
memory budget): its scratch is a fixed array inside the library instead of
a caller workspace. Two calls in
a row on different inputs must each match the workspace entry point within
the tolerance the parity tests use. This file is collected last so that a
failure here comes after every other test has run."""
import numpy as np
import pytest
import torch

from int4_routed_expert_moe_gb300 import synth
from tests._lib import binding
from tests.gpu_util import LayerPool, tol_ok

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,E,k,renorm,T", [((2048, 1024, 128), 64, 8, False, 1),
                                                ((256, 128, 64), 8, 2, True, 4),
                                                ((2048, 512, 128), 512, 10, True, 2)])
def test_noalloc_matches_workspace_entry_point_twice(shape, E, k, renorm, T):
    moe = binding()
    H = shape[0]
    dev = torch.device("cuda")
    lp = LayerPool(moe, 61, 0, shape, E)
    ws = torch.zeros(moe.moe_forward_workspace_bytes(shape, T, k, E, moe.MOE_PATH_GEMV),
                     dtype=torch.uint8, device=dev)
    for call in range(2):
        x = torch.from_numpy(synth.activations(61, call, T, H)).to(dev)
        lg = torch.from_numpy(synth.logits_normal(61, call, T, E)).to(dev)
        ids_a = torch.empty((T, k), dtype=torch.int32, device=dev)
        w_a = torch.empty((T, k), dtype=torch.float32, device=dev)
        y_a = torch.empty((T, H), dtype=torch.float16, device=dev)
        moe.moe_layer_forward(shape, x, lg, k, renorm, ids_a, w_a, lp.pool, lp.slot_of, E, None, y_a, ws,
                              moe.MOE_PATH_GEMV)
        ids_b = torch.full((T, k), -7, dtype=torch.int32, device=dev)
        w_b = torch.empty((T, k), dtype=torch.float32, device=dev)
        y_b = torch.empty((T, H), dtype=torch.float16, device=dev)
        moe.moe_layer_forward_noalloc(shape, x, lg, k, renorm, ids_b, w_b, lp.pool, lp.slot_of, E, None, y_b)
        assert moe.moe_layer_forward_noalloc_flags() == 0, call
        assert moe.moe_workspace_flags(ws) == 0, call
        assert np.array_equal(ids_a.cpu().numpy(), ids_b.cpu().numpy()), call
        assert np.allclose(w_a.cpu().numpy(), w_b.cpu().numpy(), rtol=1e-6, atol=0), call
        ok, err, bound = tol_ok(y_b.float().cpu().numpy(), y_a.float().cpu().numpy())
        assert ok, (call, err, bound)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    moe = binding()
    shape, E, k = (2048, 1024, 128), 64, 8
    T = 64  # 64 * 8 * 1024 * 2 bytes = 1 MiB of intermediate, plus headers: too large
    dev = torch.device("cuda")
    lp = LayerPool(moe, 62, 0, (256, 128, 64), 8)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward_noalloc(
            shape, torch.zeros((T, 2048), dtype=torch.float16, device=dev),
            torch.zeros((T, E), dtype=torch.float32, device=dev), k, False,
            torch.empty((T, k), dtype=torch.int32, device=dev), torch.empty((T, k), device=dev),
            torch.zeros(E * moe.moe_expert_block_bytes(shape), dtype=torch.uint8, device=dev),
            torch.arange(E, dtype=torch.int32, device=dev), E, None,
            torch.empty((T, 2048), dtype=torch.float16, device=dev))
    assert ei.value.status == moe.MOE_ERR_CAPACITY
    del lp
