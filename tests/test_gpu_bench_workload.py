"""Parity at full size on the benchmark's own workloads (needs a GB300).

The decode stacks that bench.py times -- OLMoE-shaped (16 layers x 64 experts
of hidden 2048 / intermediate 1024, top-8) and Qwen-like (24 layers x 60
experts, intermediate 1408, top-4) -- generated on the device. For sampled layers
the same moe_layer_forward call bench.py makes run on fresh
N(0,1) activations, and the oracle recomputes the layer from the expert
blocks read back from the pool (inputs, read before the kernels run)."""
import numpy as np
import pytest
import torch

from int4_routed_expert_moe_gb300 import synth
from oracle import moe_oracle
from tests._lib import binding
from tests.gpu_util import tol_ok

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,seed,layers", [("olmoe_decode", 1, (0, 7, 15)), ("qwen_decode", 6, (0, 11, 23))])
def test_bench_decode_workload_sampled_layers(name, seed, layers):
    moe = binding()
    import bench
    wl = bench.DecodeWorkload(moe, synth.BASE_SEED + seed, 4, name=name)
    dev = torch.device("cuda")
    for l in layers:
        pool = wl.layer_pool(l)
        lg = wl.logits[1, l]
        ids_ref, _ = moe_oracle.route(lg.cpu().numpy(), wl.k, wl.renorm)
        experts = {int(e): synth.arrays_from_block(pool[int(e)].cpu().numpy(), *wl.shape)
                   for e in ids_ref.reshape(-1)}
        x16 = synth.activations(99, l, wl.T, wl.H)
        x = torch.from_numpy(x16).to(dev)
        moe.moe_layer_forward(wl.shape, x, lg, wl.k, wl.renorm, wl.ids[l], wl.w[l], pool, wl.slot_of,
                              wl.E, None, wl.y[l], wl.ws, moe.MOE_PATH_GEMV)
        torch.cuda.synchronize()
        assert moe.moe_workspace_flags(wl.ws) == 0
        ref = moe_oracle.moe_layer(x16, lg.cpu().numpy(), experts, wl.k, wl.renorm, wl.g)
        assert np.array_equal(wl.ids[l].cpu().numpy(), ref["ids"])
        ok, err, bound = tol_ok(wl.y[l].float().cpu().numpy(), ref["y"])
        assert ok, (l, err, bound)
