"""Helpers of the GPU parity tests: seeded inputs on the device, oracle
comparisons. Inputs come from the generator only; the pool is assembled with
the library's host pack call, the oracle reads the generator's arrays."""
import numpy as np
import torch

from int4_routed_expert_moe_gb300 import synth


class LayerPool:
    """E experts of one layer, packed into one device pool (slot e = expert e)."""

    def __init__(self, moe, seed, layer, shape, E, zero="eight"):
        self.moe, self.seed, self.layer, self.shape, self.E, self.zero = moe, seed, layer, shape, E, zero
        H, I, g = shape
        bb = moe.moe_expert_block_bytes(shape)
        host = torch.empty((E, bb), dtype=torch.uint8)
        hn = host.numpy()
        for e in range(E):
            moe.moe_pack_expert(shape, self.arrays(e), out=hn[e])
        self.pool = host.cuda()
        self.slot_of = torch.arange(E, dtype=torch.int32, device="cuda")
        self.block_bytes = bb

    def arrays(self, e):
        H, I, g = self.shape
        return synth.expert_arrays(self.seed, self.layer, e, H, I, g, zero=self.zero)


def tol_ok(got, ref, rel=5e-3):
    """max|got - ref| <= rel * max|ref| over the tensor; returns (ok, err, bound)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    bound = rel * float(np.max(np.abs(ref))) if ref.size else 0.0
    return err <= bound, err, bound


def run_layer(moe, lp, x16, logits, k, renorm, path, y_shared=None):
    T = x16.shape[0]
    H, I, g = lp.shape
    dev = torch.device("cuda")
    lg = torch.from_numpy(logits).to(dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    moe.moe_route(lg, k, renorm, ids, w)
    x = torch.from_numpy(x16).to(dev)
    y = torch.empty((T, H), dtype=torch.float16, device=dev)
    ysh = None if y_shared is None else torch.from_numpy(y_shared).to(dev)
    ws = torch.zeros(max(256, moe.moe_forward_workspace_bytes(lp.shape, T, k, lp.E, path)),
                     dtype=torch.uint8, device=dev)
    moe.moe_expert_forward(lp.shape, x, ids, w, lp.E, lp.pool, lp.slot_of, lp.E, ysh, y, ws, path)
    flags = moe.moe_workspace_flags(ws)
    return y.float().cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), flags
