"""Decode and grouped paths on activations that stress the FP16 arithmetic,
against the CPU oracle at the stated tolerance (needs a GB300).

"Horizon RunMap -- Prévia Técnica", "08 / Comportamento do modelo": FP16
activations, FP32 accumulation steps and explicit rounding points. The decode
kernels form FP16 products of at most 8 terms with a power-of-two scale per
32-element activation chunk; these cases put the chunk scale to work:
  (i)   one element per 32-element chunk 10^3 times the others;
  (ii)  every activation below the FP16 normal range (|x| < 2^-14);
  (iii) an activation at the FP16 maximum (65504) in every token.
Scales of the gate/up weights are chosen per case so that the SwiGLU
intermediate stays inside the FP16 range (h is rounded to FP16 on every
path), which the oracle, in FP64, does not model.
"""
import numpy as np
import pytest
import torch

from int4_routed_expert_moe_gb300 import synth
from oracle import moe_oracle
from tests._lib import binding
from tests.gpu_util import LayerPool, run_layer, tol_ok

pytestmark = pytest.mark.gpu

moe = binding() if torch.cuda.is_available() else None

SHAPE = (2048, 1024, 128)  # the OLMoE expert shape
E, K = 64, 8


class ScaledPool(LayerPool):
    """LayerPool whose gate/up scales are redrawn from U(lo, hi) (FP16)."""

    def __init__(self, seed, lo, hi):
        self.lo, self.hi = lo, hi
        super().__init__(moe, seed, 0, SHAPE, E, zero="int")

    def arrays(self, e):
        a = dict(super().arrays(e))
        r = np.random.default_rng([self.seed, 99, e])
        for name in ("s_gate", "s_up"):
            a[name] = r.uniform(self.lo, self.hi, size=a[name].shape).astype(np.float16)
        return a


def _acts(case, seed, T):
    r = np.random.default_rng([seed, 7])
    H = SHAPE[0]
    if case == "outlier":
        x = r.standard_normal((T, H)) * 1e-2
        for t in range(T):
            for c in range(H // 32):
                x[t, 32 * c + r.integers(32)] = r.choice([-10.0, 10.0])
    elif case == "subnormal":
        x = r.standard_normal((T, H)) * 2.0 ** -17
        x = np.clip(x, -(2.0 ** -14) * 0.99, (2.0 ** -14) * 0.99)
    else:  # fp16 max
        x = r.standard_normal((T, H))
        for t in range(T):
            x[t, r.integers(H)] = 65504.0 if t % 2 == 0 else -65504.0
    return x.astype(np.float16)


# Gate/up scale ranges that keep h inside the FP16 range for each case (and
# the grouped path's expanded operand 16 (q - z) s inside it: s <= 273).
SCALES = {"outlier": (1e-3, 1e-2), "subnormal": (20.0, 200.0), "fp16max": (1e-5, 1e-4)}


@pytest.fixture(scope="module", params=sorted(SCALES))
def case_pool(request):
    lo, hi = SCALES[request.param]
    return request.param, ScaledPool(60 + sorted(SCALES).index(request.param), lo, hi)


def _check(case, lp, T, path, layer_call):
    x = _acts(case, lp.seed, T)
    if case == "subnormal":
        assert np.all(np.abs(x.astype(np.float64)) < 2.0 ** -14)
    if case == "fp16max":
        assert np.all(np.max(np.abs(x.astype(np.float64)), axis=1) == 65504.0)
    lg = synth.logits_normal(lp.seed, 3, T, E)
    ref = moe_oracle.moe_layer(x, lg, lp.arrays, K, False, SHAPE[2])
    if layer_call:
        dev = torch.device("cuda")
        ids = torch.empty((T, K), dtype=torch.int32, device=dev)
        w = torch.empty((T, K), dtype=torch.float32, device=dev)
        y = torch.empty((T, SHAPE[0]), dtype=torch.float16, device=dev)
        ws = torch.zeros(moe.moe_forward_workspace_bytes(SHAPE, T, K, E, path), dtype=torch.uint8, device=dev)
        moe.moe_layer_forward(SHAPE, torch.from_numpy(x).to(dev), torch.from_numpy(lg).to(dev), K, False, ids, w,
                              lp.pool, lp.slot_of, E, None, y, ws, path)
        assert moe.moe_workspace_flags(ws) == 0
        y = y.float().cpu().numpy()
        assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    else:
        y, ids, _, flags = run_layer(moe, lp, x, lg, K, False, path)
        assert flags == 0 and np.array_equal(ids, ref["ids"])
    assert np.all(np.isfinite(ref["y"])) and np.max(np.abs(ref["y"])) < 6e4
    ok, err, bound = tol_ok(y, ref["y"])
    assert ok, (case, path, err, bound)


@pytest.mark.parametrize("T", [1, 4])
def test_decode_layer_adversarial(case_pool, T):
    case, lp = case_pool
    _check(case, lp, T, 1, layer_call=True)


def test_decode_expert_forward_adversarial(case_pool):
    case, lp = case_pool
    _check(case, lp, 2, 1, layer_call=False)


def test_unfused_gemv_adversarial(case_pool):
    case, lp = case_pool
    _check(case, lp, 2, 3, layer_call=False)


def test_grouped_adversarial(case_pool):
    case, lp = case_pool
    _check(case, lp, 24, 2, layer_call=False)
