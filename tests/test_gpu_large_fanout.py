"""The 512-expert top-10 layer (hidden 2048, expert intermediate 512, INT4
group 128, renormalised routing, Zipf(1.1) expert popularity) at the batch
sizes of the large fan-out stack -- 1, 16 and 256 tokens -- on the path
MOE_PATH_AUTO picks, against the CPU oracle (needs a GB300).

Workload: "Desenvolvedor do Strata cria mapa ao vivo de 24 576 especialistas
MoE em uma GTX 1070", section "Como 125 bilhões de parâmetros cabem em 8 GB"
(48 x 512 experts); lucashiago.com.br "local" explainer, etapa 3 (512 experts,
10 active per token; distinct experts touched by n tokens).
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

SHAPE = (2048, 512, 128)
E, K = 512, 10


@pytest.fixture(scope="module")
def pool():
    return LayerPool(moe, 70, 0, SHAPE, E)


def _layer(lp, T, tag, path=0):
    dev = torch.device("cuda")
    x16 = synth.activations(lp.seed, tag, T, SHAPE[0])
    lg = synth.logits_zipf(lp.seed, 0, tag, T, E, 1.1)
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    w = torch.empty((T, K), dtype=torch.float32, device=dev)
    y = torch.empty((T, SHAPE[0]), dtype=torch.float16, device=dev)
    ws = torch.zeros(moe.moe_forward_workspace_bytes(SHAPE, T, K, E, path), dtype=torch.uint8, device=dev)
    moe.moe_layer_forward(SHAPE, torch.from_numpy(x16).to(dev), torch.from_numpy(lg).to(dev), K, True, ids, w,
                          lp.pool, lp.slot_of, E, None, y, ws, path)
    assert moe.moe_workspace_flags(ws) == 0
    return x16, lg, ids.cpu().numpy(), w.cpu().numpy(), y.float().cpu().numpy()


@pytest.mark.parametrize("T,sample", [
    (1, None),
    (16, None),
    (256, [0, 1, 2, 63, 128, 200, 254, 255]),
])
def test_large_fanout_auto_path(pool, T, sample):
    x16, lg, ids, w, y = _layer(pool, T, 10 + T)
    rids, rw = moe_oracle.route(lg, K, True)
    assert np.array_equal(ids, rids)  # every token's routing, bit-exact
    assert np.allclose(w, rw, rtol=2e-6, atol=1e-9)
    rows = np.arange(T) if sample is None else np.asarray(sample)
    ref = moe_oracle.moe_layer(x16[rows], lg[rows], pool.arrays, K, True, SHAPE[2])
    ok, err, bound = tol_ok(y[rows], ref["y"])
    assert ok, (T, err, bound)


def test_large_fanout_b16_shares_experts(pool):
    # At 16 tokens the Zipf-popular experts repeat across tokens: fewer
    # distinct experts than (token, choice) pairs, each read once per call;
    # the streamed path and the grouped path agree.
    x16, lg, ids, w, y_auto = _layer(pool, 16, 90, path=0)
    assert len(np.unique(ids)) < ids.size
    _, _, ids_g, _, y_grp = _layer(pool, 16, 90, path=2)
    assert np.array_equal(ids, ids_g)
    ok, err, bound = tol_ok(y_auto, y_grp, rel=3e-3)
    assert ok, (err, bound)
