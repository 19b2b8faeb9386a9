"""CUDA path vs the CPU oracle, called through the C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

from int4_routed_expert_moe_gb300 import synth
from oracle import moe_oracle
from tests._lib import binding
from tests.gpu_util import LayerPool, run_layer, tol_ok

pytestmark = pytest.mark.gpu

moe = binding() if torch.cuda.is_available() else None


def _route_gpu(logits, k, renorm):
    dev = torch.device("cuda")
    T = logits.shape[0]
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    bad = torch.zeros(1, dtype=torch.int32, device=dev)
    moe.moe_route(torch.from_numpy(np.ascontiguousarray(logits)).to(dev), k, renorm, ids, w, bad)
    return ids.cpu().numpy(), w.cpu().numpy(), int(bad.item())


@pytest.mark.parametrize("T,E,k,renorm,kind", [
    (4, 8, 2, True, "normal"), (1, 64, 8, False, "normal"), (512, 64, 8, False, "uniform"),
    (16, 512, 10, True, "zipf"), (256, 512, 10, True, "zipf"), (3, 32, 32, True, "normal"),
    (7, 2000, 32, False, "normal"), (33, 100, 5, True, "normal"), (1, 1, 1, True, "normal"),
])
def test_route_matches_oracle(T, E, k, renorm, kind):
    if kind == "zipf":
        lg = synth.logits_zipf(5, 0, T, T, E, 1.1)
    elif kind == "uniform":
        lg = synth.logits_uniform(5, T, T, E)
    else:
        lg = synth.logits_normal(5, T * 7 + E, T, E)
    ids, w, bad = _route_gpu(lg, k, renorm)
    rids, rw = moe_oracle.route(lg, k, renorm)
    assert bad == 0
    assert np.array_equal(ids, rids)
    assert np.allclose(w, rw, rtol=2e-6, atol=1e-9)


def test_route_ties_and_nonfinite():
    lg = np.array([[1, 3, 3, 2, 3, 0, 0, 0], [0, 0, 0, 0, 0, 0, 0, 0],
                   [-np.inf, 1, -np.inf, 0, -np.inf, -np.inf, -np.inf, -np.inf],
                   [-0.0, 0.0, -0.0, 0.0, -1, -1, -1, -1]], dtype=np.float32)
    for renorm in (True, False):
        ids, w, bad = _route_gpu(lg, 3, renorm)
        rids, rw = moe_oracle.route(lg, 3, renorm)
        assert bad == 0 and np.array_equal(ids, rids)
        assert np.allclose(w, rw, rtol=2e-6, atol=1e-12)
    bad_lg = np.array([[0, np.nan, 1, 2], [0, 1, 2, 3], [np.inf, 0, 0, 0],
                       [-np.inf] * 4], dtype=np.float32)
    ids, w, bad = _route_gpu(bad_lg, 2, True)
    assert bad == 3
    assert ids[0].tolist() == [-1, -1] and ids[2].tolist() == [-1, -1] and ids[3].tolist() == [-1, -1]
    assert ids[1].tolist() == [3, 2] and np.all(w[0] == 0)


@pytest.mark.parametrize("T,k,E", [(4, 2, 8), (512, 8, 64), (256, 10, 512), (1, 8, 64),
                                   (4096, 16, 1024), (0, 8, 64), (1000, 3, 7)])
def test_token_sort_matches_oracle(T, k, E):
    r = np.random.default_rng(T + E)
    ids = np.zeros((T, k), dtype=np.int32)
    for t in range(T):
        ids[t] = r.permutation(E)[:k]
    dev = torch.device("cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    pt = torch.full((max(1, T * k),), -7, dtype=torch.int32, device=dev)
    pj = torch.full((max(1, T * k),), -7, dtype=torch.int32, device=dev)
    moe.moe_token_sort(torch.from_numpy(ids).to(dev), E, off, pt, pj)
    roff, rpt, rpj = moe_oracle.token_sort(ids, E)
    assert np.array_equal(off.cpu().numpy(), roff)
    if T:
        assert np.array_equal(pt.cpu().numpy(), rpt)
        assert np.array_equal(pj.cpu().numpy(), rpj)


def test_token_sort_drops_invalid_ids():
    ids = np.array([[1, -1], [3, 1], [9, 0]], dtype=np.int32)
    dev = torch.device("cuda")
    off = torch.empty(5, dtype=torch.int32, device=dev)
    pt = torch.full((6,), -7, dtype=torch.int32, device=dev)
    pj = torch.full((6,), -7, dtype=torch.int32, device=dev)
    moe.moe_token_sort(torch.from_numpy(ids).to(dev), 4, off, pt, pj)
    assert off.cpu().tolist() == [0, 1, 3, 3, 4]
    assert pt.cpu().tolist()[:4] == [2, 0, 1, 1] and pj.cpu().tolist()[:4] == [1, 0, 1, 0]


def _layer_case(shape, E, k, renorm, T, seed, zero="eight", path=1, shared=False,
                logit_kind="normal"):
    H, I, g = shape
    lp = LayerPool(moe, seed, 0, shape, E, zero=zero)
    x = synth.activations(seed, 1, T, H)
    if logit_kind == "zipf":
        lg = synth.logits_zipf(seed, 0, 3, T, E, 1.1)
    elif logit_kind == "uniform":
        lg = synth.logits_uniform(seed, 3, T, E)
    else:
        lg = synth.logits_normal(seed, 3, T, E)
    ysh = synth.activations(seed, 2, T, H) if shared else None
    y, ids, w, flags = run_layer(moe, lp, x, lg, k, renorm, path, y_shared=ysh)
    ref = moe_oracle.moe_layer(x, lg, lp.arrays, k, renorm, g, y_shared=ysh)
    assert flags == 0
    assert np.array_equal(ids, ref["ids"])
    ok, err, bound = tol_ok(y, ref["y"])
    assert ok, (err, bound)
    return y


GEMV_PATHS = [1, 3]  # streamed decode kernels, unfused two-kernel GEMV


@pytest.mark.parametrize("path", GEMV_PATHS)
@pytest.mark.parametrize("zero", ["eight", "int", "frac"])
@pytest.mark.parametrize("shared", [False, True])
def test_gemv_tiny_layer(zero, shared, path):
    _layer_case((256, 128, 64), 8, 2, True, 4, 31, zero=zero, path=path, shared=shared)


@pytest.mark.parametrize("path", GEMV_PATHS)
@pytest.mark.parametrize("T", [1, 3])
def test_gemv_olmoe_layer(T, path):
    _layer_case((2048, 1024, 128), 64, 8, False, T, 32, path=path)


@pytest.mark.parametrize("path", GEMV_PATHS)
def test_gemv_large_fanout_layer_b16(path):
    _layer_case((2048, 512, 128), 512, 10, True, 16, 33, path=path, logit_kind="zipf")


@pytest.mark.parametrize("path", GEMV_PATHS)
@pytest.mark.parametrize("shape,E,k", [((512, 192, 64), 6, 3), ((1088, 320, 32), 5, 2),
                                       ((8192, 64, 64), 3, 1), ((256, 8192, 64), 3, 1),
                                       ((2048, 1024, 128), 64, 8)])
def test_gemv_ragged_shapes(shape, E, k, path):
    # H not a multiple of 1024 (partial lane loop), I and H not multiples of
    # the block count (ragged row slices), scale rows not 16-byte multiples,
    # the largest H, the largest I; and 16 tokens x 8 choices = 128 pairs (ring reuse).
    T = 16 if shape == (2048, 1024, 128) else 2
    _layer_case(shape, E, k, False, T, 34, zero="int", path=path)


@pytest.mark.parametrize("path", GEMV_PATHS)
def test_gemv_deterministic(path):
    a = _layer_case((2048, 1024, 128), 64, 8, False, 1, 35, path=path)
    b = _layer_case((2048, 1024, 128), 64, 8, False, 1, 35, path=path)
    assert np.array_equal(a, b)


def test_gemv_fused_workspace_reuse_and_agreement():
    # Several calls on one workspace (the fused kernel resets its counters),
    # and the fused and unfused kernels agree to FP16 rounding.
    shape, E, k, T = (2048, 1024, 128), 64, 8, 2
    lp = LayerPool(moe, 38, 0, shape, E)
    dev = torch.device("cuda")
    ws = torch.zeros(moe.moe_forward_workspace_bytes(shape, T, k, E, 1), dtype=torch.uint8, device=dev)
    outs = []
    for rep in range(3):
        x = torch.from_numpy(synth.activations(38, rep, T, 2048)).to(dev)
        lg = torch.from_numpy(synth.logits_normal(38, rep, T, E)).to(dev)
        ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        w = torch.empty((T, k), dtype=torch.float32, device=dev)
        moe.moe_route(lg, k, False, ids, w)
        ys = []
        for path in (1, 3):
            y = torch.empty((T, 2048), dtype=torch.float16, device=dev)
            moe.moe_expert_forward(shape, x, ids, w, E, lp.pool, lp.slot_of, E, None, y, ws, path)
            ys.append(y.float().cpu().numpy())
        assert moe.moe_workspace_flags(ws) == 0
        ok, err, bound = tol_ok(ys[0], ys[1], rel=2e-3)
        assert ok, (rep, err, bound)
        outs.append(ys[0])
    ws_words = ws[:1024].view(torch.int32).cpu().numpy()
    assert ws_words[1] == 0 and np.all(ws_words[64:64 + T * k] == 0)  # counters back to zero


def test_gemv_absent_expert_flags_and_skips():
    shape, E, k, T = (256, 128, 64), 8, 2, 4
    lp = LayerPool(moe, 36, 0, shape, E)
    lp.slot_of[3] = -1
    x = synth.activations(36, 1, T, 256)
    lg = np.zeros((T, E), np.float32)
    lg[:, 3] = 5.0
    lg[:, 1] = 4.0
    y, ids, w, flags = run_layer(moe, lp, x, lg, k, True, 1)
    assert flags & 1
    # expert 3 contributes nothing: y = w1 * o_1
    ref_ids, ref_w = moe_oracle.route(lg, k, True)
    wg, wu, wd = moe_oracle.dequantize_expert(lp.arrays(1), 64)
    for t in range(T):
        j1 = list(ref_ids[t]).index(1)
        want = ref_w[t, j1] * moe_oracle.expert_ffn(x[t], wg, wu, wd)
        ok, err, bound = tol_ok(y[t], want)
        assert ok, (t, err, bound)


def test_gemv_bad_token_contributes_nothing():
    shape, E, k, T = (256, 128, 64), 8, 2, 3
    lp = LayerPool(moe, 37, 0, shape, E)
    x = synth.activations(37, 1, T, 256)
    lg = synth.logits_normal(37, 3, T, E)
    lg[1, 4] = np.nan
    y, ids, w, flags = run_layer(moe, lp, x, lg, k, True, 1)
    assert flags == 0 and ids[1].tolist() == [-1, -1]
    assert np.all(y[1] == 0)
    ref = moe_oracle.moe_layer(x[[0, 2]], lg[[0, 2]], lp.arrays, k, True, 64)
    ok, err, bound = tol_ok(y[[0, 2]], ref["y"])
    assert ok


def _layer_forward_case(shape, E, k, renorm, T, seed, logits=None, shared=False, path=1):
    H, I, g = shape
    lp = LayerPool(moe, seed, 0, shape, E)
    dev = torch.device("cuda")
    x16 = synth.activations(seed, 1, T, H)
    lg = synth.logits_normal(seed, 3, T, E) if logits is None else logits
    ysh = synth.activations(seed, 2, T, H) if shared else None
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    y = torch.empty((T, H), dtype=torch.float16, device=dev)
    ws = torch.zeros(moe.moe_forward_workspace_bytes(shape, T, k, E, path), dtype=torch.uint8, device=dev)
    moe.moe_layer_forward(shape, torch.from_numpy(x16).to(dev), torch.from_numpy(lg).to(dev), k, renorm,
                          ids, w, lp.pool, lp.slot_of, E,
                          None if ysh is None else torch.from_numpy(ysh).to(dev), y, ws, path)
    assert moe.moe_workspace_flags(ws) == 0
    good = [t for t in range(T) if np.all(np.isfinite(lg[t]) | (lg[t] == -np.inf)) and not np.all(lg[t] == -np.inf)]
    ref = moe_oracle.moe_layer(x16[good], lg[good], lp.arrays, k, renorm, g,
                               y_shared=None if ysh is None else ysh[good])
    got_ids = ids.cpu().numpy()
    assert np.array_equal(got_ids[good], ref["ids"])
    assert np.allclose(w.cpu().numpy()[good], ref["weights"], rtol=2e-6, atol=1e-9)
    ok, err, bound = tol_ok(y.float().cpu().numpy()[good], ref["y"])
    assert ok, (err, bound)
    return got_ids, y.float().cpu().numpy()


@pytest.mark.parametrize("shape,E,k,renorm,T,shared", [
    ((256, 128, 64), 8, 2, True, 4, True),          # tiny, shared path added
    ((2048, 1024, 128), 64, 8, False, 1, False),    # OLMoE decode: routing inside the kernels
    ((2048, 1024, 128), 64, 8, False, 3, False),
    ((2048, 512, 128), 512, 10, True, 1, False),    # large fan-out, in-kernel routing (E^2 = 2^18)
    ((2048, 512, 128), 512, 10, True, 16, False),   # routing kernel first (T*E^2 too large)
])
def test_layer_forward_matches_oracle(shape, E, k, renorm, T, shared):
    _layer_forward_case(shape, E, k, renorm, T, 40 + T, shared=shared)


def test_layer_forward_ties_and_bad_tokens():
    E = 8
    lg = np.array([[1, 3, 3, 2, 3, 0, 0, 0], [0, 0, 0, 0, 0, 0, 0, 0],
                   [-np.inf, 1, -np.inf, 0, -np.inf, -np.inf, -np.inf, -np.inf],
                   [0, np.nan, 1, 2, 0, 0, 0, 0], [-np.inf] * 8], dtype=np.float32)
    ids, y = _layer_forward_case((256, 128, 64), E, 3, False, 5, 44, logits=lg)
    assert ids[3].tolist() == [-1, -1, -1] and ids[4].tolist() == [-1, -1, -1]
    assert np.all(y[3] == 0) and np.all(y[4] == 0)


_ONE_TOKEN_ROWS = [[1, 3, 3, 2, 3, 0, 0, 0], [0, 0, 0, 0, 0, 0, 0, 0],
                   [-np.inf, 1, -np.inf, 0, -np.inf, -np.inf, -np.inf, -np.inf],
                   [0, np.nan, 1, 2, 0, 0, 0, 0], [-np.inf] * 8, [np.inf, 0, 0, 0, 0, 0, 0, 0],
                   [-0.0, 0.0, -0.0, 0.0, 1, 1, -1, -1]]


@pytest.mark.parametrize("row", range(len(_ONE_TOKEN_ROWS)))
def test_layer_forward_one_token_ties_and_bad(row):
    # One token routed inside the kernels: ties by lower index, -inf last,
    # a NaN/+inf or all -inf token chooses nobody and contributes 0.
    lg = np.array([_ONE_TOKEN_ROWS[row]], dtype=np.float32)
    ids, y = _layer_forward_case((256, 128, 64), 8, 3, False, 1, 45, logits=lg)
    if row in (3, 4, 5):
        assert ids[0].tolist() == [-1, -1, -1] and np.all(y == 0)


@pytest.mark.parametrize("shape,E,k,renorm", [
    ((512, 192, 64), 40, 8, True),      # E not a multiple of 32
    ((2048, 1408, 128), 60, 4, False),  # Qwen-like expert count
    ((1088, 320, 32), 5, 2, False),     # E below one warp
    ((512, 256, 64), 64, 8, False),     # k = the ring's stage count
])
def test_layer_forward_one_token_shapes(shape, E, k, renorm):
    _layer_forward_case(shape, E, k, renorm, 1, 46)


def _routing_rows(E, k, seed):
    # Token 0: one lane's experts (5, 37, 69, ...) hold the largest logits, so
    # one warp lane owns every pick; token 1: a few values only, +0/-0 mixed
    # (ties by index); token 2: fewer finite logits than k, the rest -inf;
    # token 3: normal logits.
    r = np.random.default_rng([seed, 5])
    lg = r.standard_normal((4, E)).astype(np.float32)
    own = np.arange(5, E, 32)
    lg[0, own] = 10.0 + np.arange(len(own))[::-1]
    lg[1] = r.choice(np.array([-0.0, 0.0, 1.0, 2.0], dtype=np.float32), size=E)
    lg[2] = -np.inf
    lg[2, r.choice(E, size=max(1, k // 2), replace=False)] = r.standard_normal(max(1, k // 2))
    return lg


@pytest.mark.parametrize("E,k", [(64, 8), (100, 12), (512, 10), (1024, 32)])
def test_layer_forward_batched_routing_edges(E, k):
    # Several tokens routed inside the kernels (one warp per token): picks by
    # (logit desc, index asc) whatever lane holds them, ties by index.
    lg = _routing_rows(E, k, 47)
    _layer_forward_case((256, 128, 64), E, k, False, 4, 47, logits=lg)


def test_one_token_h_words_across_calls_and_paths():
    # One token's h crosses the blocks as words marked with a per-call
    # counter: a sequence of one-token calls on one workspace, with a
    # several-token call (FP16 h in the same bytes) in between, must each use
    # only its own words.
    shape, E, k = (2048, 1024, 128), 64, 8
    lp = LayerPool(moe, 48, 0, shape, E)
    dev = torch.device("cuda")
    ws = torch.zeros(moe.moe_forward_workspace_bytes(shape, 2, k, E, 1), dtype=torch.uint8, device=dev)
    for i, T in enumerate([1, 2, 1, 1, 2, 1]):
        x16 = synth.activations(48, 10 + i, T, shape[0])
        lg = synth.logits_normal(48, 20 + i, T, E)
        ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        w = torch.empty((T, k), dtype=torch.float32, device=dev)
        y = torch.empty((T, shape[0]), dtype=torch.float16, device=dev)
        moe.moe_layer_forward(shape, torch.from_numpy(x16).to(dev), torch.from_numpy(lg).to(dev), k, False, ids, w,
                              lp.pool, lp.slot_of, E, None, y, ws, 1)
        assert moe.moe_workspace_flags(ws) == 0
        ref = moe_oracle.moe_layer(x16, lg, lp.arrays, k, False, shape[2])
        ok, err, bound = tol_ok(y.float().cpu().numpy(), ref["y"])
        assert ok, (i, T, err, bound)
