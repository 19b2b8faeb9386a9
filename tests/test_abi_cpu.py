"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and its host-only calls (layout, pack/unpack, argument checks) behave."""
import os
import re

import numpy as np
import pytest

from int4_routed_expert_moe_gb300 import synth
from tests._lib import ROOT, binding

moe = binding()


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    import ctypes
    lib = ctypes.CDLL(moe.lib_path())
    names = header_functions()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(names) == set(moe.EXPORTED), set(names) ^ set(moe.EXPORTED)


def test_status_strings_and_version():
    assert moe.moe_version() == 1
    assert moe.moe_status_string(0) == "MOE_OK"
    assert moe.moe_status_string(-3) == "MOE_ERR_CAPACITY"
    assert moe.moe_status_string(-99) == "MOE_ERR_UNKNOWN"


@pytest.mark.parametrize("shape,want", [((256, 128, 64), 57344), ((2048, 1024, 128), 3342336),
                                         ((2048, 512, 128), 1671168), ((192, 64, 64), 64 * 224 + 192 * 48),
                                         ((2048, 1408, 128), 1408 * 2176 + 2048 * 752)])
def test_block_layout(shape, want):
    # Unpadded shapes hold exactly 3*H*I/2 + 3*(H*I/g)*4 bytes; rows whose
    # contents are not a 16-byte multiple are padded (tiny: down rows 72 -> 80;
    # Qwen-like inter 1408: down rows 748 -> 752).
    H, I, g = shape
    assert moe.moe_expert_block_bytes(shape) == want
    lay = moe.moe_expert_block_layout(shape)
    assert lay["total"] == want and lay["d_offset"] == I * lay["gu_row_bytes"]
    assert lay["gu_row_bytes"] % 16 == 0 and lay["d_row_bytes"] % 16 == 0
    assert lay["gu_q_up"] == H // 2 and lay["gu_sz"] == H and lay["d_sz"] == I // 2
    assert lay["gu_sz"] + 8 * (H // g) <= lay["gu_row_bytes"]
    assert lay["d_sz"] + 4 * (I // g) <= lay["d_row_bytes"]
    syn = synth.block_layout(H, I, g)
    assert (syn["gu_row"], syn["d_row"], syn["total"]) == (lay["gu_row_bytes"], lay["d_row_bytes"], want)


@pytest.mark.parametrize("shape", [(0, 128, 64), (256, 100, 64), (256, 128, 48), (256, 128, 96),
                                   (16384, 128, 64)])
def test_invalid_shapes(shape):
    assert moe.moe_expert_block_bytes(shape) == 0
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_expert_block_layout(shape)
    assert ei.value.status == moe.MOE_ERR_SHAPE


@pytest.mark.parametrize("zero", ["eight", "int", "frac"])
def test_pack_unpack_round_trip(zero):
    H, I, g = 256, 128, 64
    arrs = synth.expert_arrays(3, 0, 5, H, I, g, zero=zero)
    # every code value appears, at both nibble positions
    arrs["qp_gate"][0, :16] = np.arange(16, dtype=np.uint8) * 17
    blk = moe.moe_pack_expert((H, I, g), arrs)
    assert blk.nbytes == moe.moe_expert_block_bytes((H, I, g))
    back = moe.moe_unpack_expert((H, I, g), blk)
    for n, a in arrs.items():
        assert np.array_equal(back[n].view(np.uint8), a.view(np.uint8)), n
    lay = moe.moe_expert_block_layout((H, I, g))
    gu = blk[:lay["d_offset"]].reshape(I, lay["gu_row_bytes"])
    assert np.array_equal(gu[:, :H // 2], arrs["qp_gate"])
    assert np.array_equal(gu[:, H // 2:H], arrs["qp_up"])
    # the generator's reader of block bytes agrees with the library's packer
    back2 = synth.arrays_from_block(blk, H, I, g)
    for n, a in arrs.items():
        assert np.array_equal(back2[n].view(np.uint8), a.view(np.uint8)), n


def test_gpu_entry_points_reject_bad_arguments_before_touching_the_gpu():
    import ctypes
    lib = moe._lib
    # k > E, k = 0, E too large: rejected on the host.
    assert lib.moe_route(None, 4, 8, 9, 1, None, None, None, None) == moe.MOE_ERR_ARG
    assert lib.moe_route(None, 4, 8, 0, 1, None, None, None, None) == moe.MOE_ERR_ARG
    assert lib.moe_route(None, 4, 5000, 2, 1, None, None, None, None) == moe.MOE_ERR_ARG
    assert lib.moe_route(None, 0, 8, 2, 1, None, None, None, None) == moe.MOE_OK  # T = 0: no-op
    assert lib.moe_token_sort(None, 4, 2, 2000, None, None, None, None) == moe.MOE_ERR_ARG
    s = moe.moe_expert_shape(256, 128, 64)
    bad = moe.moe_expert_shape(256, 100, 64)
    assert lib.moe_expert_forward(ctypes.byref(bad), None, 1, None, None, 2, 8, None, None, 8,
                                  None, None, None, 0, 0, None) == moe.MOE_ERR_SHAPE
    assert lib.moe_expert_forward(ctypes.byref(s), None, 1, None, None, 2, 8, None, None, 8,
                                  None, None, None, 0, 7, None) == moe.MOE_ERR_ARG
    assert lib.moe_expert_forward(ctypes.byref(s), None, 0, None, None, 2, 8, None, None, 8,
                                  None, None, None, 0, 0, None) == moe.MOE_OK
    assert "path" in moe.moe_last_error() or moe.moe_last_error() == ""


def test_workspace_sizes():
    s = (2048, 1024, 128)
    assert moe.moe_forward_workspace_bytes(s, 1, 8, 64, moe.MOE_PATH_GEMV) == 512 + 8 * 1024 * 4
    assert moe.moe_forward_workspace_bytes((2048, 100, 128), 1, 8, 64) == 0


@pytest.mark.parametrize("shape", [(256, 128, 64), (2048, 512, 128), (192, 64, 64)])
def test_device_pool_generator_layout_matches_library(shape):
    # The generator's device-side pool (run here on the CPU device) and its
    # reader agree with the library's unpacker byte for byte.
    H, I, g = shape
    pool = synth.device_pool(2, H, I, g, seed=3, device="cpu").numpy()
    for b in range(2):
        lib = moe.moe_unpack_expert(shape, pool[b])
        syn = synth.arrays_from_block(pool[b], H, I, g)
        for n in lib:
            assert np.array_equal(lib[n].view(np.uint8), syn[n].view(np.uint8)), n
        for n in ("s_gate", "s_up", "s_down"):
            v = lib[n].astype(np.float64)
            assert v.min() >= 9e-4 and v.max() <= 1.01e-2
        for n in ("z_gate", "z_up", "z_down"):
            assert np.all(lib[n] == 8.0)


def test_more_argument_checks_before_touching_the_gpu():
    # Every case below fails in the host-side checks; fake non-NULL pointers
    # (aligned addresses) are never dereferenced.
    import ctypes
    lib = moe._lib
    s = moe.moe_expert_shape(256, 128, 64)
    P = ctypes.c_void_p
    A = P(1 << 20)  # an aligned fake address
    fwd = lambda T, k, E, pool, ws, ws_bytes, path=1, x=A, ids=A: lib.moe_expert_forward(  # noqa: E731
        ctypes.byref(s), x, T, ids, A, k, E, pool, A, 8, None, A, ws, ws_bytes, path, None)
    assert fwd(1, 33, 64, A, A, 1 << 20) == moe.MOE_ERR_ARG          # k > 32
    assert fwd(1, 2, 0, A, A, 1 << 20) == moe.MOE_ERR_ARG            # E = 0
    assert fwd(1, 2, 8, None, A, 1 << 20) == moe.MOE_ERR_ARG         # NULL pool
    assert fwd(1, 2, 8, P((1 << 20) + 16), A, 1 << 20) == moe.MOE_ERR_ARG  # pool not 256-aligned
    assert fwd(1, 2, 8, A, P((1 << 20) + 8), 1 << 20) == moe.MOE_ERR_ARG   # workspace not 256-aligned
    assert fwd(1, 2, 8, A, A, 1 << 20, x=P((1 << 20) + 2)) == moe.MOE_ERR_ARG  # x not 16-aligned
    assert fwd(1, 2, 8, A, A, 16) == moe.MOE_ERR_CAPACITY            # workspace too small
    assert fwd(-1, 2, 8, A, A, 1 << 20) == moe.MOE_ERR_ARG           # T < 0
    # Zero-copy: the host source must be given, page-locked and mapped.
    zc = lambda host: lib.moe_expert_forward_zero_copy(  # noqa: E731
        ctypes.byref(s), A, 1, A, A, 2, 8, A, A, 8, host, None, A, A, 1 << 20, None)
    assert zc(None) == moe.MOE_ERR_ARG
    buf = (ctypes.c_uint8 * 4096)()
    assert zc(ctypes.cast(buf, P)) == moe.MOE_ERR_ARG                # pageable memory
    # Layer call: k > E, bad path.
    assert lib.moe_layer_forward(ctypes.byref(s), A, A, 1, 4, 8, 0, A, A, A, A, 4, None, A, A,
                                 1 << 20, 1, None) == moe.MOE_ERR_ARG
    assert lib.moe_layer_forward(ctypes.byref(s), A, A, 1, 8, 2, 0, A, A, A, A, 8, None, A, A,
                                 1 << 20, 9, None) == moe.MOE_ERR_ARG
    # Shared FFN: sizes must be positive multiples of 64; T = 0 is a no-op.
    assert lib.moe_shared_forward(A, 4, 100, 128, A, A, A, A, A, 1 << 20, None) == moe.MOE_ERR_ARG
    assert lib.moe_shared_forward(A, 4, 256, 0, A, A, A, A, A, 1 << 20, None) == moe.MOE_ERR_ARG
    assert lib.moe_shared_forward(None, 0, 256, 128, None, None, None, None, None, 0, None) == moe.MOE_OK
    assert lib.moe_shared_forward(None, 4, 256, 128, A, A, A, A, A, 1 << 20, None) == moe.MOE_ERR_ARG
    # Residency calls on a NULL handle.
    n = ctypes.c_size_t(0)
    assert lib.moe_residency_prepare(None, 0, None, 0) == moe.MOE_ERR_ARG
    assert lib.moe_residency_prefetch(None, 0, None, 0, None) == moe.MOE_ERR_ARG
    assert lib.moe_residency_ops(None, None, 0, ctypes.byref(n)) == moe.MOE_ERR_ARG
    assert lib.moe_residency_trace(None, None, 0, ctypes.byref(n)) == moe.MOE_ERR_ARG
