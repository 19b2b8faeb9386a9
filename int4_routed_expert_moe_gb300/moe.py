"""Python binding of libmoe.so: the C ABI in include/moe.h, same names.

Argument marshalling only -- every step of the path runs in the library's
CUDA kernels. Device buffers are torch tensors (torch supplies memory and
streams); each wrapper checks dtype/device/contiguity/size, passes raw
pointers, and raises MoeError on a non-zero status. Importing this module
raises ImportError when the library has not been built: there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

MOE_OK = 0
MOE_ERR_ARG = -1
MOE_ERR_SHAPE = -2
MOE_ERR_CAPACITY = -3
MOE_ERR_CUDA = -4
MOE_ERR_NONFINITE = -5
MOE_ERR_STATE = -6
MOE_ERR_TIMEOUT = -7
MOE_ERR_INJECTED = -8
MOE_ERR_UNSUPPORTED = -9

MOE_PATH_AUTO, MOE_PATH_GEMV, MOE_PATH_GROUPED, MOE_PATH_GEMV_UNFUSED = 0, 1, 2, 3


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {moe_status_string(status)}: {detail}")


class moe_expert_shape(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("group", ctypes.c_int32)]


class moe_block_layout(ctypes.Structure):
    _fields_ = [("total", ctypes.c_uint64), ("d_offset", ctypes.c_uint64),
                ("gu_row_bytes", ctypes.c_uint32), ("d_row_bytes", ctypes.c_uint32)] + [
        (n, ctypes.c_uint32) for n in ("gu_q_gate", "gu_q_up", "gu_sz", "d_q", "d_sz")]


MOE_POLICY_DECAY, MOE_POLICY_LRU, MOE_POLICY_PINNED = 0, 1, 2


class moe_residency_cfg(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int32), ("experts", ctypes.c_int32),
                ("slots", ctypes.c_int32), ("spares", ctypes.c_int32),
                ("max_ids_per_step", ctypes.c_int32), ("dry_run", ctypes.c_int32),
                ("block_bytes", ctypes.c_uint64), ("decay", ctypes.c_double),
                ("policy", ctypes.c_int32), ("pinned", ctypes.c_int32),
                ("profile", ctypes.c_void_p), ("log_ops", ctypes.c_int32)]


class moe_residency_op(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("kind", "stream", "event", "layer", "slot", "expert")]


MOE_OP_RECORD, MOE_OP_WAIT, MOE_OP_COPY, MOE_OP_PUBLISH = 0, 1, 2, 3


class moe_residency_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in
                ("steps", "hits", "misses", "evictions", "copies", "h2d_bytes", "prefetched",
                 "prefetch_copies")]


class moe_residency_event(ctypes.Structure):
    _fields_ = [("step", ctypes.c_int64), ("layer", ctypes.c_int32),
                ("expert", ctypes.c_int32), ("slot", ctypes.c_int32),
                ("victim", ctypes.c_int32)]


if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is not built; run int4_routed_expert_moe_gb300.build.build()")
_lib = ctypes.CDLL(_LIB_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_SHAPE = ctypes.POINTER(moe_expert_shape)

_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_version": (_I, []),
    "moe_expert_block_bytes": (_SZ, [_SHAPE]),
    "moe_expert_block_layout": (_I, [_SHAPE, ctypes.POINTER(moe_block_layout)]),
    "moe_pack_expert": (_I, [_SHAPE] + [_P] * 10),
    "moe_unpack_expert": (_I, [_SHAPE] + [_P] * 10),
    "moe_route": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P]),
    "moe_token_sort": (_I, [_P, _I, _I, _I, _P, _P, _P, _P]),
    "moe_forward_workspace_bytes": (_SZ, [_SHAPE, _I, _I, _I, _I]),
    "moe_expert_forward": (_I, [_SHAPE, _P, _I, _P, _P, _I, _I, _P, _P, _I, _P, _P, _P, _SZ, _I, _P]),
    "moe_expert_forward_zero_copy": (_I, [_SHAPE, _P, _I, _P, _P, _I, _I, _P, _P, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_layer_forward": (_I, [_SHAPE, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _P, _P, _SZ, _I, _P]),
    "moe_layer_forward_noalloc": (_I, [_SHAPE, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _P, _P]),
    "moe_layer_forward_noalloc_flags": (_I, [ctypes.POINTER(ctypes.c_int32), _P]),
    "moe_workspace_clear_flags": (_I, [_P, _P]),
    "moe_workspace_flags": (_I, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
    "moe_shared_workspace_bytes": (_SZ, [_I, _I, _I]),
    "moe_shared_forward": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_residency_create": (_I, [ctypes.POINTER(moe_residency_cfg), _P, _P, _P, _P, _P,
                                  ctypes.POINTER(_P)]),
    "moe_residency_prepare": (_I, [_P, _I, _P, _I]),
    "moe_residency_prefetch": (_I, [_P, _I, _P, _I, ctypes.POINTER(ctypes.c_int)]),
    "moe_residency_get_stats": (_I, [_P, _I, ctypes.POINTER(moe_residency_stats)]),
    "moe_residency_trace": (_I, [_P, _P, _SZ, ctypes.POINTER(_SZ)]),
    "moe_residency_ops": (_I, [_P, _P, _SZ, ctypes.POINTER(_SZ)]),
    "moe_residency_slot_table": (_I, [_P, _I, _P]),
    "moe_residency_counts": (_I, [_P, _I, _P]),
    "moe_residency_inject_copy_failure": (_I, [_P, ctypes.c_int64]),
    "moe_residency_destroy": (None, [_P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


def lib_path() -> str:
    return _LIB_PATH


def moe_status_string(status: int) -> str:
    return _lib.moe_status_string(status).decode()


def moe_last_error() -> str:
    return _lib.moe_last_error().decode()


def moe_version() -> int:
    return _lib.moe_version()


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where, moe_last_error())


def _shape(shape) -> moe_expert_shape:
    H, I, g = shape
    return moe_expert_shape(int(H), int(I), int(g))


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor | None, dtype, name: str, numel: int | None = None, nullable=False):
    if t is None:
        if nullable:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")
    return t.data_ptr()


# ---- expert block layout (host) --------------------------------------------
def moe_expert_block_bytes(shape) -> int:
    s = _shape(shape)
    return _lib.moe_expert_block_bytes(ctypes.byref(s))


def moe_expert_block_layout(shape) -> dict:
    s = _shape(shape)
    out = moe_block_layout()
    _check(_lib.moe_expert_block_layout(ctypes.byref(s), ctypes.byref(out)), "moe_expert_block_layout")
    return {n: int(getattr(out, n)) for n, _ in moe_block_layout._fields_}


_ARRAY_ORDER = ("qp_gate", "qp_up", "qp_down", "s_gate", "z_gate", "s_up", "z_up",
                "s_down", "z_down")


def _np_ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def moe_pack_expert(shape, arrays: dict, out: np.ndarray | None = None) -> np.ndarray:
    """Copies the canonical arrays of one expert into one block (host)."""
    H, I, g = shape
    nbytes = moe_expert_block_bytes(shape)
    if nbytes == 0:
        raise MoeError(MOE_ERR_SHAPE, "moe_pack_expert", f"invalid shape {shape}")
    want = {"qp_gate": ((I, H // 2), np.uint8), "qp_up": ((I, H // 2), np.uint8),
            "qp_down": ((H, I // 2), np.uint8)}
    for n in ("gate", "up"):
        want[f"s_{n}"] = want[f"z_{n}"] = ((I, H // g), np.float16)
    want["s_down"] = want["z_down"] = ((H, I // g), np.float16)
    arrs = []
    for n in _ARRAY_ORDER:
        a = np.ascontiguousarray(arrays[n])
        shp, dt = want[n]
        if a.shape != shp or a.dtype != dt:
            raise ValueError(f"{n}: expected {shp} {dt}, got {a.shape} {a.dtype}")
        arrs.append(a)
    if out is None:
        out = np.empty(nbytes, dtype=np.uint8)
    assert out.nbytes >= nbytes and out.flags.c_contiguous
    s = _shape(shape)
    _check(_lib.moe_pack_expert(ctypes.byref(s), *[_np_ptr(a) for a in arrs], _np_ptr(out)),
           "moe_pack_expert")
    return out


def moe_unpack_expert(shape, block: np.ndarray) -> dict:
    H, I, g = shape
    out = {"qp_gate": np.empty((I, H // 2), np.uint8), "qp_up": np.empty((I, H // 2), np.uint8),
           "qp_down": np.empty((H, I // 2), np.uint8)}
    for n in ("gate", "up"):
        out[f"s_{n}"] = np.empty((I, H // g), np.float16)
        out[f"z_{n}"] = np.empty((I, H // g), np.float16)
    out["s_down"] = np.empty((H, I // g), np.float16)
    out["z_down"] = np.empty((H, I // g), np.float16)
    block = np.ascontiguousarray(block, dtype=np.uint8)
    s = _shape(shape)
    _check(_lib.moe_unpack_expert(ctypes.byref(s), _np_ptr(block),
                                  *[_np_ptr(out[n]) for n in _ARRAY_ORDER]), "moe_unpack_expert")
    return out


# ---- GPU calls -------------------------------------------------------------
def moe_route(logits: torch.Tensor, k: int, renorm: bool, ids: torch.Tensor,
              weights: torch.Tensor, bad_tokens: torch.Tensor | None = None, stream=None) -> None:
    T, E = logits.shape
    _check(_lib.moe_route(_dev(logits, torch.float32, "logits"), T, E, k, int(bool(renorm)),
                          _dev(ids, torch.int32, "ids", T * k),
                          _dev(weights, torch.float32, "weights", T * k),
                          _dev(bad_tokens, torch.int32, "bad_tokens", 1, nullable=True),
                          _stream(stream)), "moe_route")


def moe_token_sort(ids: torch.Tensor, E: int, offsets: torch.Tensor, pair_tok: torch.Tensor,
                   pair_j: torch.Tensor, stream=None) -> None:
    T, k = ids.shape
    _check(_lib.moe_token_sort(_dev(ids, torch.int32, "ids"), T, k, E,
                               _dev(offsets, torch.int32, "offsets", E + 1),
                               _dev(pair_tok, torch.int32, "pair_tok", T * k),
                               _dev(pair_j, torch.int32, "pair_j", T * k),
                               _stream(stream)), "moe_token_sort")


def moe_forward_workspace_bytes(shape, T: int, k: int, E: int, path: int = MOE_PATH_AUTO) -> int:
    s = _shape(shape)
    return _lib.moe_forward_workspace_bytes(ctypes.byref(s), T, k, E, path)


def moe_expert_forward(shape, x: torch.Tensor, ids: torch.Tensor, weights: torch.Tensor, E: int,
                       pool: torch.Tensor, slot_of: torch.Tensor, n_slots: int,
                       y_shared: torch.Tensor | None, y: torch.Tensor, workspace: torch.Tensor,
                       path: int = MOE_PATH_AUTO, stream=None) -> None:
    H, I, g = shape
    T, k = ids.shape
    s = _shape(shape)
    bb = moe_expert_block_bytes(shape)
    _check(_lib.moe_expert_forward(
        ctypes.byref(s), _dev(x, torch.float16, "x", T * H), T,
        _dev(ids, torch.int32, "ids", T * k), _dev(weights, torch.float32, "weights", T * k), k, E,
        _dev(pool, torch.uint8, "pool", n_slots * bb), _dev(slot_of, torch.int32, "slot_of", E), n_slots,
        _dev(y_shared, torch.float16, "y_shared", T * H, nullable=True),
        _dev(y, torch.float16, "y", T * H), _dev(workspace, torch.uint8, "workspace"),
        workspace.numel(), path, _stream(stream)), "moe_expert_forward")


def moe_expert_forward_zero_copy(shape, x: torch.Tensor, ids: torch.Tensor, weights: torch.Tensor, E: int,
                                 pool: torch.Tensor, slot_of: torch.Tensor, n_slots: int,
                                 host_src: torch.Tensor, y_shared: torch.Tensor | None, y: torch.Tensor,
                                 workspace: torch.Tensor, stream=None) -> None:
    """moe_expert_forward on the two-kernel GEMV path; experts with slot -1
    are read in place from host_src (pinned CPU uint8 [E][block])."""
    H, I, g = shape
    T, k = ids.shape
    s = _shape(shape)
    bb = moe_expert_block_bytes(shape)
    if not isinstance(host_src, torch.Tensor) or host_src.is_cuda or host_src.dtype != torch.uint8:
        raise TypeError("host_src must be a CPU uint8 tensor")
    if not host_src.is_contiguous() or host_src.numel() < E * bb:
        raise ValueError(f"host_src must be contiguous with >= {E * bb} bytes")
    _check(_lib.moe_expert_forward_zero_copy(
        ctypes.byref(s), _dev(x, torch.float16, "x", T * H), T,
        _dev(ids, torch.int32, "ids", T * k), _dev(weights, torch.float32, "weights", T * k), k, E,
        _dev(pool, torch.uint8, "pool", n_slots * bb), _dev(slot_of, torch.int32, "slot_of", E), n_slots,
        host_src.data_ptr(), _dev(y_shared, torch.float16, "y_shared", T * H, nullable=True),
        _dev(y, torch.float16, "y", T * H), _dev(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream(stream)), "moe_expert_forward_zero_copy")


def moe_layer_forward(shape, x: torch.Tensor, logits: torch.Tensor, k: int, renorm: bool,
                      ids: torch.Tensor, weights: torch.Tensor, pool: torch.Tensor,
                      slot_of: torch.Tensor, n_slots: int, y_shared: torch.Tensor | None,
                      y: torch.Tensor, workspace: torch.Tensor, path: int = MOE_PATH_AUTO,
                      stream=None) -> None:
    H, I, g = shape
    T, E = logits.shape
    s = _shape(shape)
    bb = moe_expert_block_bytes(shape)
    _check(_lib.moe_layer_forward(
        ctypes.byref(s), _dev(x, torch.float16, "x", T * H), _dev(logits, torch.float32, "logits"), T, E,
        k, int(bool(renorm)), _dev(ids, torch.int32, "ids", T * k), _dev(weights, torch.float32, "weights", T * k),
        _dev(pool, torch.uint8, "pool", n_slots * bb), _dev(slot_of, torch.int32, "slot_of", E), n_slots,
        _dev(y_shared, torch.float16, "y_shared", T * H, nullable=True), _dev(y, torch.float16, "y", T * H),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), path, _stream(stream)), "moe_layer_forward")


def moe_layer_forward_noalloc(shape, x: torch.Tensor, logits: torch.Tensor, k: int, renorm: bool,
                              ids: torch.Tensor, weights: torch.Tensor, pool: torch.Tensor,
                              slot_of: torch.Tensor, n_slots: int, y_shared: torch.Tensor | None,
                              y: torch.Tensor, stream=None) -> None:
    """moe_layer_forward without a workspace (scratch is a fixed array inside the library)."""
    H, I, g = shape
    T, E = logits.shape
    s = _shape(shape)
    bb = moe_expert_block_bytes(shape)
    _check(_lib.moe_layer_forward_noalloc(
        ctypes.byref(s), _dev(x, torch.float16, "x", T * H), _dev(logits, torch.float32, "logits"), T, E,
        k, int(bool(renorm)), _dev(ids, torch.int32, "ids", T * k), _dev(weights, torch.float32, "weights", T * k),
        _dev(pool, torch.uint8, "pool", n_slots * bb), _dev(slot_of, torch.int32, "slot_of", E), n_slots,
        _dev(y_shared, torch.float16, "y_shared", T * H, nullable=True), _dev(y, torch.float16, "y", T * H),
        _stream(stream)), "moe_layer_forward_noalloc")


def moe_layer_forward_noalloc_flags(stream=None) -> int:
    """Error word of the last moe_layer_forward_noalloc call on the current device (synchronises)."""
    v = ctypes.c_int32(0)
    _check(_lib.moe_layer_forward_noalloc_flags(ctypes.byref(v), _stream(stream)), "moe_layer_forward_noalloc_flags")
    return v.value


def moe_workspace_clear_flags(workspace: torch.Tensor, stream=None) -> None:
    _check(_lib.moe_workspace_clear_flags(_dev(workspace, torch.uint8, "workspace"), _stream(stream)),
           "moe_workspace_clear_flags")


def moe_workspace_flags(workspace: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(_lib.moe_workspace_flags(_dev(workspace, torch.uint8, "workspace"), ctypes.byref(v),
                                    _stream(stream)), "moe_workspace_flags")
    return v.value


def moe_shared_workspace_bytes(T: int, H: int, Is: int) -> int:
    return _lib.moe_shared_workspace_bytes(T, H, Is)


def moe_shared_forward(x: torch.Tensor, wg: torch.Tensor, wu: torch.Tensor, wd: torch.Tensor,
                       y: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    T, H = x.shape
    Is = wg.shape[0]
    _check(_lib.moe_shared_forward(
        _dev(x, torch.float16, "x", T * H), T, H, Is, _dev(wg, torch.float16, "wg", Is * H),
        _dev(wu, torch.float16, "wu", Is * H), _dev(wd, torch.float16, "wd", H * Is),
        _dev(y, torch.float16, "y", T * H), _dev(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream(stream)), "moe_shared_forward")


# ---- residency manager -----------------------------------------------------
def moe_residency_create(cfg: dict, host_src: torch.Tensor | None, dev_pool: torch.Tensor | None,
                         dev_slot_of: torch.Tensor | None, compute=None, copy=None) -> int:
    policy = cfg.get("policy", MOE_POLICY_DECAY)
    if isinstance(policy, str):
        policy = {"decay": MOE_POLICY_DECAY, "lru": MOE_POLICY_LRU, "pinned": MOE_POLICY_PINNED}[policy]
    prof = cfg.get("profile")
    prof_arr = None
    if prof is not None:
        prof_arr = np.ascontiguousarray(np.asarray(prof, dtype=np.float64).reshape(-1))
        if prof_arr.size != int(cfg["layers"]) * int(cfg["experts"]):
            raise ValueError("profile must hold layers x experts values")
    c = moe_residency_cfg(int(cfg["layers"]), int(cfg["experts"]), int(cfg["slots"]),
                          int(cfg.get("spares", 0)), int(cfg["max_ids_per_step"]),
                          int(cfg.get("dry_run", 0)), int(cfg["block_bytes"]),
                          float(cfg["decay"]), int(policy), int(cfg.get("pinned", 0)),
                          prof_arr.ctypes.data if prof_arr is not None else None, int(cfg.get("log_ops", 0)))
    dry = bool(c.dry_run)
    src = pool = slot = None
    cs = cp = None
    if not dry:
        if host_src is None or not host_src.is_pinned():
            raise ValueError("host_src must be a pinned CPU tensor")
        src = host_src.data_ptr()
        pool = _dev(dev_pool, torch.uint8, "dev_pool")
        slot = _dev(dev_slot_of, torch.int32, "dev_slot_of", c.layers * c.experts)
        cs, cp = _stream(compute), _stream(copy)
    h = ctypes.c_void_p()
    _check(_lib.moe_residency_create(ctypes.byref(c), src, pool, slot, cs, cp, ctypes.byref(h)),
           "moe_residency_create")
    return h.value


def moe_residency_prepare(handle: int, layer: int, host_ids) -> None:
    a = np.ascontiguousarray(np.asarray(host_ids, dtype=np.int32).reshape(-1))
    _check(_lib.moe_residency_prepare(handle, layer, a.ctypes.data if a.size else None, a.size),
           "moe_residency_prepare")


def moe_residency_prefetch(handle: int, layer: int, host_ids) -> int:
    """Copy predicted misses into free spare slots; returns how many were copied."""
    a = np.ascontiguousarray(np.asarray(host_ids, dtype=np.int32).reshape(-1))
    n = ctypes.c_int(0)
    _check(_lib.moe_residency_prefetch(handle, layer, a.ctypes.data if a.size else None, a.size,
                                       ctypes.byref(n)), "moe_residency_prefetch")
    return int(n.value)


def moe_residency_get_stats(handle: int, layer: int = -1) -> dict:
    st = moe_residency_stats()
    _check(_lib.moe_residency_get_stats(handle, layer, ctypes.byref(st)), "moe_residency_get_stats")
    return {n: int(getattr(st, n)) for n, _ in moe_residency_stats._fields_}


def moe_residency_trace(handle: int) -> list:
    n = ctypes.c_size_t(0)
    _check(_lib.moe_residency_trace(handle, None, 0, ctypes.byref(n)), "moe_residency_trace")
    buf = (moe_residency_event * max(1, n.value))()
    _check(_lib.moe_residency_trace(handle, buf, n.value, ctypes.byref(n)), "moe_residency_trace")
    return [(int(b.step), int(b.layer), int(b.expert), int(b.slot), int(b.victim))
            for b in buf[:n.value]]


def moe_residency_ops(handle: int) -> list:
    """Logged stream operations: (kind, stream, event, layer, slot, expert) tuples."""
    n = ctypes.c_size_t(0)
    _check(_lib.moe_residency_ops(handle, None, 0, ctypes.byref(n)), "moe_residency_ops")
    buf = (moe_residency_op * max(1, n.value))()
    _check(_lib.moe_residency_ops(handle, buf, n.value, ctypes.byref(n)), "moe_residency_ops")
    return [(o.kind, o.stream, o.event, o.layer, o.slot, o.expert) for o in buf[:n.value]]


def moe_residency_slot_table(handle: int, layer: int, E: int) -> np.ndarray:
    out = np.empty(E, dtype=np.int32)
    _check(_lib.moe_residency_slot_table(handle, layer, out.ctypes.data), "moe_residency_slot_table")
    return out


def moe_residency_counts(handle: int, layer: int, E: int) -> np.ndarray:
    out = np.empty(E, dtype=np.float64)
    _check(_lib.moe_residency_counts(handle, layer, out.ctypes.data), "moe_residency_counts")
    return out


def moe_residency_inject_copy_failure(handle: int, nth_copy: int) -> None:
    _check(_lib.moe_residency_inject_copy_failure(handle, nth_copy), "moe_residency_inject_copy_failure")


def moe_residency_destroy(handle: int) -> None:
    _lib.moe_residency_destroy(handle)
