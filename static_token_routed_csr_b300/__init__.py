"""Python binding of the L³ C ABI (``include/l3.h``): argument marshalling only.

Every computation runs in the CUDA library ``libl3.so`` built in this directory (see
``build.py``). The functions carry the C names; they take torch tensors (device memory)
or numpy arrays (host memory), pass raw pointers, and raise ``L3Error`` on a non-OK
status. The library is loaded on first use; if it has not been built, that first use
raises ImportError. There is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

__all__ = [
    "L3Error", "L3Layer", "lib", "make_layer", "L3_F32", "L3_BF16",
    "L3_PASS_FORWARD", "L3_PASS_BACKWARD", "L3_PASS_FORWARD_HOST", "L3_PASS_BACKWARD_ROWS",
    "L3_FWD_STAGES", "l3_backward_rows", "l3_stage_rows", "L3_PASS_STAGE",
    "STAGE_NAMES", "l3_alloc_offsets", "l3_workspace_size", "l3_saved_size",
    "l3_check_layer", "l3_route", "l3_route_noalloc", "l3_forward", "l3_forward_timed", "l3_forward_host",
    "l3_backward", "l3_get_error", "l3_status_string", "l3_launch_count", "l3_abi_version",
    "l3_selftest_wait_timeout", "l3_count_ids", "l3_alloc_offsets_counts",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libl3.so")

L3_F32, L3_BF16 = 0, 1
L3_PASS_FORWARD, L3_PASS_BACKWARD, L3_PASS_FORWARD_HOST, L3_PASS_BACKWARD_ROWS = 0, 1, 2, 3
L3_PASS_STAGE = 4
L3_FWD_STAGES = 5
STAGE_NAMES = ("route", "attend", "attend_long", "up", "mix")
STATUS = {0: "L3_OK", 1: "L3_ERR_INVALID_ARG", 2: "L3_ERR_INFEASIBLE", 3: "L3_ERR_UNSUPPORTED",
          4: "L3_ERR_WORKSPACE", 5: "L3_ERR_TOKEN_RANGE", 6: "L3_ERR_CUDA", 7: "L3_ERR_LAYER",
          8: "L3_ERR_TIMEOUT"}


class L3Error(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(self.status, self.status)}")


class L3Layer(ctypes.Structure):
    _fields_ = [("vocab", ctypes.c_int64), ("v", ctypes.c_int64), ("d", ctypes.c_int64),
                ("d_v", ctypes.c_int64), ("k_max", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("ln_eps", ctypes.c_float), ("reserved", ctypes.c_int32),
                ("offs", ctypes.c_void_p), ("K", ctypes.c_void_p), ("V", ctypes.c_void_p),
                ("W_up", ctypes.c_void_p), ("W_mix", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
_LP = ctypes.POINTER(L3Layer)

_SIGNATURES = {
    "l3_alloc_offsets": (_I32, [_P, _I64, _I64, _I32, _I32, ctypes.c_double, _P]),
    "l3_workspace_size": (_SZ, [_LP, _I64, _I32]),
    "l3_saved_size": (_SZ, [_LP, _I64]),
    "l3_check_layer": (_I32, [_LP, _P, _SZ, _P]),
    "l3_route": (_I32, [_LP, _P, _I64, _P, _P, _P, _P, _P, _SZ, _P]),
    "l3_route_noalloc": (_I32, [_LP, _P, _I64, _P, _P, _P, _P, _P]),
    "l3_forward": (_I32, [_LP, _P, _I64, _P, _P, _I32, _P, _P, _SZ, _P]),
    "l3_forward_timed": (_I32, [_LP, _P, _I64, _P, _P, _I32, _P, _P, _SZ, _P, _P]),
    "l3_forward_host": (_I32, [_LP, _P, _I64, _P, _P, _I32, _P, _SZ, _P]),
    "l3_backward": (_I32, [_LP, _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "l3_backward_rows": (_I32, [_LP, _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _P, _P,
                                _SZ, _P]),
    "l3_stage_rows": (_I32, [_LP, _P, _I64, _P, _P, _I64, _P, _P, _P, _LP, _P, _SZ, _P]),
    "l3_get_error": (_I32, [_P, _P]),
    "l3_status_string": (ctypes.c_char_p, [_I32]),
    "l3_launch_count": (ctypes.c_uint64, []),
    "l3_abi_version": (_I32, []),
    "l3_selftest_wait_timeout": (_I32, [_P, _SZ, _I64, _P]),
    "l3_count_ids": (_I32, [_P, _I64, _I64, _P, _P, _SZ, _P]),
    "l3_alloc_offsets_counts": (_I32, [_P, _I64, _I64, _I32, _I32, ctypes.c_double,
                                       ctypes.c_double, _P]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if ``libl3.so`` has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m static_token_routed_csr_b300.build`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(h, name)
            f.restype, f.argtypes = res, args
        _lib = h
    return _lib


def _check(st: int, where: str):
    if st != 0:
        raise L3Error(st, where)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.float32:
        return L3_F32
    if t.dtype == torch.bfloat16:
        return L3_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def make_layer(offs, K, V, W_up, W_mix, k_max: int, ln_eps: float = 1e-5) -> L3Layer:
    """An ``l3_layer`` over device tensors (kept alive by the returned struct)."""
    v, d = K.shape
    dt = _dtype_code(K)
    for t in (V, W_up, W_mix):
        if _dtype_code(t) != dt or not t.is_contiguous():
            raise TypeError("K, V, W_up, W_mix must share the dtype and be contiguous")
    if not (K.is_contiguous() and offs.is_contiguous()):
        raise TypeError("tensors must be contiguous")
    L = L3Layer(vocab=offs.numel() - 1, v=v, d=d, d_v=V.shape[1], k_max=k_max, dtype=dt,
                ln_eps=ln_eps, reserved=0, offs=_ptr(offs), K=_ptr(K), V=_ptr(V),
                W_up=_ptr(W_up), W_mix=_ptr(W_mix))
    L._keep = (offs, K, V, W_up, W_mix)
    return L


def l3_alloc_offsets(freq, v: int, n_min: int, n_max: int, power: float) -> np.ndarray:
    """Host-only row allocation; returns offs [vocab+1] int32."""
    f = np.ascontiguousarray(freq, dtype=np.float64)
    out = np.zeros(f.shape[0] + 1, dtype=np.int32)
    _check(lib().l3_alloc_offsets(_ptr(f), f.shape[0], int(v), int(n_min), int(n_max),
                                  float(power), _ptr(out)), "l3_alloc_offsets")
    return out


def l3_count_ids(ids, vocab: int, counts, ws, stream=None) -> None:
    """counts [vocab] int64 (device) = occurrences of each id in ``ids`` (device int32)."""
    _check(lib().l3_count_ids(_ptr(ids), ids.numel(), int(vocab), _ptr(counts), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "l3_count_ids")


def l3_alloc_offsets_counts(counts, v: int, n_min: int, n_max: int, power: float,
                            smoothing: float) -> np.ndarray:
    """Host-only allocation from token counts (freq = counts + smoothing); offs [vocab+1]."""
    c = np.ascontiguousarray(counts, dtype=np.int64)
    out = np.zeros(c.shape[0] + 1, dtype=np.int32)
    _check(lib().l3_alloc_offsets_counts(_ptr(c), c.shape[0], int(v), int(n_min), int(n_max),
                                         float(power), float(smoothing), _ptr(out)),
           "l3_alloc_offsets_counts")
    return out


def l3_workspace_size(layer: L3Layer, T: int, pass_: int = L3_PASS_FORWARD) -> int:
    return int(lib().l3_workspace_size(ctypes.byref(layer), int(T), int(pass_)))


def l3_saved_size(layer: L3Layer, T: int) -> int:
    return int(lib().l3_saved_size(ctypes.byref(layer), int(T)))


def l3_check_layer(layer: L3Layer, ws, stream=None) -> None:
    _check(lib().l3_check_layer(ctypes.byref(layer), _ptr(ws), ws.numel() * ws.element_size(),
                                _stream(stream)), "l3_check_layer")


def l3_route(layer: L3Layer, ids, ws, perm=None, seg_start=None, seg_id=None, n_seg=None,
             stream=None) -> None:
    T = ids.numel()
    _check(lib().l3_route(ctypes.byref(layer), _ptr(ids), T, _ptr(perm), _ptr(seg_start),
                          _ptr(seg_id), _ptr(n_seg), _ptr(ws), ws.numel() * ws.element_size(),
                          _stream(stream)), "l3_route")


def l3_route_noalloc(layer: L3Layer, ids, n_seg, perm=None, seg_start=None, seg_id=None,
                     stream=None) -> None:
    """l3_route without a workspace (the library's own fixed scratch; see include/l3.h)."""
    _check(lib().l3_route_noalloc(ctypes.byref(layer), _ptr(ids), ids.numel(), _ptr(perm),
                                  _ptr(seg_start), _ptr(seg_id), _ptr(n_seg), _stream(stream)),
           "l3_route_noalloc")


def l3_forward(layer: L3Layer, ids, x, y, ws, saved=None, stream=None) -> None:
    _check(lib().l3_forward(ctypes.byref(layer), _ptr(ids), ids.numel(), _ptr(x), _ptr(y),
                            _dtype_code(y), _ptr(saved), _ptr(ws),
                            ws.numel() * ws.element_size(), _stream(stream)), "l3_forward")


def l3_forward_timed(layer: L3Layer, ids, x, y, ws, events: Sequence, saved=None,
                     stream=None) -> None:
    """``events``: L3_FWD_STAGES+1 recorded-once ``torch.cuda.Event(enable_timing=True)``."""
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib().l3_forward_timed(ctypes.byref(layer), _ptr(ids), ids.numel(), _ptr(x), _ptr(y),
                                  _dtype_code(y), _ptr(saved), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream),
                                  ctypes.cast(arr, ctypes.c_void_p)), "l3_forward_timed")


def l3_forward_host(layer: L3Layer, ids_host, x_host, y_host, ws, stream=None) -> None:
    """Host (pinned) torch tensors in and out; the caller synchronises the stream."""
    _check(lib().l3_forward_host(ctypes.byref(layer), _ptr(ids_host), ids_host.numel(),
                                 _ptr(x_host), _ptr(y_host), _dtype_code(y_host), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream)),
           "l3_forward_host")


def l3_backward(layer: L3Layer, ids, x, dy, saved, dx, dK, dV, dW_up, dW_mix, ws,
                stream=None) -> None:
    _check(lib().l3_backward(ctypes.byref(layer), _ptr(ids), ids.numel(), _ptr(x), _ptr(dy),
                             _ptr(saved), _ptr(dx), _ptr(dK), _ptr(dV), _ptr(dW_up),
                             _ptr(dW_mix), _ptr(ws), ws.numel() * ws.element_size(),
                             _stream(stream)), "l3_backward")


def l3_backward_rows(layer: L3Layer, ids, x, dy, saved, dx, row_index, dK_rows, dV_rows, n_rows,
                     dW_up, dW_mix, ws, stream=None) -> None:
    """Row-gradient backward (bf16 layers); the row outputs' capacity is row_index.numel()."""
    _check(lib().l3_backward_rows(ctypes.byref(layer), _ptr(ids), ids.numel(), _ptr(x), _ptr(dy),
                                  _ptr(saved), _ptr(dx), _ptr(row_index), _ptr(dK_rows),
                                  _ptr(dV_rows), _ptr(n_rows), row_index.numel(), _ptr(dW_up),
                                  _ptr(dW_mix), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)), "l3_backward_rows")


def l3_stage_rows(layer: L3Layer, ids, K_stage, V_stage, offs_stage, ids_stage, n_rows, ws,
                  stream=None) -> L3Layer:
    """Stage the batch's rows of host-resident tables into K_stage / V_stage (device); returns
    the staged layer (its capacity is K_stage.shape[0])."""
    staged = L3Layer()
    _check(lib().l3_stage_rows(ctypes.byref(layer), _ptr(ids), ids.numel(), _ptr(K_stage),
                               _ptr(V_stage), K_stage.shape[0], _ptr(offs_stage), _ptr(ids_stage),
                               _ptr(n_rows), ctypes.byref(staged), _ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream)), "l3_stage_rows")
    staged._keep = (getattr(layer, "_keep", None), K_stage, V_stage, offs_stage)
    return staged


def l3_get_error(ws, stream=None) -> int:
    """Status of the device-side checks of the last call on ``ws`` (0 = OK)."""
    return int(lib().l3_get_error(_ptr(ws), _stream(stream)))


def l3_status_string(status: int) -> str:
    return lib().l3_status_string(int(status)).decode()


def l3_launch_count() -> int:
    return int(lib().l3_launch_count())


def l3_selftest_wait_timeout(ws, limit_ns: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test on ``ws`` (read the result with l3_get_error)."""
    _check(lib().l3_selftest_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(),
                                          int(limit_ns), _stream(stream)),
           "l3_selftest_wait_timeout")


def l3_abi_version() -> int:
    return int(lib().l3_abi_version())
