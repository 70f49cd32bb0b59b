"""Python binding of libk3moe.so: the GB300 (sm_103a) MXFP4 MoE layer.

Argument marshalling only: every step of the layer runs in the library's CUDA kernels. The
functions take torch tensors (device memory and streams come from PyTorch) and pass raw
pointers through the C ABI declared in include/k3moe.h. If the library is not built, or the
call fails, an exception is raised; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB, build

__all__ = ["Config", "K3moeError", "load", "record_bytes", "workspace_bytes", "router_parts_bytes", "prepare_router",
           "route", "expert_ffn", "layer", "layer_bounded", "layer_timed", "layer_static", "pack_records",
           "rmsnorm", "residual_add", "residual_rmsnorm", "check_device_status", "status_string", "X_BF16", "X_F32"]

OK, ERR_INVALID_ARGUMENT, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_CHECK, ERR_TIMEOUT = range(7)
SCORE_SOFTMAX, SCORE_SIGMOID_BIAS = 0, 1
ACT_EXACT, ACT_MXFP4, ACT_BF16H = 0, 1, 2
X_BF16, X_F32 = 0, 1
ORDER_STORED, ORDER_DEVICE = 0, 1
SHARED_MXFP4, SHARED_BF16 = 0, 1

EXPORTS = ["k3moe_record_bytes", "k3moe_workspace_bytes", "k3moe_router_parts_bytes", "k3moe_prepare_router",
           "k3moe_route", "k3moe_expert_ffn", "k3moe_layer", "k3moe_layer_bounded", "k3moe_layer_timed",
           "k3moe_layer_static", "k3moe_pack_records", "k3moe_rmsnorm", "k3moe_residual_add",
           "k3moe_residual_rmsnorm", "k3moe_check_device_status", "k3moe_status_string"]


class Config(ctypes.Structure):
    """Mirror of k3moe_config."""
    _fields_ = [("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("n_routed", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("n_shared", ctypes.c_int32), ("score_func", ctypes.c_int32),
                ("act_mode", ctypes.c_int32), ("x_dtype", ctypes.c_int32), ("record_order", ctypes.c_int32),
                ("shared_format", ctypes.c_int32), ("record_stride", ctypes.c_int64),
                ("shared_stride", ctypes.c_int64)]

    @classmethod
    def make(cls, d_model, d_ff, n_routed, top_k, n_shared, x_dtype=X_BF16, record_stride=None,
             score_func=SCORE_SOFTMAX, act_mode=ACT_EXACT, record_order=ORDER_DEVICE, shared_format=SHARED_MXFP4,
             shared_stride=0):
        """A config. record_order defaults to ORDER_DEVICE: the records are put in the device order by
        pack_records once they are on the GPU (the C struct zero-initialised says ORDER_STORED)."""
        rec = 3 * (d_model * d_ff // 2 + d_model * d_ff // 32)
        stride = record_stride if record_stride is not None else (rec + 4095) // 4096 * 4096
        return cls(d_model, d_ff, n_routed, top_k, n_shared, score_func, act_mode, x_dtype, record_order,
                   shared_format, stride, shared_stride)


class K3moeError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def load(path: str | None = None):
    """Load libk3moe.so (building it first if the sources are newer)."""
    global _lib
    if _lib is None:
        so = path or LIB
        if path is None and not os.path.exists(so):
            build()
        L = ctypes.CDLL(so)
        cfgp = ctypes.POINTER(Config)
        L.k3moe_record_bytes.argtypes = [cfgp]
        L.k3moe_record_bytes.restype = ctypes.c_size_t
        L.k3moe_workspace_bytes.argtypes = [cfgp, _I64]
        L.k3moe_workspace_bytes.restype = ctypes.c_size_t
        L.k3moe_router_parts_bytes.argtypes = [cfgp]
        L.k3moe_router_parts_bytes.restype = ctypes.c_size_t
        L.k3moe_prepare_router.argtypes = [cfgp, _P, _P, _P]
        L.k3moe_route.argtypes = [cfgp, _P, _I64, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
        L.k3moe_expert_ffn.argtypes = [cfgp, _P, _I64, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
        L.k3moe_layer.argtypes = [cfgp, _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
        L.k3moe_layer_bounded.argtypes = [cfgp, _P, _I64, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                          ctypes.c_uint32, _P]
        L.k3moe_layer_timed.argtypes = [cfgp, _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]
        L.k3moe_layer_static.argtypes = [cfgp, _P, _I64, _P, _P, _P, _P, _P, _P]
        L.k3moe_layer_static.restype = ctypes.c_int
        L.k3moe_pack_records.argtypes = [cfgp, _P, _I64, ctypes.c_int32, _P]
        L.k3moe_rmsnorm.argtypes = [_P, _I64, ctypes.c_int32, ctypes.c_float, _P, _P]
        L.k3moe_residual_add.argtypes = [_P, _P, _I64, _P]
        L.k3moe_residual_rmsnorm.argtypes = [_P, _P, _I64, ctypes.c_int32, ctypes.c_float, _P, _P]
        L.k3moe_check_device_status.argtypes = [_P, _P]
        L.k3moe_status_string.argtypes = [ctypes.c_int]
        L.k3moe_status_string.restype = ctypes.c_char_p
        for name in ["k3moe_prepare_router", "k3moe_route", "k3moe_expert_ffn", "k3moe_layer", "k3moe_layer_bounded",
                     "k3moe_layer_timed", "k3moe_pack_records", "k3moe_rmsnorm", "k3moe_residual_add",
                     "k3moe_residual_rmsnorm", "k3moe_check_device_status"]:
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return load().k3moe_status_string(code).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(code, what):
    if code != OK:
        raise K3moeError(code, what)


def record_bytes(cfg: Config) -> int:
    return load().k3moe_record_bytes(ctypes.byref(cfg))


def workspace_bytes(cfg: Config, max_tokens: int) -> int:
    n = load().k3moe_workspace_bytes(ctypes.byref(cfg), max_tokens)
    if n == 0:
        raise K3moeError(ERR_INVALID_ARGUMENT, "k3moe_workspace_bytes")
    return n


def router_parts_bytes(cfg: Config) -> int:
    n = load().k3moe_router_parts_bytes(ctypes.byref(cfg))
    if n == 0:
        raise K3moeError(ERR_INVALID_ARGUMENT, "k3moe_router_parts_bytes")
    return n


def prepare_router(cfg, w_router, w_parts, stream=None):
    """k3moe_prepare_router: the three bf16 parts of the router weights (weight loading, once)."""
    _check(load().k3moe_prepare_router(ctypes.byref(cfg), _ptr(w_router), _ptr(w_parts), _stream(stream)),
           "k3moe_prepare_router")


def route(cfg, x, T, w_router, bias, topk_idx, topk_w, ws, stream=None, w_parts=None):
    _check(load().k3moe_route(ctypes.byref(cfg), _ptr(x), T, _ptr(w_router), _ptr(w_parts), _ptr(bias),
                              _ptr(topk_idx), _ptr(topk_w), _ptr(ws), ws.numel() * ws.element_size(),
                              _stream(stream)), "k3moe_route")


def expert_ffn(cfg, x, T, topk_idx, topk_w, routed, shared, y, ws, stream=None):
    _check(load().k3moe_expert_ffn(ctypes.byref(cfg), _ptr(x), T, _ptr(topk_idx), _ptr(topk_w), _ptr(routed),
                                   _ptr(shared), _ptr(y), _ptr(ws), ws.numel() * ws.element_size(),
                                   _stream(stream)), "k3moe_expert_ffn")


def layer(cfg, x, T, w_router, bias, routed, shared, y, ws, topk_idx=None, topk_w=None, stream=None, w_parts=None):
    _check(load().k3moe_layer(ctypes.byref(cfg), _ptr(x), T, _ptr(w_router), _ptr(w_parts), _ptr(bias),
                              _ptr(routed), _ptr(shared), _ptr(y), _ptr(topk_idx), _ptr(topk_w), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "k3moe_layer")


def layer_bounded(cfg, x, T, w_router, bias, routed, shared, y, ws, wait_limit, stream=None, w_parts=None):
    """k3moe_layer_bounded: the layer with an explicit bound on the kernels' barrier waits; returns the
    call's status code (the timeout itself is reported later by check_device_status)."""
    return load().k3moe_layer_bounded(ctypes.byref(cfg), _ptr(x), T, _ptr(w_router), _ptr(w_parts), _ptr(bias),
                                      _ptr(routed), _ptr(shared), _ptr(y), _ptr(ws), ws.numel() * ws.element_size(),
                                      wait_limit, _stream(stream))


def layer_timed(cfg, x, T, w_router, bias, routed, shared, y, ws, events, topk_idx=None, topk_w=None, stream=None,
                w_parts=None):
    """k3moe_layer recording 6 caller-created cudaEvent_t handles (ints) around its kernels."""
    if len(events) != 6:
        raise ValueError("layer_timed needs 6 events")
    ev = (ctypes.c_void_p * 6)(*events)
    _check(load().k3moe_layer_timed(ctypes.byref(cfg), _ptr(x), T, _ptr(w_router), _ptr(w_parts), _ptr(bias),
                                    _ptr(routed), _ptr(shared), _ptr(y), _ptr(topk_idx), _ptr(topk_w), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream), ev), "k3moe_layer_timed")


def layer_static(cfg, x, T, w_router, bias, routed, shared, y, stream=None):
    """k3moe_layer_static: the layer without a workspace argument, for callers that cannot allocate
    device memory; its scratch is a fixed 4 MiB array inside the library (see include/k3moe.h)."""
    _check(load().k3moe_layer_static(ctypes.byref(cfg), _ptr(x), T, _ptr(w_router), _ptr(bias), _ptr(routed),
                                     _ptr(shared), _ptr(y), _stream(stream)), "k3moe_layer_static")


def pack_records(cfg, records, n_records, to_device=True, stream=None):
    """k3moe_pack_records: put n records (in place) into the device order that the compute calls
    read (to_device=True), or back into the stored order."""
    _check(load().k3moe_pack_records(ctypes.byref(cfg), _ptr(records), n_records, 1 if to_device else 0,
                                     _stream(stream)), "k3moe_pack_records")


def rmsnorm(x, T, d, eps, xn, stream=None):
    _check(load().k3moe_rmsnorm(_ptr(x), T, d, eps, _ptr(xn), _stream(stream)), "k3moe_rmsnorm")


def residual_add(x, y, n, stream=None):
    _check(load().k3moe_residual_add(_ptr(x), _ptr(y), n, _stream(stream)), "k3moe_residual_add")


def residual_rmsnorm(x, y, T, d, eps, xn, stream=None):
    """k3moe_residual_rmsnorm: x += y (y may be None), then xn = RMSNorm(x), in one kernel."""
    _check(load().k3moe_residual_rmsnorm(_ptr(x), _ptr(y), T, d, eps, _ptr(xn), _stream(stream)),
           "k3moe_residual_rmsnorm")


def check_device_status(ws, stream=None) -> int:
    """Returns the status code (OK, ERR_DEVICE_CHECK or ERR_TIMEOUT); raises on CUDA errors."""
    code = load().k3moe_check_device_status(_ptr(ws), _stream(stream))
    if code not in (OK, ERR_DEVICE_CHECK, ERR_TIMEOUT):
        raise K3moeError(code, "k3moe_check_device_status")
    return code
