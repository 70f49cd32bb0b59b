"""CPU oracle for the Kimi-K3-style MXFP4 MoE layer -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg may
import this package. The CUDA library never calls it and shares no code with it.

The arithmetic lives in ``k3oracle.c`` (plain fp64 loops, see its header for the
passages each step follows); this module compiles it with gcc and wraps it with
numpy arrays. Parity of the oracle itself is pinned by tests/test_oracle.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libk3oracle.so")
_SRC = os.path.join(_HERE, "k3oracle.c")

FAULTS = {
    "none": 0, "nibble_order": 1, "scale_bias": 2, "drop_shared": 3, "no_renorm": 4,
    "tie_high": 5, "down_transposed": 6, "glu_on_up": 7, "bias_in_gate": 8, "no_bias_select": 9,
    "silu_sign": 10, "e2m1_table": 11, "shared_gated": 12, "select_lowest": 13, "renorm_short": 14,
    "rms_sum": 15, "scale_block": 16,
}
SCORES = {"softmax": 0, "sigmoid_bias": 1}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, no fast-math, no FMA contraction, OpenMP over tokens)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-o", _SO, _SRC, "-lm"])
    return _SO


_lib = None
_P = ctypes.c_void_p


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.k3o_set_fault.argtypes = [ctypes.c_int]
        L.k3o_e2m1.argtypes = [ctypes.c_int]
        L.k3o_e2m1.restype = ctypes.c_double
        L.k3o_e8m0.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
        L.k3o_e8m0.restype = ctypes.c_int
        L.k3o_record_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
        L.k3o_record_bytes.restype = ctypes.c_int64
        L.k3o_decode_matrix.argtypes = [_P, _P, ctypes.c_int64, ctypes.c_int64, _P]
        L.k3o_decode_matrix.restype = ctypes.c_int
        L.k3o_bf16.argtypes = [ctypes.c_uint16]
        L.k3o_bf16.restype = ctypes.c_double
        L.k3o_route_token.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P, _P, _P,
                                      ctypes.c_int32]
        L.k3o_route_token.restype = ctypes.c_int
        L.k3o_route_tokens.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, ctypes.c_int32,
                                       ctypes.c_int64, _P, _P, _P, _P, _P, ctypes.c_int32]
        L.k3o_route_tokens.restype = ctypes.c_int
        L.k3o_expert_token.argtypes = [ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P]
        L.k3o_expert_token.restype = ctypes.c_int
        L.k3o_expert_token_bf16.argtypes = [ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P]
        L.k3o_expert_token_bf16.restype = ctypes.c_int
        L.k3o_layer.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                _P, ctypes.c_int32, ctypes.c_int64, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int32,
                                ctypes.c_int32]
        L.k3o_layer.restype = ctypes.c_int
        L.k3o_rmsnorm.argtypes = [_P, ctypes.c_int64, ctypes.c_int32, ctypes.c_double, _P]
        L.k3o_rmsnorm.restype = None
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


class fault:
    """Context manager that switches the oracle to a deliberately wrong variant (tests only)."""

    def __init__(self, name: str):
        self.code = FAULTS[name]

    def __enter__(self):
        lib().k3o_set_fault(self.code)

    def __exit__(self, *exc):
        lib().k3o_set_fault(0)


def e2m1(code: int) -> float:
    return lib().k3o_e2m1(code)


def e8m0(b: int) -> float:
    v = ctypes.c_double()
    if lib().k3o_e8m0(b, ctypes.byref(v)):
        raise ValueError(f"E8M0 byte {b} is not a finite scale")
    return v.value


def record_bytes(d: int, f: int) -> int:
    return lib().k3o_record_bytes(d, f)


def split_record(rec: np.ndarray, d: int, f: int):
    """Views (codes, scales) of gate, up, down inside one record."""
    nc, ns = d * f // 2, d * f // 32
    parts, off = [], 0
    for _ in range(3):
        parts.append((rec[off:off + nc], rec[off + nc:off + nc + ns]))
        off += nc + ns
    return parts


def decode_matrix(codes: np.ndarray, scales: np.ndarray, rows: int, cols: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.empty((rows, cols), dtype=np.float64)
    if lib().k3o_decode_matrix(_ptr(codes), _ptr(scales), rows, cols, _ptr(out)):
        raise ValueError("decode_matrix: bad scale byte or shape")
    return out


def route_token(x: np.ndarray, W: np.ndarray, k: int, bias: np.ndarray | None = None, score: str = "softmax"):
    """-> (logits[E], idx[k], w[k]) for one token given as exact float64 values. score 'softmax' (bias
    added to the logits) or 'sigmoid_bias' (logits without bias; selection by sigmoid + bias, gates
    from the unbiased sigmoid)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    W = np.ascontiguousarray(W, dtype=np.float32)
    E, d = W.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    logits = np.empty(E, np.float64)
    idx = np.empty(k, np.int32)
    w = np.empty(k, np.float64)
    if lib().k3o_route_token(E, d, k, _ptr(x), _ptr(W), _ptr(b), _ptr(logits), _ptr(idx), _ptr(w), SCORES[score]):
        raise ValueError("route_token failed")
    return logits, idx, w


def route_tokens(x: np.ndarray, x_dtype: str, W: np.ndarray, k: int, bias: np.ndarray | None = None,
                 score: str = "softmax"):
    """Routing of T tokens (route_token per token, tokens in parallel): x [T, d] uint16 bf16 bits
    ('bf16') or float32 ('f32'). -> (logits[T, E], idx[T, k], w[T, k])."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    E, d = W.shape
    xa = np.ascontiguousarray(x, dtype=np.uint16 if x_dtype == "bf16" else np.float32)
    if xa.ndim != 2 or xa.shape[1] != d:
        raise ValueError("route_tokens: x must be [T, d]")
    T = xa.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    logits = np.empty((T, E), np.float64)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    if lib().k3o_route_tokens(E, d, k, _ptr(xa), 1 if x_dtype == "bf16" else 0, T, _ptr(W), _ptr(b), _ptr(logits),
                              _ptr(idx), _ptr(w), SCORES[score]):
        raise ValueError("route_tokens failed")
    return logits, idx, w


def expert_token(record: np.ndarray, x: np.ndarray, d: int, f: int):
    """-> (o[d], h[f]) of one expert on one token (x as exact float64 values)."""
    record = np.ascontiguousarray(record, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float64)
    o = np.empty(d, np.float64)
    h = np.empty(f, np.float64)
    if lib().k3o_expert_token(d, f, _ptr(record), _ptr(x), _ptr(o), _ptr(h)):
        raise ValueError("expert_token: bad record")
    return o, h


def expert_token_bf16(record: np.ndarray, x: np.ndarray, d: int, f: int):
    """-> (o[d], h[f]) of one expert with bf16 weights (record: [gate f x d][up f x d][down d x f] uint16
    bf16 bit patterns) on one token (exact float64 values)."""
    record = np.ascontiguousarray(record, dtype=np.uint16)
    if record.size < 3 * d * f:
        raise ValueError("expert_token_bf16: record too small")
    x = np.ascontiguousarray(x, dtype=np.float64)
    o = np.empty(d, np.float64)
    h = np.empty(f, np.float64)
    if lib().k3o_expert_token_bf16(d, f, _ptr(record), _ptr(x), _ptr(o), _ptr(h)):
        raise ValueError("expert_token_bf16 failed")
    return o, h


def layer(x: np.ndarray, x_dtype: str, W: np.ndarray, bias, routed: dict | list, shared: list,
          d: int, f: int, k: int, score: str = "softmax", shared_format: str = "mxfp4"):
    """One MoE layer on T tokens.

    x: [T, d] uint16 bf16 bits (x_dtype 'bf16') or float32 ('f32').
    routed: list of E records, or dict {expert id: record} holding at least the selected experts.
    shared: S records, MXFP4 (shared_format 'mxfp4', uint8) or bf16 ('bf16', uint16 bit patterns).
    Returns (y[T, d] float64, idx[T, k] int32, w[T, k] float64, logits[T, E] float64).
    """
    W = np.ascontiguousarray(W, dtype=np.float32)
    E = W.shape[0]
    T = x.shape[0]
    if x_dtype == "bf16":
        xa = np.ascontiguousarray(x, dtype=np.uint16)
    elif x_dtype == "f32":
        xa = np.ascontiguousarray(x, dtype=np.float32)
    else:
        raise ValueError(x_dtype)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    keep = []
    rp = (ctypes.c_void_p * E)()
    for e in range(E):
        r = routed.get(e) if isinstance(routed, dict) else routed[e]
        if r is not None:
            r = np.ascontiguousarray(r, dtype=np.uint8)
            keep.append(r)
            rp[e] = r.ctypes.data
    if shared_format not in ("mxfp4", "bf16"):
        raise ValueError(shared_format)
    sp = (ctypes.c_void_p * max(1, len(shared)))()
    for s, r in enumerate(shared):
        r = np.ascontiguousarray(r, dtype=np.uint8 if shared_format == "mxfp4" else np.uint16)
        keep.append(r)
        sp[s] = r.ctypes.data
    y = np.empty((T, d), np.float64)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    logits = np.empty((T, E), np.float64)
    rc = lib().k3o_layer(d, f, E, k, len(shared), _ptr(xa), 1 if x_dtype == "bf16" else 0, T, _ptr(W), _ptr(b),
                         ctypes.cast(rp, ctypes.c_void_p), ctypes.cast(sp, ctypes.c_void_p), _ptr(y), _ptr(idx),
                         _ptr(w), _ptr(logits), SCORES[score], 1 if shared_format == "bf16" else 0)
    if rc:
        raise ValueError(f"oracle layer failed ({rc})")
    return y, idx, w, logits


def rmsnorm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    lib().k3o_rmsnorm(_ptr(x), x.shape[0], x.shape[1], eps, _ptr(out))
    return out
