"""Seeded synthetic inputs for the MXFP4 MoE layer (shared by the oracle side and the CUDA side).

This module holds none of the method's arithmetic. It draws reproducible inputs
with the shapes and value distributions of the workloads:

* expert records: uniform 4-bit E2M1 codes (two per byte, low nibble first) and
  E8M0 scale bytes 127 + e with e uniform in {-6..-2}, one per 32 weights
  (host: ``synth_host.c``; device: ``synth_dev.cu``, bit-identical);
* router weights: fp32 N(0, 1/d);
* token activations: N(0, 1), stored as bf16 (round-to-nearest-even) or fp32;
* an optional Zipf(s) routing bias b_e = -s * ln(r_e), r a seeded permutation of 1..E;
* bf16 shared-expert records (the bf16 variant): N(0, 1/8^2) weights rounded to bf16, [gate f x d]
  [up f x d][down d x f] row-major, zero padding to the stride.

All randomness comes from SplitMix64 (Steele, Lea, Flood, OOPSLA 2014) used
counter-based; normals use the Box-Muller cosine branch.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
GAMMA = 0x9E3779B97F4A7C15
_M64 = (1 << 64) - 1

KIND_CODES, KIND_SCALES, KIND_ROUTER, KIND_TOKENS, KIND_BIAS, KIND_SHARED_BF16 = 1, 2, 3, 4, 5, 6


# --------------------------------------------------------------------------- configs
@dataclass(frozen=True)
class LayerShape:
    d_model: int
    d_ff: int
    n_routed: int
    top_k: int
    n_shared: int

    @property
    def record_bytes(self) -> int:
        return 3 * (self.d_model * self.d_ff // 2 + self.d_model * self.d_ff // 32)

    @property
    def record_stride(self) -> int:
        return (self.record_bytes + 4095) // 4096 * 4096


@dataclass(frozen=True)
class Workload:
    name: str
    shape: LayerShape
    tokens: tuple
    x_dtype: str  # "bf16" or "f32"
    seeds: tuple  # one seed per layer
    zipf_s: float | None = None
    prenorm_residual: bool = False
    notes: str = ""


K3 = LayerShape(d_model=7168, d_ff=1536, n_routed=896, top_k=16, n_shared=2)
TINY = LayerShape(d_model=256, d_ff=128, n_routed=32, top_k=4, n_shared=1)

WORKLOADS = {
    "tiny": Workload("tiny", TINY, (8,), "f32", (0,),
                     notes="d_model 256, d_ff 128, 32 routed top-4 + 1 shared, 8 tokens, fp32 x"),
    "decode_b1": Workload("decode_b1", K3, (1,), "bf16", (1,),
                          notes="one token, d_model 7168, d_ff 1536, 896 routed top-16 + 2 shared"),
    "decode_b64_zipf": Workload("decode_b64_zipf", K3, (64,), "bf16", (2,), zipf_s=1.1,
                                notes="64 tokens, Zipf(1.1)-skewed routing bias"),
    "prefill_4096": Workload("prefill_4096", K3, (4096,), "bf16", (3,),
                             notes="4096 tokens, unbiased router"),
    "stack4_zipf": Workload("stack4_zipf", K3, (1, 8, 64, 512, 4096, 16384), "f32", (40, 41, 42, 43),
                            zipf_s=1.1, prenorm_residual=True,
                            notes="4 layers, pre-norm residual, Zipf(1.1) routing bias"),
}


# --------------------------------------------------------------------------- splitmix64 (numpy)
def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=False)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def _mix64_int(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def stream_key(seed: int, kind: int, layer: int, expert: int = 0, matrix: int = 0) -> int:
    tag = ((kind & 0xFF) << 56) | ((layer & 0xFFFF) << 40) | ((expert & 0xFFFFFFFF) << 8) | (matrix & 0xFF)
    return _mix64_int(((seed * GAMMA) & _M64) ^ _mix64_int(tag))


def stream_values(key: int, start: int, n: int) -> np.ndarray:
    """Outputs start .. start+n-1 of the counter-based stream with state `key`."""
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(key) + i * np.uint64(GAMMA))


def normals(key: int, n: int, chunk: int = 1 << 22) -> np.ndarray:
    """n standard normals (float64), Box-Muller cosine branch on output pairs (2i, 2i+1)."""
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        v = stream_values(key, 2 * s, 2 * m)
        u1 = ((v[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (v[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        out[s:s + m] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 -> bfloat16 (nearest-even), returned as uint16 bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------- dense inputs
def router_weights(shape: LayerShape, seed: int, layer: int = 0) -> np.ndarray:
    """fp32 [E, d] with entries N(0, 1/d)."""
    z = normals(stream_key(seed, KIND_ROUTER, layer), shape.n_routed * shape.d_model)
    return (z / math.sqrt(shape.d_model)).astype(np.float32).reshape(shape.n_routed, shape.d_model)


def tokens(shape: LayerShape, seed: int, T: int, x_dtype: str, batch: int = 0) -> np.ndarray:
    """Token activations N(0,1): uint16 bf16 bits [T, d] if x_dtype == 'bf16', else float32 [T, d]."""
    z = normals(stream_key(seed, KIND_TOKENS, 0, batch), T * shape.d_model).astype(np.float32)
    z = z.reshape(T, shape.d_model)
    if x_dtype == "bf16":
        return f32_to_bf16_bits(z)
    if x_dtype == "f32":
        return z
    raise ValueError(x_dtype)


def tokens_as_f64(x: np.ndarray, x_dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(x).astype(np.float64) if x_dtype == "bf16" else np.asarray(x, np.float64)


def shared_bf16_record_bytes(shape: LayerShape) -> int:
    return 3 * shape.d_model * shape.d_ff * 2


def shared_bf16_stride(shape: LayerShape) -> int:
    return (shared_bf16_record_bytes(shape) + 4095) // 4096 * 4096


def shared_records_bf16(shape: LayerShape, seed: int, layer: int, n: int, stride: int | None = None) -> np.ndarray:
    """n bf16 shared-expert records as uint16 [n, stride/2]: N(0, 1/64) values rounded to bf16
    (nearest-even), gate, up and down matrices row-major, then zero padding."""
    stride = stride or shared_bf16_stride(shape)
    m = 3 * shape.d_model * shape.d_ff
    out = np.zeros((n, stride // 2), dtype=np.uint16)
    for s_ in range(n):
        z = normals(stream_key(seed, KIND_SHARED_BF16, layer, s_), m) * 0.125
        out[s_, :m] = f32_to_bf16_bits(z.astype(np.float32))
    return out


def zipf_bias(shape: LayerShape, seed: int, s: float, layer: int = 0) -> np.ndarray:
    """Routing bias b_e = -s ln(r_e), r = seeded permutation of 1..E (float32 [E])."""
    v = stream_values(stream_key(seed, KIND_BIAS, layer), 0, shape.n_routed)
    ranks = np.empty(shape.n_routed, dtype=np.int64)
    ranks[np.argsort(v, kind="stable")] = np.arange(1, shape.n_routed + 1)
    return (-s * np.log(ranks.astype(np.float64))).astype(np.float32)


# --------------------------------------------------------------------------- expert records
def _build_host_lib() -> str:
    so = os.path.join(_HERE, "libk3synth_host.so")
    src = os.path.join(_HERE, "synth_host.c")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", so, src])
    return so


_host_lib = None


def _host():
    global _host_lib
    if _host_lib is None:
        lib = ctypes.CDLL(_build_host_lib())
        lib.k3s_fill_records.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                                         ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int64, ctypes.c_int64]
        lib.k3s_fill_records.restype = ctypes.c_int
        lib.k3s_key.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
        lib.k3s_key.restype = ctypes.c_uint64
        lib.k3s_value.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.k3s_value.restype = ctypes.c_uint64
        _host_lib = lib
    return _host_lib


def records_host(shape: LayerShape, seed: int, layer: int, experts, stride: int | None = None) -> np.ndarray:
    """Records of the given expert ids (routed 0..E-1, shared E..E+S-1) as uint8 [n, stride]."""
    stride = stride or shape.record_stride
    experts = list(experts)
    out = np.empty((len(experts), stride), dtype=np.uint8)
    lib = _host()
    for i, e in enumerate(experts):
        rc = lib.k3s_fill_records(out[i].ctypes.data, shape.d_model, shape.d_ff, seed, layer, e, 1, stride)
        if rc != 0:
            raise ValueError("k3s_fill_records failed")
    return out


def records_host_numpy(shape: LayerShape, seed: int, layer: int, expert: int, stride: int | None = None) -> np.ndarray:
    """Pure-numpy twin of the C generator for one record (used to pin the generator itself)."""
    stride = stride or shape.record_stride
    d, f = shape.d_model, shape.d_ff
    nc, ns = d * f // 2, d * f // 32
    out = np.zeros(stride, dtype=np.uint8)
    for m in range(3):
        base = m * (nc + ns)
        words = stream_values(stream_key(seed, KIND_CODES, layer, expert, m), 0, (nc + 7) // 8)
        out[base:base + nc] = words.view(np.uint8)[:nc] if np.little_endian else words.byteswap().view(np.uint8)[:nc]
        v = stream_values(stream_key(seed, KIND_SCALES, layer, expert, m), 0, ns)
        e5 = ((v >> np.uint64(32)) * np.uint64(5)) >> np.uint64(32)
        out[base + nc:base + nc + ns] = (121 + e5).astype(np.uint8)
    return out


# Device generator: libk3synth_dev.so (built by __graft_entry__.build or build_device_lib()).
_dev_lib = None


def build_device_lib(force: bool = False) -> str:
    so = os.path.join(_HERE, "libk3synth_dev.so")
    src = os.path.join(_HERE, "synth_dev.cu")
    if force or not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                               "-Xcompiler", "-fPIC", "-shared", "-o", so, src])
    return so


def _dev():
    global _dev_lib
    if _dev_lib is None:
        so = os.path.join(_HERE, "libk3synth_dev.so")
        if not os.path.exists(so):
            raise RuntimeError("libk3synth_dev.so is not built; run __graft_entry__.build()")
        lib = ctypes.CDLL(so)
        lib.k3s_fill_records_device.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                                                ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_void_p]
        lib.k3s_fill_records_device.restype = ctypes.c_int
        _dev_lib = lib
    return _dev_lib


def records_device(shape: LayerShape, seed: int, layer: int, e0: int, n: int, dst_ptr: int, stride: int,
                   stream_ptr: int = 0) -> None:
    """Fill n records (ids e0..e0+n-1) at device pointer dst_ptr, asynchronously on stream_ptr."""
    rc = _dev().k3s_fill_records_device(ctypes.c_void_p(dst_ptr), shape.d_model, shape.d_ff, seed, layer, e0, n,
                                        stride, ctypes.c_void_p(stream_ptr))
    if rc != 0:
        raise RuntimeError(f"k3s_fill_records_device failed ({rc})")
