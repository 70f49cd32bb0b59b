"""The C ABI: libk3moe.so loads, exports every function include/k3moe.h declares, and rejects invalid
arguments on the host before any CUDA call (CPU only, no compute)."""
import ctypes
import os
import re

import pytest

import mxfp4_routed_expert_k3moe_gb300 as k3

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "k3moe.h")).read()
    return sorted(set(re.findall(r"K3MOE_API\s+[\w\s\*]*?\b(k3moe_\w+)\s*\(", src)))


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ["k3moe_route", "k3moe_expert_ffn", "k3moe_layer", "k3moe_workspace_bytes", "k3moe_check_device_status"]:
        assert n in names
    assert sorted(names) == sorted(k3.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = k3.load()
    for n in declared_functions():
        assert hasattr(lib, n), n


K3CFG = dict(d_model=7168, d_ff=1536, n_routed=896, top_k=16, n_shared=2)


def test_record_and_workspace_sizes():
    cfg = k3.Config.make(**K3CFG)
    assert k3.record_bytes(cfg) == 17547264
    assert cfg.record_stride == 17547264  # already a multiple of 4096
    w1, w64 = k3.workspace_bytes(cfg, 1), k3.workspace_bytes(cfg, 64)
    assert 0 < w1 < w64


@pytest.mark.parametrize("act_mode", [k3.ACT_EXACT, k3.ACT_BF16H])
@pytest.mark.parametrize("x_dtype", [k3.X_BF16, k3.X_F32])
def test_workspace_never_shrinks_as_tokens_grow(x_dtype, act_mode):
    """A workspace sized for T tokens serves every call with fewer (the router's partial logits vary
    in count with the token tiles, the activation form changes at 3 tokens, the router at 16, x's
    terms are also kept in position order from 256)."""
    cfg = k3.Config.make(**K3CFG, x_dtype=x_dtype, act_mode=act_mode)
    Ts = sorted(set(list(range(1, 300)) + [383, 384, 385, 511, 512, 513, 600, 640, 700, 1023, 1024, 1025,
                                           2047, 2048, 4095, 4096, 4097, 16384, 19456, 19457, 20000]))
    sizes = [k3.workspace_bytes(cfg, T) for T in Ts]
    assert all(s > 0 for s in sizes)
    assert all(b >= a for a, b in zip(sizes, sizes[1:]))


@pytest.mark.parametrize("field,value,code", [
    ("d_model", 100, k3.ERR_INVALID_ARGUMENT),   # not a multiple of 32
    ("d_model", 160, k3.ERR_UNSUPPORTED),        # a multiple of 32, not of 128: legal, not implemented
    ("d_ff", 0, k3.ERR_INVALID_ARGUMENT),
    ("d_ff", 1504, k3.ERR_UNSUPPORTED),
    ("top_k", 0, k3.ERR_INVALID_ARGUMENT),
    ("top_k", 33, k3.ERR_INVALID_ARGUMENT),
    ("n_routed", 5000, k3.ERR_INVALID_ARGUMENT),
    ("n_shared", -1, k3.ERR_INVALID_ARGUMENT),
    ("record_stride", 17547264 - 4096, k3.ERR_INVALID_ARGUMENT),  # below the record size
    ("record_stride", 17547264 + 256, k3.ERR_INVALID_ARGUMENT),   # not 4 KiB aligned
    ("record_stride", 17547264 + 8, k3.ERR_INVALID_ARGUMENT),
    ("shared_stride", 4096, k3.ERR_INVALID_ARGUMENT),             # below the shared record size
    ("shared_stride", 17547264 + 100, k3.ERR_INVALID_ARGUMENT),
    ("x_dtype", 7, k3.ERR_INVALID_ARGUMENT),
    ("score_func", 7, k3.ERR_INVALID_ARGUMENT),
    ("record_order", 7, k3.ERR_INVALID_ARGUMENT),
    ("shared_format", 7, k3.ERR_INVALID_ARGUMENT),
    ("act_mode", k3.ACT_MXFP4, k3.ERR_UNSUPPORTED),
    ("act_mode", 3, k3.ERR_INVALID_ARGUMENT),
    ("record_order", k3.ORDER_STORED, k3.ERR_UNSUPPORTED),        # records never packed are refused
])
def test_invalid_config_rejected_on_host(field, value, code):
    cfg = k3.Config.make(**K3CFG)
    setattr(cfg, field, value)
    lib = k3.load()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    rc = lib.k3moe_layer(ctypes.byref(cfg), fake, 1, fake, None, None, fake, fake, fake, None, None, fake, 1 << 30, None)
    assert rc == code
    rc = lib.k3moe_expert_ffn(ctypes.byref(cfg), fake, 1, fake, fake, fake, fake, fake, fake, 1 << 30, None)
    assert rc == code
    rc = lib.k3moe_layer_static(ctypes.byref(cfg), fake, 1, fake, None, fake, fake, fake, None)
    assert rc == code


def test_stored_order_is_refused_only_by_calls_that_read_records():
    cfg = k3.Config.make(**K3CFG, record_order=k3.ORDER_STORED)
    lib = k3.load()
    a = ctypes.c_void_p(1 << 20)
    assert lib.k3moe_route(ctypes.byref(cfg), a, 0, a, None, None, a, a, a, 1 << 30, None) == k3.OK
    assert lib.k3moe_layer(ctypes.byref(cfg), a, 0, a, None, None, a, a, a, None, None, a, 0, None) == k3.ERR_UNSUPPORTED
    # a zero-initialised config (no order given) is the stored order
    assert k3.Config().record_order == k3.ORDER_STORED


def test_invalid_pointers_rejected_on_host():
    cfg = k3.Config.make(**K3CFG)
    lib = k3.load()
    a = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 8)
    big = 1 << 34
    assert lib.k3moe_layer(ctypes.byref(cfg), None, 1, a, None, None, a, a, a, None, None, a, big, None) == 1
    assert lib.k3moe_layer(ctypes.byref(cfg), mis, 1, a, None, None, a, a, a, None, None, a, big, None) == 1
    assert lib.k3moe_layer(ctypes.byref(cfg), a, -1, a, None, None, a, a, a, None, None, a, big, None) == 1
    assert lib.k3moe_layer(ctypes.byref(cfg), a, 1, a, mis, None, a, a, a, None, None, a, big, None) == 1  # parts
    assert lib.k3moe_route(ctypes.byref(cfg), a, 1, a, None, None, None, a, a, big, None) == 1
    assert lib.k3moe_expert_ffn(ctypes.byref(cfg), a, 1, a, a, a, None, a, a, big, None) == 1  # shared missing
    ws_mis = ctypes.c_void_p((1 << 20) + 16)
    assert lib.k3moe_layer(ctypes.byref(cfg), a, 1, a, None, None, a, a, a, None, None, ws_mis, big, None) == 1
    assert lib.k3moe_layer(ctypes.byref(cfg), a, 4, a, None, None, a, a, a, None, None, a, 1024, None) == k3.ERR_WORKSPACE
    assert lib.k3moe_layer_bounded(ctypes.byref(cfg), a, 1, a, None, None, a, a, a, a, big, 0, None) == 1  # bound 0
    assert lib.k3moe_prepare_router(ctypes.byref(cfg), None, a, None) == 1
    assert lib.k3moe_prepare_router(ctypes.byref(cfg), a, mis, None) == 1
    assert lib.k3moe_residual_rmsnorm(a, None, 1, 7166, 1e-6, a, None) == 1   # d not a multiple of 4
    assert lib.k3moe_residual_rmsnorm(a, mis, 1, 7168, 1e-6, a, None) == 1
    assert lib.k3moe_residual_rmsnorm(a, None, 0, 7168, 1e-6, a, None) == k3.OK


def test_bf16_shared_config():
    """bf16 shared records: the default stride is the bf16 record rounded to 4 KiB; a smaller one is
    rejected; the workspace holds the shared GEMMs' partial sums and h (and grows with T)."""
    lib = k3.load()
    a = ctypes.c_void_p(1 << 20)
    cfg = k3.Config.make(**K3CFG, shared_format=k3.SHARED_BF16)
    assert lib.k3moe_layer(ctypes.byref(cfg), a, 0, a, None, None, a, a, a, None, None, a, 0, None) == k3.OK
    assert k3.workspace_bytes(cfg, 1) > k3.workspace_bytes(k3.Config.make(**K3CFG), 1)
    sizes = [k3.workspace_bytes(cfg, T) for T in (1, 2, 15, 16, 127, 128, 129, 1000, 4096)]
    assert all(b >= a_ for a_, b in zip(sizes, sizes[1:]))
    cfg.shared_stride = 6 * 7168 * 1536 - 4096
    assert lib.k3moe_layer(ctypes.byref(cfg), a, 0, a, None, None, a, a, a, None, None, a, 0, None) == 1
    cfg.shared_stride = (6 * 7168 * 1536 + 4095) // 4096 * 4096
    assert lib.k3moe_layer(ctypes.byref(cfg), a, 0, a, None, None, a, a, a, None, None, a, 0, None) == k3.OK


def test_router_parts_bytes():
    cfg = k3.Config.make(**K3CFG)
    assert k3.router_parts_bytes(cfg) == 3 * 896 * 7168 * 2


def test_pack_records_rejects_bad_arguments_on_host():
    cfg = k3.Config.make(**K3CFG)
    lib = k3.load()
    a = ctypes.c_void_p(1 << 20)
    assert lib.k3moe_pack_records(ctypes.byref(cfg), None, 1, 1, None) == k3.ERR_INVALID_ARGUMENT
    assert lib.k3moe_pack_records(ctypes.byref(cfg), ctypes.c_void_p((1 << 20) + 8), 1, 1, None) == 1
    assert lib.k3moe_pack_records(ctypes.byref(cfg), a, -1, 1, None) == k3.ERR_INVALID_ARGUMENT
    assert lib.k3moe_pack_records(ctypes.byref(cfg), a, 1, 2, None) == k3.ERR_INVALID_ARGUMENT
    assert lib.k3moe_pack_records(ctypes.byref(cfg), a, 0, 1, None) == k3.OK
    bad = k3.Config.make(**K3CFG)
    bad.d_ff = 100
    assert lib.k3moe_pack_records(ctypes.byref(bad), a, 1, 1, None) == k3.ERR_INVALID_ARGUMENT
    bad.d_ff = 1504  # a multiple of 32, not of 128: the device order is defined on 128-row tiles
    assert lib.k3moe_pack_records(ctypes.byref(bad), a, 1, 1, None) == k3.ERR_UNSUPPORTED


def test_zero_tokens_launches_nothing():
    cfg = k3.Config.make(**K3CFG)
    lib = k3.load()
    a = ctypes.c_void_p(1 << 20)
    assert lib.k3moe_layer(ctypes.byref(cfg), a, 0, a, None, None, a, a, a, None, None, a, 0, None) == k3.OK


def test_status_strings():
    for code in range(7):
        assert k3.status_string(code)
    assert k3.status_string(99) == "unknown status"


def test_static_scratch_limit_on_host():
    """k3moe_layer_static serves calls whose workspace fits its 4 MiB array: at the K3 shape up to 6
    tokens; 7 are refused with K3MOE_ERR_WORKSPACE before any CUDA call (the header's statement)."""
    src = open(os.path.join(ROOT, "include", "k3moe.h")).read()
    m = re.search(r"#define K3MOE_STATIC_SCRATCH_BYTES \((\d+)u << (\d+)\)", src)
    size = int(m.group(1)) << int(m.group(2))
    assert size == 4 << 20
    cfg = k3.Config.make(**K3CFG)
    assert k3.workspace_bytes(cfg, 6) <= size < k3.workspace_bytes(cfg, 7)
    lib = k3.load()
    a = ctypes.c_void_p(1 << 20)
    assert lib.k3moe_layer_static(ctypes.byref(cfg), a, 7, a, None, a, a, a, None) == k3.ERR_WORKSPACE
    assert lib.k3moe_layer_static(ctypes.byref(cfg), a, 0, a, None, a, a, a, None) == k3.OK
    assert lib.k3moe_layer_static(ctypes.byref(cfg), a, -1, a, None, a, a, a, None) == k3.ERR_INVALID_ARGUMENT


C_CLIENT = r"""
#include <stdio.h>
#include "k3moe.h"
int main(void) {
  k3moe_config c = {7168, 1536, 896, 16, 2, K3MOE_SCORE_SOFTMAX, K3MOE_ACT_EXACT, K3MOE_X_BF16,
                    K3MOE_ORDER_DEVICE, K3MOE_SHARED_MXFP4, 17547264, 0};
  printf("%zu %zu %zu %d %s\n", k3moe_record_bytes(&c), k3moe_workspace_bytes(&c, 1),
         k3moe_router_parts_bytes(&c), (int)k3moe_layer(&c, NULL, 1, NULL, NULL, NULL, NULL, NULL, NULL, NULL,
                                                    NULL, NULL, 0, NULL),
         k3moe_status_string(K3MOE_ERR_WORKSPACE));
  return 0;
}
"""


def test_plain_c_client(tmp_path):
    """The header is plain C99 (no CUDA or C++ types) and a C program links the library and calls it:
    host-only queries, and a compute call refused on the host (NULL x) before any CUDA call."""
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        pytest.skip("gcc not found")
    lib = k3.load()
    libdir = os.path.dirname(lib._name)
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I",
                           os.path.join(ROOT, "include"), str(src), "-L", libdir, "-lk3moe",
                           "-Wl,-rpath," + libdir, "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split(None, 4)
    cfg = k3.Config.make(**K3CFG)
    assert int(out[0]) == 17547264
    assert int(out[1]) == k3.workspace_bytes(cfg, 1)
    assert int(out[2]) == 3 * 896 * 7168 * 2
    assert int(out[3]) == k3.ERR_INVALID_ARGUMENT
    assert out[4].strip() == k3.status_string(k3.ERR_WORKSPACE)
