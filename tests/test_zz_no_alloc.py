"""The allocation-free entry point k3moe_layer_static (GPU).

Callers that cannot allocate device memory (a host program whose own pool owns every allocation,
or a latency-critical path that cannot afford cudaMalloc's synchronisation) use k3moe_layer_static,
which takes its scratch from a fixed array inside the library. These tests call it through the C ABI
twice in a row and compare each result with k3moe_layer run on a caller-allocated workspace, within
the suite's tolerance. This file is collected last on purpose, and passes alone or after the others.
"""
import ctypes

import numpy as np
import pytest

import synth
from harness import REL_TOL, DeviceLayer, rel_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU machine
    pytest.skip("needs a GPU", allow_module_level=True)

import mxfp4_routed_expert_k3moe_gb300 as k3  # noqa: E402

MID = synth.LayerShape(d_model=512, d_ff=256, n_routed=64, top_k=6, n_shared=2)


def _static_call(L, xd, T, y):
    lib = k3.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.k3moe_layer_static(ctypes.byref(L.cfg), ctypes.c_void_p(xd.data_ptr()), T,
                                  ctypes.c_void_p(L.W.data_ptr()),
                                  None if L.bias is None else ctypes.c_void_p(L.bias.data_ptr()),
                                  ctypes.c_void_p(L.routed.data_ptr()), ctypes.c_void_p(L.shared.data_ptr()),
                                  ctypes.c_void_p(y.data_ptr()), stream)


def _workspace_call(L, xd, T):
    y = torch.empty((T, L.shape.d_model), dtype=torch.float32, device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.layer(L.cfg, xd, T, L.W, L.bias, L.routed, L.shared, y, ws)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("shape,T,x_dtype,zipf", [(MID, 13, "bf16", 1.1), (MID, 5, "f32", None),
                                                  (synth.K3, 1, "bf16", None)])
def test_static_scratch_matches_workspace_entry_point(shape, T, x_dtype, zipf):
    L = DeviceLayer(shape, seed=21, zipf_s=zipf, x_dtype=x_dtype)
    for call in range(2):  # two calls in a row: the second reuses the array left by the first
        _, xd = L.tokens(T, batch=call)
        y = torch.full((T, shape.d_model), float("nan"), dtype=torch.float32, device="cuda")
        rc = _static_call(L, xd, T, y)
        assert rc == k3.OK, k3.status_string(rc)
        torch.cuda.synchronize()
        y_static = y.cpu().numpy()
        assert np.isfinite(y_static).all()
        err = rel_err(y_static, _workspace_call(L, xd, T))
        assert err <= REL_TOL, (call, err)


def test_static_scratch_rejects_calls_beyond_its_size():
    """The documented limit at the K3 shape: up to 6 tokens are served, 7 are refused."""
    L = DeviceLayer(synth.K3, seed=22)
    T = next(t for t in range(1, 64) if k3.workspace_bytes(L.cfg, t) > (4 << 20))
    assert T == 7
    _, xd = L.tokens(T)
    y = torch.empty((T, synth.K3.d_model), dtype=torch.float32, device="cuda")
    assert _static_call(L, xd, T, y) == k3.ERR_WORKSPACE
