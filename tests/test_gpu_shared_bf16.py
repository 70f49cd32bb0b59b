"""Shared experts in bf16 (the kimi-k3-in-c README's parameter budget counts every non-routed parameter
in bfloat16) on the GPU, against the oracle's bf16 shared mode: the layer through the C ABI, with bf16
and fp32 tokens, through both router paths, at the MID and K3 shapes, and the expert FFN for given
routing. A bf16 record holding exactly the values of an MXFP4 record must give the MXFP4 layer's result
(the oracle gives the two bit-identical outputs)."""
import numpy as np
import pytest

import synth
from harness import REL_TOL, DeviceLayer, gate_err, index_parity, rel_err, GATE_TOL

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU machine
    pytest.skip("needs a GPU", allow_module_level=True)

import mxfp4_routed_expert_k3moe_gb300 as k3  # noqa: E402

MID = synth.LayerShape(d_model=512, d_ff=256, n_routed=64, top_k=6, n_shared=2)


def run(L: DeviceLayer, xd, T):
    sh = L.shape
    y = torch.full((T, sh.d_model), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, sh.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, sh.top_k), dtype=torch.float32, device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.layer(L.cfg, xd, T, L.W, L.bias, L.routed, L.shared, y, ws, idx, w)
    assert k3.check_device_status(ws) == k3.OK
    torch.cuda.synchronize()
    return y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def check(L: DeviceLayer, T: int, rows=None):
    xh, xd = L.tokens(T)
    y, idx, w = run(L, xd, T)
    rows = np.arange(T) if rows is None else np.asarray(rows)
    y_ref, idx_ref, w_ref, logits_ref = L.oracle(xh, rows)
    ok, near, msg = index_parity(idx[rows], idx_ref, L.sel_keys(logits_ref), L.shape.top_k)
    assert ok, msg
    keep = [i for i in range(len(rows)) if i not in near]
    assert gate_err(idx[rows][keep], w[rows][keep], idx_ref[keep], w_ref[keep]) < GATE_TOL
    err = rel_err(y[rows][keep], y_ref[keep])
    assert err <= REL_TOL, err
    return err


@pytest.mark.parametrize("T,x_dtype", [(1, "bf16"), (5, "bf16"), (37, "bf16"), (3, "f32"), (20, "f32")])
def test_layer_bf16_shared_mid(T, x_dtype):
    """CUDA-core router below 16 tokens, tensor-core router from 16; fp32 tokens split into three bf16
    parts for the shared GEMM (by the router's split from 16 tokens, by the shared path below)."""
    L = DeviceLayer(MID, seed=50, zipf_s=1.1, x_dtype=x_dtype, shared_format="bf16")
    check(L, T)


def test_layer_bf16_shared_k3_decode():
    L = DeviceLayer(synth.K3, seed=51, shared_format="bf16")
    err = check(L, 1)
    assert err < 1e-4


def test_layer_bf16_shared_k3_many_tokens_sampled():
    L = DeviceLayer(synth.K3, seed=52, shared_format="bf16")
    check(L, 300, rows=[0, 149, 299])


def test_expert_ffn_bf16_shared_given_routing():
    L = DeviceLayer(MID, seed=53, x_dtype="f32", shared_format="bf16")
    T = 9
    xh, xd = L.tokens(T)
    rng = np.random.default_rng(1)
    idx = np.stack([rng.choice(MID.n_routed, MID.top_k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, MID.top_k)).astype(np.float32)
    y = torch.empty((T, MID.d_model), dtype=torch.float32, device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.expert_ffn(L.cfg, xd, T, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), L.routed, L.shared, y, ws)
    assert k3.check_device_status(ws) == k3.OK
    assert rel_err(y.cpu().numpy(), L.oracle_ffn(xh, idx, w)) <= REL_TOL


@pytest.mark.parametrize("T", [2, 24])
def test_bf16_image_of_mxfp4_shared_matches_mxfp4_layer(T):
    """The same layer with its shared experts as MXFP4 records and as bf16 records holding exactly their
    values (decoded by the oracle, exact in bf16): both GPU results within the bar of the one oracle
    result."""
    import oracle
    Lm = DeviceLayer(MID, seed=54)
    Lb = DeviceLayer(MID, seed=54, shared_format="bf16")
    d, f = MID.d_model, MID.d_ff
    recs = []
    for r in Lm.host_records([MID.n_routed + s for s in range(MID.n_shared)]).values():
        dense = [oracle.decode_matrix(c, sc, *dims) for (c, sc), dims in
                 zip(oracle.split_record(r, d, f), [(f, d), (f, d), (d, f)])]
        flat = np.concatenate([m.ravel() for m in dense])
        bits = synth.f32_to_bf16_bits(flat.astype(np.float32))
        assert np.array_equal(synth.bf16_bits_to_f32(bits).astype(np.float64), flat)
        rec = np.zeros(Lb.sstride // 2, np.uint16)
        rec[:bits.size] = bits
        recs.append(rec)
    Lb.set_shared_bf16(np.stack(recs))
    xh, xd = Lm.tokens(T)
    ym, im, _ = run(Lm, xd, T)
    yb, ib, _ = run(Lb, xd, T)
    assert np.array_equal(im, ib)
    y_ref = Lm.oracle(xh)[0]
    assert rel_err(ym, y_ref) <= REL_TOL and rel_err(yb, y_ref) <= REL_TOL
