"""Parity of the CUDA path (through the C ABI) with the CPU oracle on the same seeded inputs.

Bars: expert indices exact except where the oracle's k-th and (k+1)-th logits differ by < 1e-5;
outputs within max|y_gpu - y_ref| / max|y_ref| <= 2e-3 (fp32 accumulation against fp64).
"""
import numpy as np
import pytest

import synth
from harness import REL_TOL, DeviceLayer, device_order, gate_err, index_parity, rel_err, GATE_TOL

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU machine
    pytest.skip("needs a GPU", allow_module_level=True)

import mxfp4_routed_expert_k3moe_gb300 as k3  # noqa: E402

MID = synth.LayerShape(d_model=512, d_ff=256, n_routed=64, top_k=6, n_shared=2)


def run_layer(L: DeviceLayer, xd, T, ws=None):
    sh = L.shape
    y = torch.empty((T, sh.d_model), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, sh.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, sh.top_k), dtype=torch.float32, device="cuda")
    if ws is None:
        ws = torch.zeros(k3.workspace_bytes(L.cfg, max(T, 1)), dtype=torch.uint8, device="cuda")
    k3.layer(L.cfg, xd, T, L.W, L.bias, L.routed, L.shared, y, ws, idx, w)
    assert k3.check_device_status(ws) == k3.OK
    torch.cuda.synchronize()
    return y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def check_layer(L: DeviceLayer, T: int, sample=None, batch=0):
    """The layer against the oracle. Indices and gates of EVERY token are checked (the oracle routes all
    of them); y on every token, or on `sample` where the oracle's expert FFN of all tokens would take
    too long. A token whose selection took the allowed near-tie exchange is checked against the
    oracle's FFN and combine evaluated on the GPU's own selection and gates."""
    xh, xd = L.tokens(T, batch)
    y, idx, w = run_layer(L, xd, T)
    k = L.shape.top_k
    if sample is not None:
        lg_all, idx_all, w_all = L.oracle_route(xh)
        ok, near_all, msg = index_parity(idx, idx_all, L.sel_keys(lg_all), k)
        assert ok, msg
        keep_all = [t for t in range(T) if t not in near_all]
        assert gate_err(idx[keep_all], w[keep_all], idx_all[keep_all], w_all[keep_all]) < GATE_TOL
    rows = np.arange(T) if sample is None else np.asarray(sample)
    y_ref, idx_ref, w_ref, logits_ref = L.oracle(xh, rows)
    ok, near, msg = index_parity(idx[rows], idx_ref, L.sel_keys(logits_ref), k)
    assert ok, msg
    keep = [i for i in range(len(rows)) if i not in near]
    assert gate_err(idx[rows][keep], w[rows][keep], idx_ref[keep], w_ref[keep]) < GATE_TOL
    err = rel_err(y[rows][keep], y_ref[keep])
    assert err <= REL_TOL, err
    if near:
        r = rows[near]
        y_alt = L.oracle_ffn(xh[r], idx[r], w[r])
        assert rel_err(y[r], y_alt) <= REL_TOL
    return err


# ------------------------------------------------------------------ generator


def test_device_generator_matches_host():
    sh = synth.TINY
    L = DeviceLayer(sh, seed=0, pack=False)
    dev = L.routed.cpu().numpy().reshape(sh.n_routed, L.stride)
    host = synth.records_host(sh, 0, 0, range(sh.n_routed), L.stride)
    assert np.array_equal(dev, host)
    shd = L.shared.cpu().numpy().reshape(-1, L.stride)[: sh.n_shared]
    assert np.array_equal(shd, synth.records_host(sh, 0, 0, [sh.n_routed], L.stride))


@pytest.fixture(scope="module")
def k3_decode_b1():
    return DeviceLayer(synth.K3, seed=1)


@pytest.fixture(scope="module")
def k3_decode_b64():
    return DeviceLayer(synth.K3, seed=2, zipf_s=1.1)


def test_device_generator_matches_host_k3(k3_decode_b1):
    """The fixture's records are generated on the device and put in the device order there."""
    L = k3_decode_b1
    d, f = L.shape.d_model, L.shape.d_ff
    for e in (0, 517, 895):
        dev = L.routed[e * L.stride:(e + 1) * L.stride].cpu().numpy()
        host = synth.records_host(L.shape, 1, 0, [e], L.stride)
        assert np.array_equal(dev, device_order(host, d, f)[0])


@pytest.mark.parametrize("shape", [synth.TINY, MID])
def test_pack_records_round_trip(shape):
    """Stored -> device order matches the host restatement; device -> stored restores every byte."""
    L = DeviceLayer(shape, seed=4, pack=False)
    E, d, f = shape.n_routed, shape.d_model, shape.d_ff
    stored = L.routed.cpu().numpy().reshape(E, L.stride)
    k3.pack_records(L.cfg, L.routed, E)
    packed = L.routed.cpu().numpy().reshape(E, L.stride)
    assert np.array_equal(packed, device_order(stored, d, f))
    assert not np.array_equal(packed, stored)
    k3.pack_records(L.cfg, L.routed, E, to_device=False)
    assert np.array_equal(L.routed.cpu().numpy().reshape(E, L.stride), stored)


# ------------------------------------------------------------------ layer parity


def test_layer_tiny_f32():
    L = DeviceLayer(synth.TINY, seed=0, x_dtype="f32")
    check_layer(L, 8)


@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [1, 2, 5, 37, 600])
def test_layer_mid_ragged(x_dtype, T):
    """Ragged token counts; at 600 tokens (~56 per expert) experts' token lists span several work
    groups, with the tensor-core router (partial logits) and E4M3 activation terms."""
    L = DeviceLayer(MID, seed=7, x_dtype=x_dtype)
    check_layer(L, T)


def test_layer_mid_zipf_skew():
    """Skewed routing: popular experts get many tokens (work groups split, several passes)."""
    L = DeviceLayer(MID, seed=8, zipf_s=3.0)
    check_layer(L, 45)


def test_layer_all_experts_selected_no_shared():
    sh = synth.LayerShape(d_model=256, d_ff=128, n_routed=8, top_k=8, n_shared=0)
    L = DeviceLayer(sh, seed=9)
    check_layer(L, 11)


def test_layer_decode_b1_full_size(k3_decode_b1):
    err = check_layer(k3_decode_b1, 1)
    assert err < 1e-4


def test_layer_decode_b64_zipf_full_size(k3_decode_b64):
    """Indices and gates of all 64 tokens, y of every fourth."""
    check_layer(k3_decode_b64, 64, sample=list(range(0, 64, 4)))


def test_layer_k3_f32_tokens_many_tiles_sampled():
    """fp32 tokens at the K3 width stage 4 tokens per router tile: 600 tokens make 150 tiles, each
    with its own arrival counter; tokens far past the first tiles are checked."""
    L = DeviceLayer(synth.K3, seed=14, x_dtype="f32")
    check_layer(L, 600, sample=[0, 259, 420, 599])


def test_layer_prefill_4096_sampled():
    """Indices and gates of all 4096 tokens; y of five."""
    L = DeviceLayer(synth.K3, seed=3)
    check_layer(L, 4096, sample=[0, 1, 777, 2048, 4095])


# ------------------------------------------------------------------ h as two E4M3 terms (K3MOE_ACT_BF16H)

@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [2, 3, 37, 600])
def test_layer_bf16h_mid(x_dtype, T):
    """The bf16-class h mode against the exact oracle at the same 2e-3 bound: 2 tokens take the exact
    E2M1 form, from 3 on h enters as two E4M3 terms with 32-position down work groups (600: from 256
    on, with x's terms in position order)."""
    L = DeviceLayer(MID, seed=40 + T, x_dtype=x_dtype, act="bf16h")
    err = check_layer(L, T)
    if T < 3:
        assert err < 1e-4


def test_layer_bf16h_k3_prefill_sampled():
    """Indices and gates of all 1024 tokens at the K3 shape, y of five."""
    L = DeviceLayer(synth.K3, seed=41, act="bf16h")
    check_layer(L, 1024, sample=[0, 3, 511, 800, 1023])


def test_layer_bf16h_k3_decode_b64_zipf():
    """Decode b=64 with Zipf-skewed routing at the K3 shape in the bf16-class h mode, as the bench
    times it: indices and gates of all 64 tokens, y of every fourth."""
    L = DeviceLayer(synth.K3, seed=2, zipf_s=1.1, act="bf16h")
    check_layer(L, 64, sample=list(range(0, 64, 4)))


def test_layer_bf16h_k3_prefill_4096_sampled():
    """Prefill 4096 at the K3 shape in the bf16-class h mode, as the bench times it: indices and gates
    of all 4096 tokens, y of five."""
    L = DeviceLayer(synth.K3, seed=3, act="bf16h")
    check_layer(L, 4096, sample=[0, 1, 777, 2048, 4095])


def test_expert_ffn_bf16h_given_routing():
    L = DeviceLayer(MID, seed=42, x_dtype="f32", act="bf16h")
    T = 300
    xh, xd = L.tokens(T)
    rng = np.random.default_rng(4)
    idx = np.stack([rng.choice(MID.n_routed, MID.top_k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, MID.top_k)).astype(np.float32)
    y = torch.empty((T, MID.d_model), dtype=torch.float32, device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.expert_ffn(L.cfg, xd, T, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), L.routed, L.shared, y, ws)
    assert k3.check_device_status(ws) == k3.OK
    assert rel_err(y.cpu().numpy(), L.oracle_ffn(xh, idx, w)) <= REL_TOL


# ------------------------------------------------------------------ separate entry points


@pytest.mark.parametrize("T,tol", [(5, 1e-6), (29, GATE_TOL)])
def test_route_only(T, tol):
    """Below 16 tokens the logits are fp32 dot products on the CUDA cores (gates to 1e-6); from 16 on
    they come from the tensor cores as partial sums over parts of d (gates to GATE_TOL, as below)."""
    L = DeviceLayer(MID, seed=10, zipf_s=1.1)
    xh, xd = L.tokens(T)
    idx = torch.empty((T, MID.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, MID.top_k), dtype=torch.float32, device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.route(L.cfg, xd, T, L.W, L.bias, idx, w, ws)
    torch.cuda.synchronize()
    _, idx_ref, w_ref, logits_ref = L.oracle(xh)
    ok, near, msg = index_parity(idx.cpu().numpy(), idx_ref, logits_ref, MID.top_k)
    assert ok, msg
    wn = w.cpu().numpy()
    assert np.allclose(wn.sum(axis=1), 1.0, atol=1e-6)
    keep = [t for t in range(T) if t not in near]
    assert gate_err(idx.cpu().numpy()[keep], wn[keep], idx_ref[keep], w_ref[keep]) < tol


@pytest.mark.parametrize("T,tol", [(5, 1e-6), (29, GATE_TOL)])
def test_route_sigmoid_bias(T, tol):
    """Sigmoid score with a selection-only bias (of the size of the sigmoid's spread, so that it
    reorders the selection): same selection as the oracle (near-tie rule on sigmoid + bias) and gates
    from the unbiased sigmoid; CUDA-core logits at 5 tokens, tensor-core partial logits at 29."""
    L = DeviceLayer(MID, seed=16, zipf_s=0.05, score="sigmoid_bias")
    xh, xd = L.tokens(T)
    idx = torch.empty((T, MID.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, MID.top_k), dtype=torch.float32, device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.route(L.cfg, xd, T, L.W, L.bias, idx, w, ws)
    torch.cuda.synchronize()
    assert k3.check_device_status(ws) == k3.OK
    _, idx_ref, w_ref, logits_ref = L.oracle(xh)
    ok, near, msg = index_parity(idx.cpu().numpy(), idx_ref, L.sel_keys(logits_ref), MID.top_k)
    assert ok, msg
    wn = w.cpu().numpy()
    assert np.allclose(wn.sum(axis=1), 1.0, atol=1e-6)
    keep = [t for t in range(T) if t not in near]
    assert gate_err(idx.cpu().numpy()[keep], wn[keep], idx_ref[keep], w_ref[keep]) < tol


@pytest.mark.parametrize("T", [3, 20])
def test_layer_sigmoid_bias(T):
    L = DeviceLayer(MID, seed=17, zipf_s=0.05, score="sigmoid_bias")
    check_layer(L, T)


@pytest.mark.parametrize("T,x_dtype", [(16, "bf16"), (40, "f32"), (512, "bf16"), (700, "bf16"), (600, "f32"), (1100, "bf16")])
def test_route_tensor_core_router(T, x_dtype):
    """From 16 tokens the logits come from the tensor cores (the fp32 router weights, and fp32 tokens,
    in three bf16 parts; fp32 accumulation; below ~600 tokens as partial sums over parts of d): same
    selection (near-tie rule) and gates as the oracle."""
    L = DeviceLayer(MID, seed=12, zipf_s=1.1, x_dtype=x_dtype)
    xh, xd = L.tokens(T)
    idx = torch.empty((T, MID.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, MID.top_k), dtype=torch.float32, device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.route(L.cfg, xd, T, L.W, L.bias, idx, w, ws)
    torch.cuda.synchronize()
    assert k3.check_device_status(ws) == k3.OK
    _, idx_ref, w_ref, logits_ref = L.oracle(xh)
    ok, near, msg = index_parity(idx.cpu().numpy(), idx_ref, logits_ref, MID.top_k)
    assert ok, msg
    wn = w.cpu().numpy()
    keep = [t for t in range(T) if t not in near]
    assert np.allclose(wn.sum(axis=1), 1.0, atol=1e-6)
    assert gate_err(idx.cpu().numpy()[keep], wn[keep], idx_ref[keep], w_ref[keep]) < GATE_TOL


def test_layer_mid_large_T_sampled():
    """The whole layer at 700 tokens: tensor-core router, E4M3 activation terms."""
    L = DeviceLayer(MID, seed=13)
    check_layer(L, 700, sample=[0, 5, 333, 512, 699])


def test_layer_mid_1100_tokens_sampled():
    """From 1024 tokens each token's selecting CTA also forms its activation terms."""
    L = DeviceLayer(MID, seed=15)
    check_layer(L, 1100, sample=[0, 1, 640, 1023, 1099])


def test_expert_ffn_given_routing():
    L = DeviceLayer(MID, seed=11, x_dtype="f32")
    T = 13
    xh, xd = L.tokens(T)
    rng = np.random.default_rng(0)
    idx = np.stack([rng.choice(MID.n_routed, MID.top_k, replace=False) for _ in range(T)]).astype(np.int32)
    idx[3, :] = np.arange(MID.top_k)  # overlapping expert sets
    w = rng.random((T, MID.top_k)).astype(np.float32)
    y = torch.empty((T, MID.d_model), dtype=torch.float32, device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.expert_ffn(L.cfg, xd, T, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), L.routed, L.shared, y, ws)
    assert k3.check_device_status(ws) == k3.OK
    y_ref = L.oracle_ffn(xh, idx, w)
    assert rel_err(y.cpu().numpy(), y_ref) <= REL_TOL


@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
def test_expert_ffn_given_routing_position_ordered_x(x_dtype):
    """From 256 tokens the gate/up projection reads x's terms in position order (gathered once per
    call, one tensor copy per work group and chunk); routed slots with overlapping expert sets and a
    ragged tail of tokens."""
    L = DeviceLayer(MID, seed=16, x_dtype=x_dtype)
    T = 301
    xh, xd = L.tokens(T)
    rng = np.random.default_rng(2)
    idx = np.stack([rng.choice(MID.n_routed, MID.top_k, replace=False) for _ in range(T)]).astype(np.int32)
    idx[7, :] = np.arange(MID.top_k)
    idx[8, :] = np.arange(MID.top_k)
    w = rng.random((T, MID.top_k)).astype(np.float32)
    y = torch.empty((T, MID.d_model), dtype=torch.float32, device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.expert_ffn(L.cfg, xd, T, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), L.routed, L.shared, y, ws)
    assert k3.check_device_status(ws) == k3.OK
    assert rel_err(y.cpu().numpy(), L.oracle_ffn(xh, idx, w)) <= REL_TOL


def test_bad_expert_id_with_position_ordered_x():
    """A rejected slot leaves a hole in the routed positions; the gather skips it and the layer still
    reports the bad id."""
    L = DeviceLayer(MID, seed=17)
    T = 260
    _, xd = L.tokens(T)
    rng = np.random.default_rng(3)
    idx = np.stack([rng.choice(MID.n_routed, MID.top_k, replace=False) for _ in range(T)]).astype(np.int32)
    idx[100, 2] = 999
    w = torch.full((T, MID.top_k), 1.0 / MID.top_k, device="cuda")
    y = torch.empty((T, MID.d_model), device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.expert_ffn(L.cfg, xd, T, torch.from_numpy(idx).cuda(), w, L.routed, L.shared, y, ws)
    assert k3.check_device_status(ws) == k3.ERR_DEVICE_CHECK
    assert k3.check_device_status(ws) == k3.OK


def test_zero_tokens_is_noop():
    L = DeviceLayer(MID, seed=12)
    y = torch.full((1, MID.d_model), 7.0, device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, 1), dtype=torch.uint8, device="cuda")
    _, xd = L.tokens(1)
    k3.layer(L.cfg, xd, 0, L.W, L.bias, L.routed, L.shared, y, ws)
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


def test_repeatable_and_batch_invariant():
    L = DeviceLayer(MID, seed=13)
    xh, xd = L.tokens(9)
    y1, i1, _ = run_layer(L, xd, 9)
    y2, i2, _ = run_layer(L, xd, 9)
    assert np.array_equal(i1, i2) and np.array_equal(y1, y2)
    # one token alone takes the E2M1-term form (error ~1e-7 of max|y|), nine tokens the E4M3-term form
    # (~2e-5): the same token agrees to within those bounds, not bit for bit
    y3, i3, _ = run_layer(L, xd[4:5].contiguous(), 1)
    assert np.array_equal(i3[0], i1[4])
    assert rel_err(y3[0], y1[4]) < 5e-5
    # within one form (three and nine tokens, E4M3 terms) only the accumulation order differs
    y4, i4, _ = run_layer(L, xd[2:5].contiguous(), 3)
    assert np.array_equal(i4[2], i1[4])
    assert rel_err(y4[2], y1[4]) < 1e-6


# ------------------------------------------------------------------ device-side data checks


def test_bad_expert_id_sets_device_status():
    L = DeviceLayer(MID, seed=14)
    T = 3
    _, xd = L.tokens(T)
    idx = torch.tensor([[0, 1, 2, 3, 4, 5], [6, 7, 8, 9, 10, 999], [1, 2, 3, 4, 5, 6]], dtype=torch.int32,
                       device="cuda")
    w = torch.full((T, MID.top_k), 1.0 / MID.top_k, device="cuda")
    y = torch.empty((T, MID.d_model), device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.expert_ffn(L.cfg, xd, T, idx, w, L.routed, L.shared, y, ws)
    assert k3.check_device_status(ws) == k3.ERR_DEVICE_CHECK
    assert k3.check_device_status(ws) == k3.OK  # the check clears the word


def test_nan_scale_byte_sets_device_status():
    L = DeviceLayer(MID, seed=15)
    T = 2
    xh, xd = L.tokens(T)
    _, idx_ref, _, _ = L.oracle(xh)
    e = int(idx_ref[0, 0])
    nc = MID.d_model * MID.d_ff // 2
    L.routed[e * L.stride + nc + 3] = 255  # one gate scale byte of a selected expert
    y = torch.empty((T, MID.d_model), device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.layer(L.cfg, xd, T, L.W, L.bias, L.routed, L.shared, y, ws)
    assert k3.check_device_status(ws) == k3.ERR_DEVICE_CHECK


def test_workspace_too_small_is_rejected():
    L = DeviceLayer(MID, seed=16)
    _, xd = L.tokens(4)
    y = torch.empty((4, MID.d_model), device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, 2), dtype=torch.uint8, device="cuda")
    with pytest.raises(k3.K3moeError) as ei:
        k3.layer(L.cfg, xd, 4, L.W, L.bias, L.routed, L.shared, y, ws)
    assert ei.value.code == k3.ERR_WORKSPACE


# ------------------------------------------------------------------ stack harness (pre-norm residual)


def test_stack_prenorm_residual_teacher_forced():
    """x_{l+1} = x_l + Layer_l(RMSNorm(x_l)), each layer checked on the GPU's own layer input. The first
    norm is k3moe_rmsnorm; between layers k3moe_residual_rmsnorm adds the layer output and forms the
    next layer's normalised input in one kernel (its residual sum is checked as well)."""
    import oracle
    sh = MID
    T = 7
    layers = [DeviceLayer(sh, seed=40 + l, layer=l, zipf_s=1.1, x_dtype="f32") for l in range(4)]
    x0 = synth.tokens(sh, 40, T, "f32")
    x = torch.from_numpy(x0).cuda()
    xn = torch.empty_like(x)
    y = torch.empty_like(x)
    ws = torch.zeros(k3.workspace_bytes(layers[0].cfg, T), dtype=torch.uint8, device="cuda")
    k3.rmsnorm(x, T, sh.d_model, 1e-6, xn)
    for l, L in enumerate(layers):
        torch.cuda.synchronize()
        xin = x.cpu().numpy().astype(np.float64)
        xn_h = xn.cpu().numpy()
        assert np.allclose(xn_h, oracle.rmsnorm(xin, 1e-6), rtol=2e-6, atol=1e-6)
        k3.layer(L.cfg, xn, T, L.W, L.bias, L.routed, L.shared, y, ws)
        torch.cuda.synchronize()
        y_ref, idx_ref, _, logits_ref = L.oracle(xn_h)
        err = rel_err(y.cpu().numpy(), y_ref)
        assert err <= REL_TOL, err
        y_h = y.cpu().numpy()
        k3.residual_rmsnorm(x, y, T, sh.d_model, 1e-6, xn)
        torch.cuda.synchronize()
        assert np.array_equal(x.cpu().numpy(), (xin.astype(np.float32) + y_h))  # fp32 adds, exactly
    assert torch.isfinite(x).all()


def test_prepared_router_parts_match_per_call_split():
    """k3moe_prepare_router at weight loading gives the tensor-core router the same bf16 parts as the
    per-call split: the same selection and bit-identical gates (29 tokens: tensor-core logits)."""
    L = DeviceLayer(MID, seed=18, zipf_s=1.1)
    T = 29
    _, xd = L.tokens(T)
    parts = torch.empty(k3.router_parts_bytes(L.cfg) // 2, dtype=torch.int16, device="cuda")
    k3.prepare_router(L.cfg, L.W, parts)
    outs = []
    for wp in (None, parts):
        idx = torch.empty((T, MID.top_k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, MID.top_k), dtype=torch.float32, device="cuda")
        ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
        k3.route(L.cfg, xd, T, L.W, L.bias, idx, w, ws, w_parts=wp)
        torch.cuda.synchronize()
        outs.append((idx.cpu().numpy(), w.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    # the parts add up to the fp32 weights exactly
    p = parts.view(torch.bfloat16).float().reshape(3, MID.n_routed, MID.d_model)
    assert torch.equal(p[0] + p[1] + p[2], L.W)


@pytest.mark.parametrize("T", [5, 20])
def test_bounded_wait_runs_out_and_context_stays_usable(T):
    """With a bound of one poll the first unsatisfied pipeline wait gives up: the kernels report
    K3MOE_ERR_TIMEOUT through the status word, let their copies and MMAs finish, free their tensor
    memory and exit. A normal call on the same context afterwards is correct. (5 tokens: the expert
    kernels time out; 20 tokens: the tensor-core router's GEMM as well.)"""
    L = DeviceLayer(MID, seed=19)
    xh, xd = L.tokens(T)
    y = torch.empty((T, MID.d_model), dtype=torch.float32, device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    assert k3.layer_bounded(L.cfg, xd, T, L.W, L.bias, L.routed, L.shared, y, ws, 1) == k3.OK
    assert k3.check_device_status(ws) == k3.ERR_TIMEOUT
    assert k3.check_device_status(ws) == k3.OK  # read and cleared
    # a generous bound behaves like k3moe_layer
    assert k3.layer_bounded(L.cfg, xd, T, L.W, L.bias, L.routed, L.shared, y, ws, 1 << 24) == k3.OK
    assert k3.check_device_status(ws) == k3.OK
    check_layer(L, T)
