"""The router's index contract on the GPU, case by case, through both logit paths (fp32 dot products on
the CUDA cores below 16 tokens, the tensor-core GEMM from 16 tokens on):

* exact ties (duplicated router rows give bit-equal logits on both sides): the lower expert id comes
  first, inside the selection and across the k-th place, with no near-tie excuse;
* a token whose logits are all equal (x = 0): experts 0 .. k-1, gates 1/k, and y = 0 exactly;
* the sigmoid score with a selection-only bias on the six-row fixture in which the bias swaps the
  top two experts in five rows (kimi-k3-in-c review, list of public-header invariants: the routing
  bias skews only the selection, the combine weights come from the unbiased sigmoid score).
"""
import numpy as np
import pytest

import synth
from harness import REL_TOL, DeviceLayer, gate_err, index_parity, oracle_order, rel_err, GATE_TOL

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU machine
    pytest.skip("needs a GPU", allow_module_level=True)

import mxfp4_routed_expert_k3moe_gb300 as k3  # noqa: E402

MID = synth.LayerShape(d_model=512, d_ff=256, n_routed=64, top_k=6, n_shared=2)
SHAPES = {"MID": MID, "K3": synth.K3}


def route(L: DeviceLayer, xd, T):
    sh = L.shape
    idx = torch.empty((T, sh.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, sh.top_k), dtype=torch.float32, device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.route(L.cfg, xd, T, L.W, L.bias, idx, w, ws)
    assert k3.check_device_status(ws) == k3.OK
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def layer(L: DeviceLayer, xd, T):
    sh = L.shape
    y = torch.empty((T, sh.d_model), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, sh.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, sh.top_k), dtype=torch.float32, device="cuda")
    ws = torch.zeros(k3.workspace_bytes(L.cfg, T), dtype=torch.uint8, device="cuda")
    k3.layer(L.cfg, xd, T, L.W, L.bias, L.routed, L.shared, y, ws, idx, w)
    assert k3.check_device_status(ws) == k3.OK
    torch.cuda.synchronize()
    return y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def copy_router_row(L: DeviceLayer, dst: int, src: int):
    """Router row dst := row src, on the host copy (oracle) and on the device."""
    L.W_host[dst] = L.W_host[src]
    L.W[dst].copy_(L.W[src])


@pytest.mark.parametrize("shape,T", [("MID", 5), ("MID", 29), ("K3", 1), ("K3", 20)])
def test_exact_ties_lower_id_first(shape, T):
    """Duplicated router rows: a tie across the k-th place (one copy in, one out), a tie inside the
    selection and a three-way tie. Built around token 0's ranking; the other tokens get the same ties
    at other ranks. Every token must follow the lower-id rule exactly."""
    sh = SHAPES[shape]
    L = DeviceLayer(sh, seed=31, pack=False)
    k = sh.top_k
    xh, xd = L.tokens(T)
    lg, _, _ = L.oracle_route(xh[:1])
    order = [int(e) for e in oracle_order(lg[0])]
    # c, token 0's 2nd expert, is duplicated to two unselected ones (d1, d2), which moves token 0's
    # experts from the 3rd on down two places: a, its (k-2)-th, becomes the k-th and is duplicated to
    # an unselected b, so that one of a, b is selected and the other is not
    c, d1, d2 = order[1], order[k + 1], order[k + 2]
    a = order[k - 3]
    b = order[k + 3]
    copy_router_row(L, b, a)
    copy_router_row(L, d1, c)
    copy_router_row(L, d2, c)
    torch.cuda.synchronize()
    lg_all, idx_ref, w_ref = L.oracle_route(xh)
    assert lg_all[0, a] == lg_all[0, b] and lg_all[0, c] == lg_all[0, d1] == lg_all[0, d2]
    assert (min(a, b) in idx_ref[0]) and (max(a, b) not in idx_ref[0])
    assert all(e in idx_ref[0] for e in (c, d1, d2))
    idx, w = route(L, xd, T)
    ok, near, msg = index_parity(idx, idx_ref, lg_all, k)
    assert ok, msg
    # the tied selections of token 0 are exact: ranks of c, d1, d2 in ascending id, the lower of a, b in
    assert idx[0].tolist() == idx_ref[0].tolist()
    keep = [t for t in range(T) if t not in near]
    assert gate_err(idx[keep], w[keep], idx_ref[keep], w_ref[keep]) < GATE_TOL
    # tied experts get equal gates, bit for bit
    pos = {int(e): i for i, e in enumerate(idx[0])}
    assert w[0, pos[c]] == w[0, pos[d1]] == w[0, pos[d2]]


@pytest.mark.parametrize("T", [3, 20])
def test_zero_token_all_logits_equal(T):
    """x = 0 for tokens 0 and T-1: every logit is 0, so the selection is experts 0 .. k-1 (lower id
    first) with gates 1/k, and y = 0 exactly (SiLU(0) * 0 = 0 in every expert). The other tokens are
    checked against the oracle as usual."""
    L = DeviceLayer(MID, seed=32)
    k = MID.top_k
    xh, _ = L.tokens(T)
    xh = xh.copy()
    xh[0] = 0
    xh[T - 1] = 0x8000  # -0.0 in bf16: products of either sign of zero
    xd = torch.from_numpy(xh.view(np.int16)).cuda()
    y, idx, w = layer(L, xd, T)
    for t in (0, T - 1):
        assert idx[t].tolist() == list(range(k))
        assert np.all(w[t] == np.float32(1.0 / k))
        assert np.all(y[t] == 0.0)
    rows = list(range(1, min(T - 1, 4)))
    y_ref, idx_ref, w_ref, logits_ref = L.oracle(xh, rows)
    ok, near, msg = index_parity(idx[rows], idx_ref, logits_ref, k)
    assert ok, msg
    keep = [i for i in range(len(rows)) if i not in near]
    assert rel_err(y[rows][keep], y_ref[keep]) <= REL_TOL


# The six-row fixture of the sigmoid score (also pinned on the oracle in test_oracle.py): per row the
# logits of six experts and the selection bias; top-2. In rows 0-4 the bias swaps the unbiased top two,
# in row 5 it pulls expert 4 into the selection.
FIXTURE = [
    ([2.0, 1.75, 0.5, -0.25, -1.0, 0.0], [0.0, 0.25, 0.0, 0.0, 0.0, 0.0]),
    ([0.5, 1.0, -2.0, 3.0, 2.5, 0.0], [0.0, 0.0, 0.0, 0.0, 0.125, 0.0]),
    ([-1.0, -0.5, -0.75, -2.0, -3.0, -0.25], [0.0, 0.5, 0.0, 0.0, 0.0, 0.0]),
    ([4.0, 3.5, 0.0, 0.0, 0.0, 0.0], [0.0, 0.0625, 0.0, 0.0, 0.0, 0.0]),
    ([0.0, 0.0, 0.0, 1.0, 0.875, 0.0], [0.0, 0.0, 0.0, 0.0, 0.5, 0.0]),
    ([2.0, 1.75, 0.5, -0.25, -1.0, 0.0], [0.0, 0.0, 0.0, 0.0, 1.0, 0.0]),
]


def _brute_topk(keys, k):
    """Expert e is selected iff fewer than k experts beat it (larger value, or equal value and lower id)."""
    n = len(keys)
    sel = []
    for e in range(n):
        beaten = sum(1 for j in range(n) if keys[j] > keys[e] or (keys[j] == keys[e] and j < e))
        if beaten < k:
            sel.append((beaten, e))
    return [e for _, e in sorted(sel)]


@pytest.mark.parametrize("T", [1, 16])
def test_sigmoid_fixture_bias_swaps_top_two(T):
    """Each fixture row as a router of 6 experts over d_model 128 whose logits are the row exactly
    (W = the row on the diagonal, x = ones: one nonzero product per logit, exact in fp32 and in the
    bf16 parts of the tensor-core path). T copies of the token: 1 takes the CUDA-core logits, 16 the
    tensor-core ones. Selection = brute-force ranking of sigmoid + bias (scipy's expit); gates = the
    unbiased sigmoid renormalised; the bias swaps the top two in exactly five rows."""
    from scipy.special import expit
    sh = synth.LayerShape(d_model=128, d_ff=128, n_routed=6, top_k=2, n_shared=0)
    L = DeviceLayer(sh, seed=33, score="sigmoid_bias", pack=False)
    swapped = 0
    x = torch.full((T, sh.d_model), 1.0, dtype=torch.bfloat16, device="cuda").view(torch.int16)
    for logits, bias in FIXTURE:
        W = np.zeros((6, sh.d_model), np.float32)
        W[np.arange(6), np.arange(6)] = np.asarray(logits, np.float32)
        L.W.copy_(torch.from_numpy(W))
        s = expit(np.asarray(logits, np.float64))
        keys = s + np.asarray(bias, np.float64)
        want = _brute_topk(list(keys), 2)
        unbiased = _brute_topk(list(s), 2)
        for b in (bias, None):
            L.bias = None if b is None else torch.tensor(b, dtype=torch.float32, device="cuda")
            idx, w = route(L, x, T)
            exp_idx = want if b is not None else unbiased
            for t in range(T):
                assert idx[t].tolist() == exp_idx, (logits, b, idx[t])
                assert np.allclose(w[t], s[exp_idx] / s[exp_idx].sum(), rtol=5e-6, atol=0)
        swapped += int(want == unbiased[::-1])
    assert swapped == 5
