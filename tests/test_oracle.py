"""Pins of the CPU oracle against what the pages and the mathematics fix (CPU only).

Each pin is a function that raises AssertionError when the oracle is wrong.
`test_planted_mistakes_are_caught` switches the oracle to deliberately wrong
variants and checks that at least one pin fails for each: wrong nibble order, scale
bias, a wrong E2M1 table entry, the next block's scale byte, dropped shared
experts, shared experts weighted by a gate, missing renormalisation, a
renormalising sum short of one gate, wrong tie order, the lowest logits
selected, transposed down projection, SiLU on the wrong branch, SiLU with the
wrong sign, RMSNorm over the sum of squares, and for the sigmoid score: the bias
in the gates, the bias left out of the selection.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from conftest import read_golden

# ----------------------------------------------------------------------------- helpers


def _e2m1_table():
    g = read_golden("ocp_e2m1.txt")
    return {int(k): float(v) for k, v in g.items()}


def _pack_codes(nibbles: np.ndarray) -> np.ndarray:
    """[rows, cols] 4-bit codes -> [rows, cols/2] bytes, even column in the low nibble (record format)."""
    nib = np.asarray(nibbles, dtype=np.uint8)
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)


def _make_record(gate, up, down, gate_s, up_s, down_s):
    """Assemble a record from nibble matrices and scale-byte matrices."""
    parts = []
    for codes, sc in ((gate, gate_s), (up, up_s), (down, down_s)):
        parts.append(_pack_codes(codes).ravel())
        parts.append(np.asarray(sc, dtype=np.uint8).ravel())
    return np.concatenate(parts)


def _silu(z):
    return z / (1.0 + np.exp(-z))


# ----------------------------------------------------------------------------- pins: formats


def pin_e2m1_table():
    tab = _e2m1_table()
    assert len(tab) == 16
    for code, val in tab.items():
        got = oracle.e2m1(code)
        assert got == val, (code, got, val)
        assert math.copysign(1.0, got) == math.copysign(1.0, val), code  # code 8 is -0.0


def pin_e8m0():
    assert oracle.e8m0(127) == 1.0
    assert oracle.e8m0(128) == 2.0
    assert oracle.e8m0(126) == 0.5
    assert oracle.e8m0(0) == 2.0 ** -127
    assert oracle.e8m0(254) == 2.0 ** 127
    with pytest.raises(ValueError):
        oracle.e8m0(255)


def pin_record_bytes():
    g = read_golden("shard_census.txt")
    params = int(g["params_per_expert"])
    # the census factors as three 7168 x 1536 matrices (gate, up, down)
    assert 3 * 7168 * 1536 == params
    assert oracle.record_bytes(7168, 1536) == int(g["bytes_per_expert"])
    assert params * float(g["bytes_per_weight"]) == int(g["bytes_per_expert"])
    assert int(g["moe_layers"]) * int(g["routed_experts_per_layer"]) == int(g["routed_experts_total"])
    tb = int(g["routed_experts_total"]) * int(g["bytes_per_expert"]) / 1e12
    # the census prints 1.447 TB for 1,446,456,066,048 B (its rounding), so compare to 1e-3 TB
    assert abs(tb - float(g["routed_expert_set_tb"])) < 1e-3
    assert oracle.record_bytes(256, 128) == 52224  # the tiny workload's record
    assert synth.K3.record_bytes == oracle.record_bytes(7168, 1536)


def pin_decode_single_nonzero():
    """One non-zero nibble at (r, c): the decoded matrix is zero except at (r, c) (layout and nibble order)."""
    rows, cols = 3, 96
    tab = _e2m1_table()
    for (r, c, code, sb) in [(0, 0, 7, 127), (0, 1, 5, 130), (1, 2, 9, 120), (2, 33, 15, 127), (2, 95, 3, 200),
                             (1, 64, 2, 0)]:
        nib = np.zeros((rows, cols), np.uint8)
        nib[r, c] = code
        sc = np.full((rows, cols // 32), 127, np.uint8)
        sc[r, c // 32] = sb
        dense = oracle.decode_matrix(_pack_codes(nib), sc, rows, cols)
        want = np.zeros((rows, cols))
        want[r, c] = tab[code] * 2.0 ** (sb - 127)
        assert np.array_equal(dense, want), (r, c)


def pin_decode_block_scale_axis():
    """A scale byte covers 32 consecutive columns of its row and nothing else."""
    rows, cols = 2, 128
    nib = np.full((rows, cols), 2, np.uint8)  # all 1.0
    sc = np.full((rows, cols // 32), 127, np.uint8)
    sc[1, 2] = 129  # x4 for row 1, columns 64..95
    dense = oracle.decode_matrix(_pack_codes(nib), sc, rows, cols)
    want = np.ones((rows, cols))
    want[1, 64:96] = 4.0
    assert np.array_equal(dense, want)


# ----------------------------------------------------------------------------- pins: router


def _brute_topk(logits, k):
    """Select e iff fewer than k experts beat it (higher logit, or equal logit and lower index)."""
    E = len(logits)
    sel = []
    for e in range(E):
        beaten_by = sum(1 for j in range(E) if logits[j] > logits[e] or (logits[j] == logits[e] and j < e))
        if beaten_by < k:
            sel.append((beaten_by, e))
    return [e for _, e in sorted(sel)]


def pin_router_bruteforce():
    rng = np.random.default_rng(11)
    for E, d, k in [(8, 16, 3), (32, 64, 4), (40, 32, 7)]:
        x = rng.standard_normal(d)
        W = (rng.standard_normal((E, d)) / math.sqrt(d)).astype(np.float32)
        bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
        for b in (None, bias):
            logits, idx, w = oracle.route_token(x, W, k, b)
            ref_logits = W.astype(np.float64) @ x + (0.0 if b is None else b.astype(np.float64))
            assert np.allclose(logits, ref_logits, rtol=0, atol=1e-12)
            assert list(idx) == _brute_topk(list(logits), k)
            assert len(set(idx.tolist())) == k
            # renormalised gates = softmax restricted to the k selected logits
            ex = np.exp(logits[idx] - logits[idx].max())
            assert np.allclose(w, ex / ex.sum(), rtol=1e-13, atol=0)
            assert abs(w.sum() - 1.0) < 1e-12
            assert np.all(np.diff(w) <= 0)


def pin_router_ties_lower_index():
    d = 16
    rng = np.random.default_rng(5)
    base = rng.standard_normal(d).astype(np.float32)
    W = np.stack([base * 0.5, base, base * 0.25, base, base, base * -1.0]).astype(np.float32)
    x = base.astype(np.float64)
    _, idx, w = oracle.route_token(x, W, 3)
    assert list(idx) == [1, 3, 4]  # three equal top logits: ascending index
    assert np.allclose(w, 1.0 / 3.0, rtol=1e-14)


def pin_router_counts_k3_shape():
    """Full-size router: exactly 16 distinct routed experts per token; 16 x 92 = 1472 per token."""
    g = read_golden("shard_census.txt")
    sh = synth.K3
    W = synth.router_weights(sh, seed=1)
    x = synth.tokens_as_f64(synth.tokens(sh, 1, 1, "bf16"), "bf16")[0]
    logits, idx, w = oracle.route_token(x, W, sh.top_k)
    assert sh.top_k == int(g["top_k"]) and sh.n_shared == int(g["shared_experts"])
    assert len(set(idx.tolist())) == sh.top_k and idx.min() >= 0 and idx.max() < sh.n_routed
    assert sh.top_k * int(g["moe_layers"]) == int(g["expert_evaluations_per_token"])
    assert abs(w.sum() - 1.0) < 1e-12
    order = np.argsort(-logits, kind="stable")[: sh.top_k]
    assert list(order) == list(idx)


def _diag_router(logit_rows):
    """Router weights whose logits are the given values exactly: W = diag(l), x = ones (all values are
    exact in fp32)."""
    l = np.asarray(logit_rows, dtype=np.float32)
    return np.diag(l).astype(np.float32), np.ones(len(l))


def pin_router_sigmoid_bias_selection_only():
    """Sigmoid score (review, list of public-header invariants): the routing bias changes only which
    experts are selected; the gates are the unbiased sigmoid scores renormalised over the selection.
    Six rows; in five of them a bias swaps the order of the top two (checked against scipy's expit
    and brute-force ranking), in the sixth it pulls a low expert into the selection."""
    from scipy.special import expit
    k = 2
    rows = [
        ([2.0, 1.75, 0.5, -0.25, -1.0, 0.0], [0.0, 0.25, 0.0, 0.0, 0.0, 0.0]),
        ([0.5, 1.0, -2.0, 3.0, 2.5, 0.0], [0.0, 0.0, 0.0, 0.0, 0.125, 0.0]),
        ([-1.0, -0.5, -0.75, -2.0, -3.0, -0.25], [0.0, 0.5, 0.0, 0.0, 0.0, 0.0]),
        ([4.0, 3.5, 0.0, 0.0, 0.0, 0.0], [0.0, 0.0625, 0.0, 0.0, 0.0, 0.0]),
        ([0.0, 0.0, 0.0, 1.0, 0.875, 0.0], [0.0, 0.0, 0.0, 0.0, 0.5, 0.0]),
        ([2.0, 1.75, 0.5, -0.25, -1.0, 0.0], [0.0, 0.0, 0.0, 0.0, 1.0, 0.0]),
    ]
    swapped = 0
    for l, b in rows:
        W, x = _diag_router(l)
        b = np.asarray(b, dtype=np.float32)
        s = expit(np.asarray(l, dtype=np.float64))
        keys = s + b.astype(np.float64)
        logits, idx, w = oracle.route_token(x, W, k, b, score="sigmoid_bias")
        assert np.array_equal(logits, np.asarray(l, dtype=np.float64))  # no bias in the logits
        assert list(idx) == _brute_topk(list(keys), k)
        assert np.allclose(w, s[idx] / s[idx].sum(), rtol=1e-14, atol=0)
        _, idx0, w0 = oracle.route_token(x, W, k, None, score="sigmoid_bias")
        assert list(idx0) == _brute_topk(list(s), k)
        swapped += int(list(idx) == list(idx0[::-1]))
        # a constant added to every bias changes nothing
        _, idx1, w1 = oracle.route_token(x, W, k, b + np.float32(0.5), score="sigmoid_bias")
        assert list(idx1) == list(idx) and np.allclose(w1, w, rtol=1e-15, atol=0)
    assert swapped == 5


def pin_router_sigmoid_unbiased_matches_softmax_selection():
    """Without a bias the sigmoid is monotone in the logit: the same experts, in the same order, as the
    softmax score selects (ties to the lower index in both)."""
    rng = np.random.default_rng(12)
    for E, d, k in [(8, 16, 3), (40, 32, 7)]:
        x = rng.standard_normal(d)
        W = (rng.standard_normal((E, d)) / math.sqrt(d)).astype(np.float32)
        _, idx_s, _ = oracle.route_token(x, W, k, None, score="softmax")
        _, idx_g, w_g = oracle.route_token(x, W, k, None, score="sigmoid_bias")
        assert list(idx_s) == list(idx_g)
        assert abs(w_g.sum() - 1.0) < 1e-12 and np.all(np.diff(w_g) <= 0)


# ----------------------------------------------------------------------------- pins: expert FFN


def _numpy_expert(record, x, d, f):
    """Second code path: dense dequantisation with numpy + numpy matmuls (no nibble loop)."""
    tab = np.array([_e2m1_table()[c] for c in range(16)])
    outs = []
    off = 0
    for rows, cols in ((f, d), (f, d), (d, f)):
        nc, ns = rows * cols // 2, rows * cols // 32
        codes = record[off:off + nc].reshape(rows, cols // 2)
        scales = record[off + nc:off + nc + ns].reshape(rows, cols // 32).astype(np.int64)
        nib = np.empty((rows, cols), np.int64)
        nib[:, 0::2] = codes & 0xF
        nib[:, 1::2] = codes >> 4
        outs.append(tab[nib] * np.repeat(2.0 ** (scales - 127), 32, axis=1))
        off += nc + ns
    Wg, Wu, Wd = outs
    g = Wg @ x
    u = Wu @ x
    h = _silu(g) * u
    return Wd @ h, h


def pin_expert_vs_dense():
    rng = np.random.default_rng(3)
    for d, f in [(64, 32), (96, 64)]:
        sh = synth.LayerShape(d, f, 4, 2, 1)
        rec = synth.records_host(sh, seed=7, layer=0, experts=[2])[0]
        x = rng.standard_normal(d)
        o, h = oracle.expert_token(rec, x, d, f)
        o_ref, h_ref = _numpy_expert(rec, x, d, f)
        assert np.allclose(h, h_ref, rtol=1e-11, atol=1e-12 * np.abs(h_ref).max())
        assert np.allclose(o, o_ref, rtol=1e-10, atol=1e-11 * np.abs(o_ref).max())


def pin_expert_closed_form():
    """Permutation matrices: o_i = 2 * x_{p(s(i))}... written out as a closed form."""
    d = f = 32
    rng = np.random.default_rng(9)
    pg = rng.permutation(f)  # gate row r picks column pg[r]
    pd = rng.permutation(d)  # down row i picks column pd[i]
    gate = np.zeros((f, d), np.uint8)
    gate[np.arange(f), pg] = 2  # 1.0
    up = np.zeros((f, d), np.uint8)
    up[np.arange(f), np.arange(d)] = 4  # 2.0 on the diagonal
    down = np.zeros((d, f), np.uint8)
    down[np.arange(d), pd] = 10  # -1.0
    s127 = np.full((f, 1), 127, np.uint8)
    down_s = np.full((d, 1), 128, np.uint8)  # x2
    rec = _make_record(gate, up, down, s127, s127, down_s)
    x = rng.standard_normal(d)
    o, h = oracle.expert_token(rec, x, d, f)
    h_want = _silu(x[pg]) * (2.0 * x)
    assert np.allclose(h, h_want, rtol=1e-15, atol=0)
    assert np.allclose(o, -2.0 * h_want[pd], rtol=1e-15, atol=0)


# ----------------------------------------------------------------------------- pins: layer


def _tiny_layer_inputs(seed=0, T=6):
    sh = synth.TINY
    W = synth.router_weights(sh, seed)
    x = synth.tokens(sh, seed, T, "f32")
    recs = synth.records_host(sh, seed, 0, range(sh.n_routed + sh.n_shared))
    return sh, W, x, list(recs[: sh.n_routed]), list(recs[sh.n_routed:])


def pin_layer_combine_definition():
    """y equals the gate-weighted sum of the selected experts plus the shared experts."""
    sh, W, x, routed, shared = _tiny_layer_inputs()
    y, idx, w, _ = oracle.layer(x, "f32", W, None, routed, shared, sh.d_model, sh.d_ff, sh.top_k)
    for t in range(x.shape[0]):
        xt = x[t].astype(np.float64)
        _, idx_t, w_t = oracle.route_token(xt, W, sh.top_k)
        assert list(idx_t) == list(idx[t])
        want = np.zeros(sh.d_model)
        for e, g in zip(idx_t, w_t):
            want += g * _numpy_expert(routed[e], xt, sh.d_model, sh.d_ff)[0]
        for r in shared:
            want += _numpy_expert(r, xt, sh.d_model, sh.d_ff)[0]
        assert np.allclose(y[t], want, rtol=1e-10, atol=1e-11 * np.abs(want).max())


def pin_layer_identical_experts():
    """All routed experts identical => y = expert(x) + shared(x), whatever the routing (sum of gates is 1)."""
    sh, W, x, routed, shared = _tiny_layer_inputs(seed=1, T=3)
    same = [routed[5]] * sh.n_routed
    y, _, _, _ = oracle.layer(x, "f32", W, None, same, shared, sh.d_model, sh.d_ff, sh.top_k)
    for t in range(x.shape[0]):
        xt = x[t].astype(np.float64)
        want = oracle.expert_token(routed[5], xt, sh.d_model, sh.d_ff)[0]
        want = want + oracle.expert_token(shared[0], xt, sh.d_model, sh.d_ff)[0]
        assert np.allclose(y[t], want, rtol=1e-12, atol=1e-13 * np.abs(want).max())


def pin_layer_relabel():
    """Relabelling experts together with the router rows gives the same y."""
    sh, W, x, routed, shared = _tiny_layer_inputs(seed=2, T=4)
    perm = np.random.default_rng(0).permutation(sh.n_routed)  # new id j holds old expert perm[j]
    y0, idx0, _, _ = oracle.layer(x, "f32", W, None, routed, shared, sh.d_model, sh.d_ff, sh.top_k)
    y1, idx1, _, _ = oracle.layer(x, "f32", W[perm], None, [routed[p] for p in perm], shared,
                                  sh.d_model, sh.d_ff, sh.top_k)
    assert np.array_equal(np.sort(perm[idx1], axis=1), np.sort(idx0, axis=1))
    assert np.allclose(y0, y1, rtol=1e-12, atol=1e-13 * np.abs(y0).max())


def pin_layer_token_independence():
    sh, W, x, routed, shared = _tiny_layer_inputs(seed=3, T=5)
    y, _, _, _ = oracle.layer(x, "f32", W, None, routed, shared, sh.d_model, sh.d_ff, sh.top_k)
    for t in (0, 3):
        yt, _, _, _ = oracle.layer(x[t:t + 1], "f32", W, None, routed, shared, sh.d_model, sh.d_ff, sh.top_k)
        assert np.array_equal(y[t], yt[0])


def pin_layer_zero_gate_branch():
    """Zero gate codes: SiLU(0) = 0 kills every routed contribution; only the shared expert remains."""
    sh, W, x, routed, shared = _tiny_layer_inputs(seed=4, T=2)
    nc = sh.d_model * sh.d_ff // 2
    dead = []
    for r in routed:
        r = r.copy()
        r[:nc] = 0
        dead.append(r)
    y, _, _, _ = oracle.layer(x, "f32", W, None, dead, shared, sh.d_model, sh.d_ff, sh.top_k)
    for t in range(2):
        want = oracle.expert_token(shared[0], x[t].astype(np.float64), sh.d_model, sh.d_ff)[0]
        assert np.array_equal(y[t], want)


def pin_layer_down_scale_linear():
    """+1 on every down-projection scale byte doubles y exactly (the down projection is linear)."""
    sh, W, x, routed, shared = _tiny_layer_inputs(seed=5, T=2)
    d, f = sh.d_model, sh.d_ff
    nc, ns = d * f // 2, d * f // 32
    off = 2 * (nc + ns) + nc

    def bump(r):
        r = r.copy()
        r[off:off + ns] += 1
        return r

    y0, _, _, _ = oracle.layer(x, "f32", W, None, routed, shared, d, f, sh.top_k)
    y1, _, _, _ = oracle.layer(x, "f32", W, None, [bump(r) for r in routed], [bump(r) for r in shared], d, f,
                               sh.top_k)
    assert np.array_equal(y1, 2.0 * y0)


def pin_bf16_input_exact():
    """bf16 inputs enter as their exact values."""
    bits = np.array([0x3F80, 0xC040, 0x0001, 0x7F7F], np.uint16)
    want = [1.0, -3.0, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127]
    for b, v in zip(bits, want):
        assert oracle.lib().k3o_bf16(int(b)) == v


def pin_rmsnorm():
    x = np.full((1, 64), 3.0)
    out = oracle.rmsnorm(x, eps=1e-6)
    assert np.allclose(out, 3.0 / math.sqrt(9.0 + 1e-6), rtol=1e-15)
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 128))
    out = oracle.rmsnorm(x, eps=0.0)
    assert np.allclose((out ** 2).mean(axis=1), 1.0, rtol=1e-13)


def pin_tolerance_budget():
    g = read_golden("tolerance_budget.txt")
    tol = float(g["coef"]) * math.sqrt(int(g["width"])) * float(g["factor"])
    assert f"{tol:.1e}" == g["printed_budget"]
    # the page's own measured error sits inside the budget, and the build's 2e-3 bar is looser
    assert float(g["printed_rel_err"]) < tol < 2e-3


# ----------------------------------------------------------------------------- pins: bf16 shared experts


def pin_shared_bf16_vs_dense():
    """bf16 shared expert (README parameter budget: non-routed parameters in bfloat16): the oracle's
    loop over bf16 bit patterns equals numpy's float conversion of the patterns and numpy matmuls."""
    sh = synth.LayerShape(d_model=64, d_ff=32, n_routed=4, top_k=2, n_shared=1)
    rec = synth.shared_records_bf16(sh, 5, 0, 1)[0]
    d, f = sh.d_model, sh.d_ff
    w = synth.bf16_bits_to_f32(rec[:3 * d * f]).astype(np.float64)
    Wg, Wu, Wd = w[:f * d].reshape(f, d), w[f * d:2 * f * d].reshape(f, d), w[2 * f * d:].reshape(d, f)
    x = np.random.default_rng(3).standard_normal(d)
    g, u = Wg @ x, Wu @ x
    h = _silu(g) * u
    o, h_or = oracle.expert_token_bf16(rec, x, d, f)
    assert np.allclose(h_or, h, rtol=1e-12, atol=1e-14)
    assert np.allclose(o, Wd @ h, rtol=1e-12, atol=1e-14)


def pin_shared_bf16_image_of_mxfp4_is_identical():
    """A bf16 shared record holding exactly the values of an MXFP4 record (E2M1 values times powers of
    two fit bf16's 8-bit significand) gives the same layer output, bit for bit, as the MXFP4 record."""
    sh = synth.LayerShape(d_model=64, d_ff=32, n_routed=8, top_k=2, n_shared=1)
    d, f = sh.d_model, sh.d_ff
    routed = list(synth.records_host(sh, 6, 0, range(sh.n_routed)))
    shared_mx = synth.records_host(sh, 6, 0, [sh.n_routed])[0]
    dense = [oracle.decode_matrix(c, sc, *dims) for (c, sc), dims in
             zip(oracle.split_record(shared_mx, d, f), [(f, d), (f, d), (d, f)])]
    flat = np.concatenate([m.ravel() for m in dense]).astype(np.float32)
    bits = synth.f32_to_bf16_bits(flat)
    assert np.array_equal(synth.bf16_bits_to_f32(bits).astype(np.float64), np.concatenate([m.ravel() for m in dense]))
    W = synth.router_weights(sh, 6)
    x = synth.tokens(sh, 6, 3, "f32")
    y_mx = oracle.layer(x, "f32", W, None, routed, [shared_mx], d, f, sh.top_k)[0]
    y_bf = oracle.layer(x, "f32", W, None, routed, [bits], d, f, sh.top_k, shared_format="bf16")[0]
    assert np.array_equal(y_mx, y_bf)


PINS = [pin_e2m1_table, pin_e8m0, pin_record_bytes, pin_decode_single_nonzero, pin_decode_block_scale_axis,
        pin_router_bruteforce, pin_router_ties_lower_index, pin_router_counts_k3_shape,
        pin_router_sigmoid_bias_selection_only, pin_router_sigmoid_unbiased_matches_softmax_selection, pin_expert_vs_dense,
        pin_expert_closed_form, pin_layer_combine_definition, pin_layer_identical_experts, pin_layer_relabel,
        pin_layer_token_independence, pin_layer_zero_gate_branch, pin_layer_down_scale_linear,
        pin_bf16_input_exact, pin_rmsnorm, pin_tolerance_budget, pin_shared_bf16_vs_dense,
        pin_shared_bf16_image_of_mxfp4_is_identical]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


@pytest.mark.parametrize("name", [n for n in oracle.FAULTS if n != "none"])
def test_planted_mistakes_are_caught(name):
    failed = []
    with oracle.fault(name):
        for pin in PINS:
            try:
                pin()
            except (AssertionError, ValueError):
                failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake {name!r}"


def test_route_tokens_is_route_token_per_token():
    """The batched routing the GPU tests use for every token of a prefill is the per-token routine,
    token by token (bf16 and fp32 tokens, with a bias, both scores)."""
    sh = synth.LayerShape(d_model=256, d_ff=128, n_routed=32, top_k=4, n_shared=1)
    W = synth.router_weights(sh, 3)
    bias = synth.zipf_bias(sh, 3, 1.1)
    for x_dtype in ("bf16", "f32"):
        x = synth.tokens(sh, 3, 9, x_dtype)
        xf = synth.tokens_as_f64(x, x_dtype)
        for score in ("softmax", "sigmoid_bias"):
            lg, idx, w = oracle.route_tokens(x, x_dtype, W, sh.top_k, bias, score=score)
            for t in range(x.shape[0]):
                lg1, idx1, w1 = oracle.route_token(xf[t], W, sh.top_k, bias, score=score)
                assert np.array_equal(lg[t], lg1) and np.array_equal(idx[t], idx1) and np.array_equal(w[t], w1)
