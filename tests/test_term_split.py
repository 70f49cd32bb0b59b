"""Precision of the activation terms (CPU): the bounds that include/k3moe.h states for each activation
mode (and the exactness of the router weights' three bf16 parts), checked on a model of the split
built from the formats' definitions (OCP Microscaling Formats
v1.0: E4M3 with 3 mantissa bits, bias 7, subnormal quantum 2^-9, largest finite 448; E2M1 values
0, 0.5, 1, 1.5, 2, 3, 4, 6; E8M0 scales 2^(b - 127)) and round-to-nearest-even.

The split, per 32-element block v:
  E4M3 form: r_0 = v; term j = RN_e4m3(r_j / 2^e_j) 2^e_j with e_j = floor(log2 max|r_j|) - 7;
             r_(j+1) = r_j - term j.
  E2M1 form: E = floor(log2 max|v|); term j = RN_e2m1(r_j / 2^(E - 3j)) 2^(E - 3j).
The kernels form the residuals in fp32; every residual here is exact in fp32 (a rounded value within a
factor two of the value it is subtracted from, or a multiple of that value's ulp), so the model in
double precision reproduces them. No product code is imported.
"""
import numpy as np
import pytest


def _rne_on_grid(a, quantum, largest):
    n = np.rint(a / quantum)  # half-way cases to the even count, which is the even mantissa
    return np.minimum(n * quantum, largest)


def rn_e4m3(s):
    a = np.abs(s)
    k = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    quantum = np.exp2(np.maximum(k, -6) - 3)  # 3 mantissa bits; subnormals below 2^-6
    return np.sign(s) * _rne_on_grid(a, quantum, 448.0)


def rn_e2m1(s):
    a = np.abs(s)
    quantum = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    return np.sign(s) * _rne_on_grid(a, quantum, 6.0)


def _floor_log2(a):
    return np.where(a > 0, np.floor(np.log2(np.where(a > 0, a, 1.0))), 0.0)


def split_e4m3(v, terms):
    r = np.array(v, dtype=np.float64)
    total = np.zeros_like(r)
    for _ in range(terms):
        e = np.clip(_floor_log2(np.max(np.abs(r), axis=-1, keepdims=True)) - 7, -127, 127)
        t = rn_e4m3(r * np.exp2(-e)) * np.exp2(e)
        total += t
        r = r - t
    return total


def split_e2m1(v, terms):
    r = np.array(v, dtype=np.float64)
    E = _floor_log2(np.max(np.abs(r), axis=-1, keepdims=True))
    total = np.zeros_like(r)
    for j in range(terms):
        e = np.clip(E - 3 * j, -127, 127)
        s = r * np.exp2(-e)
        assert np.all(np.abs(s) <= 2.0)  # never saturates: every scaled residual within [-2, 2]
        t = rn_e2m1(s) * np.exp2(e)
        total += t
        r = r - t
    return total


def to_bf16(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32)
    u = ((u + np.uint32(0x7FFF) + ((u >> 16) & np.uint32(1))) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


def blocks(n, seed, spread=16.0):
    """Blocks of 32 fp32 values: a block scale over 2^-20..2^20, elements down to 2^-spread below it,
    random signs, 5 % zeros; plus blocks whose maximum sits just below or at a power of two."""
    rng = np.random.default_rng(seed)
    mag = np.exp2(rng.uniform(-20, 20, (n, 1))) * np.exp2(rng.uniform(-spread, 0, (n, 32)))
    v = mag * rng.choice([-1.0, 1.0], (n, 32))
    v[rng.random((n, 32)) < 0.05] = 0.0
    edge = v[: n // 8].copy()
    edge[:, 0] = np.exp2(np.round(np.log2(np.abs(edge[:, 0]) + 1e-300))) * np.where(
        rng.random(len(edge)) < 0.5, 1.0, 1.0 - 2.0 ** -23)
    v = np.concatenate([v, edge])
    return v.astype(np.float32).astype(np.float64)


def rel_to_block_max(v, approx):
    m = np.max(np.abs(v), axis=1)
    keep = m > 0
    return np.max(np.abs(v - approx), axis=1)[keep] / m[keep]


def test_model_rounding_matches_the_format_tables():
    # E2M1: every representable value maps to itself; midpoints go to the even mantissa
    e2m1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    assert np.array_equal(rn_e2m1(e2m1), e2m1) and np.array_equal(rn_e2m1(-e2m1), -e2m1)
    assert list(rn_e2m1(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0]))) == \
        [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0]
    # E4M3: all 126 finite positive values (exponent fields 0..15, mantissa 0..7, less the NaN code)
    table = [(m / 8 * 2.0 ** -6, m) for m in range(1, 8)]
    table += [((1 + m / 8) * 2.0 ** (E - 7), m) for E in range(1, 16) for m in range(8) if not (E == 15 and m == 7)]
    vals = np.array([t[0] for t in table])
    mant = np.array([t[1] for t in table])
    assert len(vals) == 126 and vals.max() == 448.0 and vals.min() == 2.0 ** -9
    assert np.all(np.diff(vals) > 0)
    assert np.array_equal(rn_e4m3(vals), vals)
    # a midpoint between neighbours goes to the one with the even mantissa
    mids = (vals[:-1] + vals[1:]) / 2
    even = np.where(mant[:-1] % 2 == 0, vals[:-1], vals[1:])
    assert np.array_equal(rn_e4m3(mids), even)
    assert rn_e4m3(np.array([2.0 ** -10]))[0] == 0.0  # half the smallest subnormal: ties to zero
    assert rn_e4m3(np.array([1000.0]))[0] == 448.0    # satfinite


def test_e2m1_eight_terms_within_2_to_minus_23_of_the_block_maximum():
    """Activation terms at one and two tokens (both modes): x and h."""
    v = blocks(40000, 1, spread=30.0)
    err = rel_to_block_max(v, split_e2m1(v, 8))
    assert err.max() <= 2.0 ** -23


def test_bf16_in_two_e4m3_terms_exact_down_to_2_to_minus_13():
    """bf16 x from 3 tokens on: elements of at least 2^-13 of their block's maximum are exact, the rest
    within 2^-21 of the maximum."""
    v = to_bf16(blocks(40000, 2)).astype(np.float64)
    approx = split_e4m3(v, 2)
    m = np.max(np.abs(v), axis=1, keepdims=True)
    big = np.abs(v) >= 2.0 ** -13 * m
    assert np.array_equal(approx[big], v[big])
    assert rel_to_block_max(v, approx).max() <= 2.0 ** -21


@pytest.mark.parametrize("terms,bound", [(3, 2.0 ** -12), (2, 2.0 ** -8)])
def test_e4m3_terms_of_fp32_values(terms, bound):
    """fp32 x and h (three terms, the default mode) and h in the bf16-class mode (two terms). With the
    first scale 2^e the block maximum is at least 2^(e + 7) and every residual after the first term at
    most 8 2^e (half the E4M3 spacing of the top binade); each further term's scale is at least 2^4
    smaller and leaves at most 8 times its scale. n terms leave at most 2^(e + 3 - 4 (n - 1)), which
    is 2^(-4 n) of the block maximum: 2^-8 for two terms, 2^-12 for three."""
    v = blocks(40000, 3 + terms)
    err = rel_to_block_max(v, split_e4m3(v, terms))
    assert err.max() <= bound
    assert err.max() > bound / 64  # the bound is the right order: far from exact


def test_two_e4m3_terms_keep_about_eight_bits_per_element():
    """The bf16-class h: every element of at least 2^-13 of its block's maximum to 2^-8 relative."""
    v = blocks(40000, 7)
    approx = split_e4m3(v, 2)
    m = np.max(np.abs(v), axis=1, keepdims=True)
    big = (np.abs(v) >= 2.0 ** -13 * m) & (v != 0)
    assert (np.abs(v - approx)[big] / np.abs(v)[big]).max() <= 2.0 ** -8


def test_three_bf16_parts_hold_every_fp32_weight():
    """The router's weight-loading split (k3moe_prepare_router): W = W0 + W1 + W2 with each part the
    bf16 rounding of what the earlier parts leave. Each part takes 8 significant bits of the residual,
    and every residual is exact in fp32, so the three parts hold all 24 bits of a normal fp32 weight."""
    rng = np.random.default_rng(8)
    w = (rng.standard_normal(200000) * np.exp2(rng.uniform(-40, 40, 200000))).astype(np.float32)
    w = np.concatenate([w, np.array([1.0, -1.0, 2.0 ** 30, np.float32(1 + 2 ** -23), 0.0], dtype=np.float32)])
    r = w.copy()
    parts = []
    for _ in range(3):
        p = to_bf16(r)
        parts.append(p)
        r = (r - p).astype(np.float32)  # exact: see the docstring
    total = parts[0].astype(np.float64) + parts[1].astype(np.float64) + parts[2].astype(np.float64)
    assert np.array_equal(total, w.astype(np.float64))
    assert np.all(r == 0)
    two = parts[0].astype(np.float64) + parts[1].astype(np.float64)
    assert not np.array_equal(two, w.astype(np.float64))  # two parts would not do
