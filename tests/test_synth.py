"""The seeded input generator: C twin == numpy twin, and the value distributions of the workloads (CPU only)."""
import math

import numpy as np

import synth


def test_host_c_matches_numpy_twin():
    for sh, seed, layer, e in [(synth.TINY, 0, 0, 0), (synth.TINY, 0, 0, 32), (synth.LayerShape(64, 32, 4, 2, 1), 9, 3, 2)]:
        a = synth.records_host(sh, seed, layer, [e])[0]
        b = synth.records_host_numpy(sh, seed, layer, e)
        assert np.array_equal(a, b)


def test_record_layout_and_distribution():
    sh = synth.TINY
    rec = synth.records_host(sh, 0, 0, [3])[0]
    assert rec.shape == (sh.record_stride,)
    assert sh.record_stride % 4096 == 0 and sh.record_stride >= sh.record_bytes
    d, f = sh.d_model, sh.d_ff
    nc, ns = d * f // 2, d * f // 32
    for m in range(3):
        codes = rec[m * (nc + ns): m * (nc + ns) + nc]
        scales = rec[m * (nc + ns) + nc: (m + 1) * (nc + ns)]
        assert scales.min() >= 121 and scales.max() <= 125
        assert set(np.unique(scales)) == {121, 122, 123, 124, 125}
        nib = np.concatenate([codes & 0xF, codes >> 4])
        hist = np.bincount(nib, minlength=16)
        assert hist.min() > 0.8 * len(nib) / 16 and hist.max() < 1.2 * len(nib) / 16
    assert not rec[sh.record_bytes:].any()  # zero padding up to the 4 KiB stride


def test_distinct_streams():
    sh = synth.TINY
    r = synth.records_host(sh, 0, 0, [0, 1])
    assert not np.array_equal(r[0], r[1])
    r2 = synth.records_host(sh, 1, 0, [0])
    assert not np.array_equal(r[0], r2[0])


def test_normals_and_router_weights():
    z = synth.normals(synth.stream_key(5, synth.KIND_TOKENS, 0), 200000)
    assert abs(z.mean()) < 0.01 and abs(z.var() - 1.0) < 0.02
    W = synth.router_weights(synth.TINY, 0)
    assert W.dtype == np.float32 and W.shape == (32, 256)
    assert abs(W.astype(np.float64).var() * 256 - 1.0) < 0.05


def test_bf16_rounding():
    a = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38], np.float32)
    b = synth.f32_to_bf16_bits(a)
    back = synth.bf16_bits_to_f32(b)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0 + 2 ** -6 and back[3] == -2.5
    x = synth.tokens(synth.K3, 1, 2, "bf16")
    assert x.dtype == np.uint16 and x.shape == (2, 7168)


def test_zipf_bias():
    b = synth.zipf_bias(synth.K3, 2, 1.1)
    r = np.exp(-b.astype(np.float64) / 1.1)
    assert np.allclose(np.sort(r), np.arange(1, 897), rtol=1e-5)
    assert math.isclose(b.max(), 0.0, abs_tol=1e-7)
