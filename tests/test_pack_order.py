"""The device scale order of include/k3moe.h (k3moe_pack_records), as restated on the host by
tests/harness.device_order, checked position by position against the header's formula (CPU only)."""
import numpy as np

from harness import device_order


def test_device_order_matches_the_header_formula():
    d, f = 256, 384
    nc, ns = d * f // 2, d * f // 32
    n = 3 * (nc + ns)
    rec = np.arange(2 * n, dtype=np.int64).reshape(2, n)  # unique value per byte position
    out = device_order(rec, d, f)
    rng = np.random.default_rng(0)
    for m, (rows, cols) in enumerate(((f, d), (f, d), (d, f))):
        nb = cols // 32
        base = m * (nc + ns)
        assert np.array_equal(out[:, base:base + nc], rec[:, base:base + nc])  # codes untouched
        for _ in range(200):
            r, b = int(rng.integers(rows)), int(rng.integers(nb))
            t, rr = divmod(r, 128)
            c, i = divmod(rr, 32)
            g, e = divmod(b, 4)
            tile = base + nc + t * 128 * nb
            assert out[1, tile + 512 * g + 16 * i + 4 * c + e] == rec[1, base + nc + r * nb + b]


def test_device_order_is_a_permutation_of_each_tile():
    d, f = 128, 256
    nc, ns = d * f // 2, d * f // 32
    rec = np.random.default_rng(1).integers(0, 1 << 40, size=(1, 3 * (nc + ns)))
    out = device_order(rec, d, f)
    for m, cols in enumerate((d, d, f)):
        nb = cols // 32
        s0 = m * (nc + ns) + nc
        for t in range(ns // (128 * nb)):
            a = rec[0, s0 + t * 128 * nb: s0 + (t + 1) * 128 * nb]
            b = out[0, s0 + t * 128 * nb: s0 + (t + 1) * 128 * nb]
            assert np.array_equal(np.sort(a), np.sort(b))
