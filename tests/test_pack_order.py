"""The device order of include/k3moe.h (k3moe_pack_records), as restated on the host by
tests/harness.device_order, checked position by position against the header's formulas (CPU only)."""
import numpy as np

from harness import device_order


def _geometry(d, f):
    nc, ns = d * f // 2, d * f // 32
    return nc, ns, 3 * (nc + ns)


def test_gate_up_stacked_tiles_match_the_header_formula():
    d, f = 256, 384
    nc, ns, n = _geometry(d, f)
    rec = np.arange(2 * n, dtype=np.int64).reshape(2, n)  # unique value per byte position
    out = device_order(rec, d, f)
    rng = np.random.default_rng(0)
    nb = d // 32
    for _ in range(400):
        u, h, r, b = (int(rng.integers(f // 128)), int(rng.integers(2)), int(rng.integers(128)),
                      int(rng.integers(nb)))
        # stacked tile 2u + h, row r: gate row 128u + 64h + r (r < 64) or up row 128u + 64h + r - 64
        mat, row = (0, 128 * u + 64 * h + r) if r < 64 else (1, 128 * u + 64 * h + r - 64)
        src_codes = mat * (nc + ns) + row * (d // 2)
        src_scale = mat * (nc + ns) + nc + row * nb + b
        dst_mat = h  # stacked tile 2u replaces gate tile u, 2u + 1 replaces up tile u
        dst_codes = dst_mat * (nc + ns) + (128 * u + r) * (d // 2)
        assert np.array_equal(out[1, dst_codes:dst_codes + d // 2], rec[1, src_codes:src_codes + d // 2])
        c, i = divmod(r, 32)
        g, e = divmod(b, 4)
        dst_scale = dst_mat * (nc + ns) + nc + u * 128 * nb + 512 * g + 16 * i + 4 * c + e
        assert out[1, dst_scale] == rec[1, src_scale]


def test_down_tiles_match_the_header_formula():
    d, f = 256, 384
    nc, ns, n = _geometry(d, f)
    rec = np.arange(2 * n, dtype=np.int64).reshape(2, n)
    out = device_order(rec, d, f)
    base = 2 * (nc + ns)
    assert np.array_equal(out[:, base:base + nc], rec[:, base:base + nc])  # down codes untouched
    rng = np.random.default_rng(1)
    nb = f // 32
    for _ in range(200):
        r, b = int(rng.integers(d)), int(rng.integers(nb))
        t, rr = divmod(r, 128)
        c, i = divmod(rr, 32)
        g, e = divmod(b, 4)
        tile = base + nc + t * 128 * nb
        assert out[1, tile + 512 * g + 16 * i + 4 * c + e] == rec[1, base + nc + r * nb + b]


def test_device_order_is_a_permutation_of_each_region_pair():
    d, f = 128, 256
    nc, ns, n = _geometry(d, f)
    rec = np.random.default_rng(2).integers(0, 1 << 40, size=(1, n))
    out = device_order(rec, d, f)
    gu = np.r_[0:2 * (nc + ns)]
    assert np.array_equal(np.sort(rec[0, gu]), np.sort(out[0, gu]))
    dn = np.r_[2 * (nc + ns):n]
    assert np.array_equal(np.sort(rec[0, dn]), np.sort(out[0, dn]))
    # codes stay codes and scales stay scales
    codes = np.r_[0:nc, nc + ns:2 * nc + ns]
    assert np.array_equal(np.sort(rec[0, codes]), np.sort(out[0, codes]))
