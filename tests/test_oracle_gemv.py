"""Pins for oracle.gemv (CPU only): closed forms and brute force."""

import numpy as np

from oracle import gemv, quant


def test_constant_codes_closed_form():
    n, k = 5, 384
    for c in (-8, -3, 0, 7):
        codes = np.full((n, k), c, dtype=np.int8)
        scales = np.full((n, k // 128), 0.25, dtype=np.float16)
        y = gemv.gemv_ref(np.ones(k, dtype=np.float16), codes, scales)
        assert np.all(y == k * c * 0.25)


def test_one_hot_picks_a_column_and_its_group_scale():
    r = np.random.default_rng(5)
    n, k = 6, 512
    codes = r.integers(-8, 8, size=(n, k)).astype(np.int8)
    scales = (r.random((n, k // 128)) + 0.5).astype(np.float16)
    for col in (0, 127, 128, 300, 511):
        x = np.zeros(k, dtype=np.float16)
        x[col] = 1
        y = gemv.gemv_ref(x, codes, scales)
        want = codes[:, col].astype(np.float64) * scales[:, col // 128].astype(np.float64)
        assert np.array_equal(y, want)


def test_brute_force_loops_tiny():
    r = np.random.default_rng(6)
    n, k, m = 3, 256, 2
    codes = r.integers(-8, 8, size=(n, k)).astype(np.int8)
    scales = (r.random((n, k // 128)) * 0.1).astype(np.float16)
    x = r.standard_normal((m, k)).astype(np.float16)
    bias = r.standard_normal(n).astype(np.float16)
    res = r.standard_normal((m, n)).astype(np.float16)
    y = gemv.gemv_ref(x, codes, scales, bias=bias, residual=res)
    for mi in range(m):
        for ni in range(n):
            acc = 0.0
            for ki in range(k):
                acc += float(x[mi, ki]) * int(codes[ni, ki]) * float(scales[ni, ki // 128])
            acc += float(bias[ni]) + float(res[mi, ni])
            assert abs(acc - y[mi, ni]) <= 1e-12 * max(1.0, abs(acc))


def test_rows_subset_matches_full():
    r = np.random.default_rng(8)
    w = r.standard_normal((40, 256)).astype(np.float32) * np.float32(0.02)
    codes, scales = quant.quantize_g128(w)
    x = r.standard_normal(256).astype(np.float16)
    full = gemv.gemv_ref(x, codes, scales)
    rows = np.array([0, 7, 39])
    assert np.allclose(gemv.gemv_rows_ref(x, codes, scales, rows), full[rows], rtol=0, atol=1e-15)


def test_matches_dequantised_dot_library_routine():
    r = np.random.default_rng(9)
    w = r.standard_normal((16, 384)).astype(np.float32) * np.float32(0.02)
    codes, scales = quant.quantize_g128(w)
    x = r.standard_normal(384).astype(np.float16)
    deq = quant.dequantize(codes, scales)
    ref = np.array([np.dot(deq[i], x.astype(np.float64)) for i in range(16)])
    assert np.allclose(gemv.gemv_ref(x, codes, scales), ref, rtol=1e-14, atol=1e-15)
