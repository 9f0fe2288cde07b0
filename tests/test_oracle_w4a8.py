"""Pins of the W4A8 oracle (oracle/w4a8.py) to properties fixed by its definition:
the activation quantiser's error bound and saturation, exactness on inputs
already on the INT8 grid, a one-hot closed form, and the bound that ties it
to the exact W4A16 product."""

import numpy as np

import synth
from oracle import gemv as ogemv, quant as oquant, w4a8


def test_activation_quantiser_bound_and_saturation():
    x = synth.gemv_x(3, 4, 1024)
    q, s = w4a8.quantize_activations_g128(x)
    x64 = x.astype(np.float64).reshape(4, 8, 128)
    s64 = s.astype(np.float64)[:, :, None]
    err = np.abs(x64 - q.reshape(4, 8, 128).astype(np.float64) * s64)
    # rint of the fp32 quotient: half a step, plus the quotient's own rounding
    assert np.all(err <= s64 / 2 + np.abs(x64) * 2.0 ** -23)
    # the largest magnitude of each group maps to +-127
    assert np.all(np.max(np.abs(q.reshape(4, 8, 128).astype(np.int32)), axis=2) == 127)
    assert q.min() >= -127 and q.max() <= 127


def test_zero_group_quantises_to_zero():
    x = np.zeros((1, 256), np.float16)
    x[0, 200] = 3.0
    q, s = w4a8.quantize_activations_g128(x)
    assert s[0, 0] == 0 and np.all(q[0, :128] == 0)
    assert q[0, 200] == 127


def test_integer_grid_inputs_are_exact():
    # x already integral with a 127 in every group: s = 1, q = x, and W4A8 equals W4A16 exactly
    rng = np.random.default_rng(4)
    x = rng.integers(-127, 128, size=(2, 512)).astype(np.float16)
    x[:, ::128] = 127
    w = synth.gemv_w(4, 40, 512)
    codes, sc = oquant.quantize_g128(w)
    q, s = w4a8.quantize_activations_g128(x)
    assert np.all(s == 1) and np.array_equal(q.astype(np.float16), x)
    assert np.array_equal(w4a8.gemv_w4a8_ref(x, codes, sc), ogemv.gemv_ref(x, codes, sc))


def test_one_hot_closed_form():
    w = synth.gemv_w(5, 16, 256)
    codes, sc = oquant.quantize_g128(w)
    for col in (0, 77, 128, 255):
        x = np.zeros((1, 256), np.float16)
        x[0, col] = 1
        s = np.float32(1) / np.float32(127)
        want = codes[:, col].astype(np.float64) * 127 * sc[:, col // 128].astype(np.float64) * np.float64(s)
        assert np.array_equal(w4a8.gemv_w4a8_ref(x, codes, sc)[0], want)


def test_error_bound_against_w4a16():
    # |y_a8 - y_a16| <= sum_k |q_w s_w| * s_x / 2 per row: the quantiser's bound carried through
    x = synth.gemv_x(6, 3, 1024)
    w = synth.gemv_w(6, 64, 1024)
    codes, sc = oquant.quantize_g128(w)
    _, s = w4a8.quantize_activations_g128(x)
    wd = np.abs(oquant.dequantize(codes, sc))                          # [N][K]
    bound = np.einsum("ngk,mg->mn", wd.reshape(64, 8, 128), s.astype(np.float64) / 2) * (1 + 1e-6)
    diff = np.abs(w4a8.gemv_w4a8_ref(x, codes, sc) - ogemv.gemv_ref(x, codes, sc))
    assert np.all(diff <= bound)
    assert diff.max() > 0
