"""Pins for oracle.quant: quantisation, packing and unpacking (CPU only)."""

import os

import numpy as np
import pytest

from oracle import quant

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_pack_hand_worked_words():
    codes_line, words_line = _golden_lines("pack_words.txt")
    codes = np.array([int(c) for c in codes_line], dtype=np.int8)[None, :]
    words = np.array([int(w, 16) for w in words_line], dtype=np.uint32)[None, :]
    assert np.array_equal(quant.pack(codes), words)
    assert np.array_equal(quant.unpack(words), codes)


def test_pack_every_value_every_slot():
    # each code value at each of the 16 positions of a two-word row, others 0
    base = 0x88888888  # all nibbles u = 8, i.e. q = 0
    for pos in range(16):
        for qv in range(-8, 8):
            codes = np.zeros((1, 16), dtype=np.int8)
            codes[0, pos] = qv
            slot = quant.slot_of_element(pos % 8)
            want = [base, base]
            w = want[pos // 8]
            w &= ~(0xF << (4 * slot)) & 0xFFFFFFFF
            w |= (qv + 8) << (4 * slot)
            want[pos // 8] = w
            got = quant.pack(codes)
            assert [int(v) for v in got[0]] == want, (pos, qv)
            assert np.array_equal(quant.unpack(got), codes)


def test_slot_pairs_share_halfword_position():
    # elements 2i and 2i+1 sit 16 bits apart, at bit 4i of each half
    for i in range(4):
        assert quant.slot_of_element(2 * i) == i
        assert quant.slot_of_element(2 * i + 1) == i + 4


def test_pack_unpack_roundtrip_random():
    r = np.random.default_rng(3)
    codes = r.integers(-8, 8, size=(7, 256)).astype(np.int8)
    assert np.array_equal(quant.unpack(quant.pack(codes)), codes)


def test_ramp_group_hand_worked():
    lines = _golden_lines("ramp_group.txt")
    scale = float(lines[0][0])
    table = [tuple(int(v) for v in ln) for ln in lines[1:]]
    w = ((np.arange(128, dtype=np.float32) - 64) / np.float32(64))[None, :]
    codes, scales = quant.quantize_g128(w)
    assert scales.dtype == np.float16 and float(scales[0, 0]) == scale
    for k in range(128):
        d = k - 64
        mag = next(q for lo, hi, q in table if lo <= abs(d) <= hi)
        assert int(codes[0, k]) == int(np.sign(d)) * mag, k


def test_single_nonzero_group():
    w = np.zeros((1, 256), dtype=np.float32)
    w[0, 5] = -0.75
    w[0, 200] = 3.5
    codes, scales = quant.quantize_g128(w)
    assert float(scales[0, 0]) == float(np.float16(np.float32(0.75) / np.float32(7)))
    assert float(scales[0, 1]) == 0.5  # 3.5 / 7 exactly
    assert codes[0, 5] == -7 and codes[0, 200] == 7
    assert np.count_nonzero(codes) == 2


def test_exact_grid_roundtrips():
    # w = j * 2^-4 with j covering -7..7: the scale is exactly 2^-4 and q = j
    j = np.tile(np.arange(-7, 8), 9)[:128].astype(np.float32)
    w = (j * np.float32(2.0 ** -4))[None, :]
    codes, scales = quant.quantize_g128(w)
    assert float(scales[0, 0]) == 2.0 ** -4
    assert np.array_equal(codes[0], j.astype(np.int8))


def test_zero_group():
    w = np.zeros((2, 128), dtype=np.float32)
    codes, scales = quant.quantize_g128(w)
    assert np.all(scales == 0) and np.all(codes == 0)


def test_invariants_random():
    r = np.random.default_rng(11)
    w = (r.standard_normal((64, 1024), dtype=np.float32) * np.float32(0.02))
    codes, scales = quant.quantize_g128(w)
    assert codes.min() >= -8 and codes.max() <= 7
    s = scales.astype(np.float64)
    deq = quant.dequantize(codes, scales)
    err = np.abs(w.astype(np.float64) - deq).reshape(64, 8, 128)
    assert np.all(err <= (s / 2 * (1 + 2.0 ** -20))[:, :, None])
    # every non-zero group reaches |q| = 7 (its largest element)
    assert np.all(np.abs(codes.reshape(64, 8, 128)).max(axis=2) == 7)


def test_nonfinite_and_overflow_rejected():
    w = np.zeros((1, 128), dtype=np.float32)
    w[0, 3] = np.nan
    with pytest.raises(quant.NonFiniteError):
        quant.quantize_g128(w)
    w[0, 3] = np.inf
    with pytest.raises(quant.NonFiniteError):
        quant.quantize_g128(w)
    w[0, 3] = 1e6  # 1e6 / 7 > 65504
    with pytest.raises(quant.NonFiniteError):
        quant.quantize_g128(w)


def test_minus_eight_roundtrips_through_pack():
    codes = np.full((1, 8), -8, dtype=np.int8)
    assert int(quant.pack(codes)[0, 0]) == 0
    assert np.array_equal(quant.unpack(quant.pack(codes)), codes)
