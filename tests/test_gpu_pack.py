"""GPU pack_int4_g128 against the oracle: codes, packed words and scales bit-exact."""

import numpy as np
import pytest
import torch

import synth
from oracle import quant as oquant

pytestmark = pytest.mark.gpu


def _pack(lib, w):
    packed, scales = lib.pack_int4_g128(torch.from_numpy(np.ascontiguousarray(w)).cuda())
    torch.cuda.synchronize()
    return packed.cpu().numpy().view(np.uint32), scales.cpu().numpy()


def _assert_matches_oracle(lib, w):
    got_p, got_s = _pack(lib, w)
    codes, scales = oquant.quantize_g128(w)
    assert np.array_equal(got_s.view(np.uint16), scales.view(np.uint16))
    assert np.array_equal(got_p, oquant.pack(codes))
    assert np.array_equal(oquant.unpack(got_p), codes)


@pytest.mark.parametrize("n,k", [(512, 3584), (37, 128), (3, 1024), (4608, 3584), (1, 18944)])
def test_pack_bit_exact(lib, n, k):
    _assert_matches_oracle(lib, synth.gemv_w(11, n, k))


def test_pack_every_projection_shape(lib):
    for i, (_, n, k) in enumerate(synth.LAYER_PROJECTIONS):
        _assert_matches_oracle(lib, synth.gemv_w(20 + i, n, k))


def test_pack_lm_head_rows_sample(lib):
    # the full 152064 x 3584 LM head, packed on the GPU, checked on sampled rows
    w = synth.gemv_w(31, 152064, 3584)
    got_p, got_s = _pack(lib, w)
    rows = np.random.default_rng(0).choice(152064, 64, replace=False)
    codes, scales = oquant.quantize_g128(w[rows])
    assert np.array_equal(got_s[rows].view(np.uint16), scales.view(np.uint16))
    assert np.array_equal(got_p[rows], oquant.pack(codes))


def test_pack_special_groups(lib):
    w = np.zeros((4, 256), dtype=np.float32)
    w[1, :128] = (np.arange(128, dtype=np.float32) - 64) / np.float32(64)   # ramp
    w[2, 5] = -0.75                                                         # single non-zero
    w[3] = np.tile(np.arange(-7, 8), 18)[:256].astype(np.float32) * np.float32(2.0 ** -4)  # exact grid
    w[3, :] *= np.where(np.arange(256) < 128, 1.0, -1.0).astype(np.float32)
    w[0, 130] = 1e-30                                                       # scale underflows to 0
    _assert_matches_oracle(lib, w)
    got_p, got_s = _pack(lib, w)
    assert float(got_s[1, 0]) == 0.142822265625
    assert float(got_s[0, 1]) == 0.0 and np.all(oquant.unpack(got_p)[0] == 0)


def test_pack_nonfinite_flags_and_zeroes_the_group(lib):
    w = synth.gemv_w(12, 8, 512)
    w[3, 200] = np.nan
    w[5, 10] = 1e6   # scale 1e6/7 overflows fp16
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.device_error(clear=True)
    packed, scales = lib.pack_int4_g128(torch.from_numpy(w).cuda(), flags=flags)
    torch.cuda.synchronize()
    f = int(flags.item())
    assert f & lib.DEVERR["NONFINITE"] and f & lib.DEVERR["SCALE_OVF"]
    assert lib.device_error(clear=True) & lib.DEVERR["NONFINITE"]
    p = packed.cpu().numpy().view(np.uint32)
    s = scales.cpu().numpy()
    assert s[3, 1] == 0 and np.all(oquant.unpack(p)[3, 128:256] == 0)
    assert s[5, 0] == 0
    # untouched groups still match the oracle
    good = np.delete(np.arange(8), [3, 5])
    codes, sc = oquant.quantize_g128(w[good])
    assert np.array_equal(p[good], oquant.pack(codes))
