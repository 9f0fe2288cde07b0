"""GPU gemv_w4a16 against the float64 oracle: max|err| <= 1e-2 * rms(ref)."""

import numpy as np
import pytest
import torch

import synth
from oracle import gemv as ogemv, quant as oquant

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _case(lib, seed, m, n, k):
    x = synth.gemv_x(seed, m, k)
    w = synth.gemv_w(seed, n, k)
    packed, scales = lib.pack_int4_g128(torch.from_numpy(w).cuda())
    codes, sc = oquant.quantize_g128(w)
    return x, packed, scales, codes, sc


def _check(y, ref, tol=TOL):
    y = y.float().cpu().numpy().astype(np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(y - ref).max()
    assert np.all(np.isfinite(y))
    assert err <= tol * rms, "max err %.3e > %.1e * rms %.3e" % (err, tol, rms)
    return err / rms


@pytest.fixture(autouse=True)
def _default_tuning(lib):
    lib.gemv_tune()
    yield
    lib.gemv_tune()


# variant 0: the streaming CUDA-core kernel at m = 1, the mma.sync kernel at
# m = 2..11, the tcgen05 kernel at m = 12..16; variant 1: the mma.sync kernel at
# every m; variant 3: the tcgen05 kernel at every m
@pytest.mark.parametrize("variant", [0, 1, 3])
def test_k_proj_512x3584(lib, variant):
    lib.gemv_tune(variant)
    x, packed, scales, codes, sc = _case(lib, 1, 1, 512, 3584)
    y = lib.gemv_w4a16(torch.from_numpy(x).cuda(), packed, scales)
    _check(y, ogemv.gemv_ref(x, codes, sc))


def test_all_seven_projections_of_a_layer(lib):
    for i, (_, n, k) in enumerate(synth.LAYER_PROJECTIONS):
        x, packed, scales, codes, sc = _case(lib, 100 + i, 1, n, k)
        y = lib.gemv_w4a16(torch.from_numpy(x).cuda(), packed, scales)
        _check(y, ogemv.gemv_ref(x, codes, sc))


@pytest.mark.parametrize("variant", [0, 3])
@pytest.mark.parametrize("m", [1, 2, 3, 4, 8, 16])
def test_batched_gate_up_down(lib, m, variant):
    lib.gemv_tune(variant)
    for i, (n, k) in enumerate([(18944, 3584), (3584, 18944)]):
        x, packed, scales, codes, sc = _case(lib, 200 + 10 * m + i, m, n, k)
        y = lib.gemv_w4a16(torch.from_numpy(x).cuda(), packed, scales)
        _check(y, ogemv.gemv_ref(x, codes, sc))


@pytest.mark.parametrize("variant", [0, 1, 3])
@pytest.mark.parametrize("n,k", [(1, 128), (17, 384), (100, 3584), (513, 18944), (33, 256), (5, 640),
                                 (4608, 3584), (3584, 18944), (7, 32768), (129, 4608), (300, 9344)])
def test_ragged_shapes_batch_1(lib, n, k, variant):
    # k = 32768 is longer than the streaming kernel's ring takes: batch 1 falls back to
    # the mma.sync kernel (variant 0)
    lib.gemv_tune(variant)
    x, packed, scales, codes, sc = _case(lib, 300 + n + k, 1, n, k)
    y = lib.gemv_w4a16(torch.from_numpy(x).cuda(), packed, scales)
    _check(y, ogemv.gemv_ref(x, codes, sc))


@pytest.mark.parametrize("m", [1, 3])
@pytest.mark.parametrize("variant", [0, 1, 3])
def test_bias_and_residual(lib, variant, m):
    lib.gemv_tune(variant)
    n, k = 4608, 3584
    x, packed, scales, codes, sc = _case(lib, 400, m, n, k)
    bias = synth.gemv_bias(400, n)
    res = synth.gemv_x(401, m, n)
    y = lib.gemv_w4a16(torch.from_numpy(x).cuda(), packed, scales, bias=torch.from_numpy(bias).cuda(),
                       residual=torch.from_numpy(res).cuda())
    _check(y, ogemv.gemv_ref(x, codes, sc, bias=bias, residual=res))


@pytest.mark.parametrize("variant", [0, 1, 3])
@pytest.mark.parametrize("m", [1, 2, 5, 9, 11, 12, 16])
@pytest.mark.parametrize("n,k", [(1, 128), (17, 384), (130, 640), (513, 18944), (4608, 3584), (200, 3584)])
def test_tensor_core_batches_ragged(lib, variant, m, n, k):
    # the mma.sync kernel (variant 1 at every m, variant 0 at m = 2..11) and the tcgen05
    # kernel (variant 3 at every m, variant 0 at m = 12..16): row tiles with a ragged
    # tail, one to many split-K pieces, one and two n-tiles
    lib.gemv_tune(variant)
    x, packed, scales, codes, sc = _case(lib, 800 + m + n + k, m, n, k)
    y = lib.gemv_w4a16(torch.from_numpy(x).cuda(), packed, scales)
    _check(y, ogemv.gemv_ref(x, codes, sc))


@pytest.mark.parametrize("m", [1, 16])
def test_tensor_core_kernel_layer_shapes(lib, m):
    # the tensor-core kernel on the projection shapes of a layer (at m = 1 by variant 1)
    lib.gemv_tune(1)
    for n, k in ((4608, 3584), (3584, 3584), (18944, 3584), (3584, 18944), (513, 18944)):
        x, packed, scales, codes, sc = _case(lib, 950 + m + n, m, n, k)
        y = lib.gemv_w4a16(torch.from_numpy(x).cuda(), packed, scales)
        _check(y, ogemv.gemv_ref(x, codes, sc))


@pytest.mark.parametrize("variant", [1, 3])
def test_tensor_core_one_hot_rows_pick_columns(lib, variant):
    # closed form: activation row i = e_{c_i} gives y[i] = q[:, c_i] * s[:, c_i/128] exactly
    # (one nonzero product per sum); checks the K order of the fragments position by position
    lib.gemv_tune(variant)
    n, k, m = 200, 1024, 16
    w = synth.gemv_w(501, n, k)
    packed, scales = lib.pack_int4_g128(torch.from_numpy(w).cuda())
    codes, sc = oquant.quantize_g128(w)
    for cols in (range(0, 16), range(16, 32), range(112, 144), (0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15),
                 (1023, 777, 128, 513, 31, 32, 33, 63, 64, 65, 95, 96, 97, 100, 900, 1000)):
        cols = list(cols)[:m]
        x = np.zeros((m, k), np.float16)
        for i, c in enumerate(cols):
            x[i, c] = 1
        y = lib.gemv_w4a16(torch.from_numpy(x).cuda(), packed, scales).cpu().numpy()
        for i, c in enumerate(cols):
            want = (codes[:, c].astype(np.float64) * sc[:, c // 128].astype(np.float64)).astype(np.float16)
            assert np.array_equal(y[i], want), (i, c)


@pytest.mark.parametrize("variant", [0, 3])
@pytest.mark.parametrize("n,k", [(37, 1152), (6, 4224), (5, 18944), (130, 640)])
def test_batch_1_one_hot_columns(lib, n, k, variant):
    # closed form at batch 1 (variant 0: the streaming kernel; 3: the tcgen05 kernel,
    # split K at 18944): x = e_c gives y = q[:, c] * s[:, c/128] exactly.  The columns
    # cover every element slot of a word, every word of a group, several groups and
    # the last columns of a row, so a dot that reads the wrong K index fails
    lib.gemv_tune(variant)
    w = synth.gemv_w(502 + n, n, k)
    packed, scales = lib.pack_int4_g128(torch.from_numpy(w).cuda())
    codes, sc = oquant.quantize_g128(w)
    cols = sorted(c for c in set(list(range(0, 40)) + [127, 128, 129, 255, 256, 511, 512, 640, 1000, 1023, 1024,
                                                       1025, k - 33, k - 32, k - 9, k - 8, k - 1]) if c < k)
    for c in cols:
        x = np.zeros((1, k), np.float16)
        x[0, c] = 1
        y = lib.gemv_w4a16(torch.from_numpy(x).cuda(), packed, scales).cpu().numpy()
        want = (codes[:, c].astype(np.float64) * sc[:, c // 128].astype(np.float64)).astype(np.float16)
        assert np.array_equal(y[0], want), c


@pytest.mark.parametrize("m", [1, 16])
@pytest.mark.parametrize("variant", [1, 3])
def test_tensor_core_split_k_deterministic(lib, m, variant):
    # 3584 x 18944 splits K over several CTAs per row block (both tensor-core kernels);
    # the last CTA adds the partials in a fixed order and puts its ticket back to zero
    lib.gemv_tune(variant)
    x, packed, scales, _, _ = _case(lib, 601, m, 3584, 18944)
    xt = torch.from_numpy(x).cuda()
    ws = lib.gemv_workspace(m, 3584, 18944)
    a = lib.gemv_w4a16(xt, packed, scales, workspace=ws).clone()
    b = lib.gemv_w4a16(xt, packed, scales, workspace=ws).clone()
    assert torch.equal(a, b)
    row_blocks = 3584 // 128   # the tickets: the workspace's last row_blocks words
    assert int(ws[-4 * row_blocks:].sum()) == 0
    assert lib.device_error() == 0


def test_one_hot_activation_picks_a_column(lib):
    # closed form on the GPU: x = e_k gives y = q[:, k] * s[:, k/128] (exact products; only fp16 output rounding)
    n, k = 64, 1024
    w = synth.gemv_w(500, n, k)
    packed, scales = lib.pack_int4_g128(torch.from_numpy(w).cuda())
    codes, sc = oquant.quantize_g128(w)
    for col in (0, 127, 128, 777, 1023):
        x = np.zeros((1, k), np.float16)
        x[0, col] = 1
        y = lib.gemv_w4a16(torch.from_numpy(x).cuda(), packed, scales).cpu().numpy()
        want = (codes[:, col].astype(np.float64) * sc[:, col // 128].astype(np.float64)).astype(np.float16)
        assert np.array_equal(y[0], want)


def test_streaming_kernel_deterministic(lib):
    x, packed, scales, _, _ = _case(lib, 600, 1, 3584, 18944)
    xt = torch.from_numpy(x).cuda()
    ws = lib.gemv_workspace(1, 3584, 18944)
    a = lib.gemv_w4a16(xt, packed, scales, workspace=ws).clone()
    b = lib.gemv_w4a16(xt, packed, scales, workspace=ws).clone()
    assert torch.equal(a, b)
    assert lib.device_error() == 0


def test_lm_head_sampled_rows(lib):
    # full-size 152064 x 3584 GEMV in the launch configuration the decode step uses; sampled rows checked
    n, k = 152064, 3584
    x = synth.gemv_x(700, 1, k)
    w = synth.gemv_w(700, n, k)
    packed, scales = lib.pack_int4_g128(torch.from_numpy(w).cuda())
    y = lib.gemv_w4a16(torch.from_numpy(x).cuda(), packed, scales).float().cpu().numpy()[0]
    rows = np.random.default_rng(1).choice(n, 256, replace=False)
    codes, sc = oquant.quantize_g128(w[rows])
    ref = ogemv.gemv_ref(x, codes, sc)[0]
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.abs(y[rows] - ref).max() <= TOL * rms


@pytest.mark.parametrize("n,k", [(512, 3584), (18944, 3584), (3584, 18944), (100, 640)])
def test_w4a8_variant_against_its_oracle(lib, n, k):
    # variant 2 (INT8 activations per 128-group, dp4a) against the W4A8 oracle, which
    # decides the INT8 codes in the same fp32 arithmetic: only fp32 rounding of the
    # scaled group sums separates them
    from oracle import w4a8
    lib.gemv_tune(2)
    x, packed, scales, codes, sc = _case(lib, 1200 + n, 1, n, k)
    y = lib.gemv_w4a16(torch.from_numpy(x).cuda(), packed, scales).float().cpu().numpy().astype(np.float64)
    ref = w4a8.gemv_w4a8_ref(x, codes, sc)
    # within one fp16 ulp of the exact W4A8 value, plus the fp32 accumulation error of the
    # 112..592 scaled group sums (bounded here by 1e-4 of the output rms)
    ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
    rms8 = np.sqrt(np.mean(ref ** 2))
    assert np.all(np.abs(y - ref) <= ulp + 1e-4 * rms8), np.max(np.abs(y - ref) - ulp) / rms8
    # and, as a different product, within its quantisation bound of exact W4A16
    rms = np.sqrt(np.mean(ogemv.gemv_ref(x, codes, sc) ** 2))
    assert np.abs(y - ogemv.gemv_ref(x, codes, sc)).max() <= 5e-2 * rms
