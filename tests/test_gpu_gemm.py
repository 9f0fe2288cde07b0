"""GPU W4A16 GEMM (w4_gemm_w4a16, tcgen05 kernel) against the oracle.

y[t][r] = sum_k x[t][k] q[r][k] s[r][k/128] for n activation rows.  The kernel
expands each weight to fp16 (q * s rounded once) and accumulates in fp32 on
the tensor cores, so against the oracle's float64 product the error is a few
fp16 roundings of the weights: checked at the GEMV bar of 1e-2 * rms, and at
1e-4 * rms (growing with K past 6700, see _acc_tol) against the same product
with the weights rounded to fp16 first.
A one-hot activation reads single weights back exactly, which pins the
operand layout (nibble order, K permutation, 128-byte swizzle or the TMEM
operand columns, TMEM lanes).  Both placements of the expanded weights (shared
memory, TMEM) are checked.
"""

import numpy as np
import pytest
import torch

import synth
from int4_weight_only_w4a16_gb300 import binding
from int4_weight_only_w4a16_gb300 import model as gmodel
from oracle import gemv as ogemv, quant as oquant

pytestmark = pytest.mark.gpu


def _case(seed, n, N, K):
    x = synth.gemv_x(seed, n, K)
    w = synth.gemv_w(seed, N, K)
    packed, scales = gmodel.pack_host_matrix(w)
    codes, sc = oquant.quantize_g128(w)
    return x, packed, scales, codes, sc


def _fp16_weights_ref(x, codes, sc):
    w16 = oquant.dequantize(codes, sc).astype(np.float16).astype(np.float64)
    return x.astype(np.float64) @ w16.T


def _acc_tol(K):
    """Bound for the fp32 accumulation against the fp16-weight product, per rms: the
    tensor cores add each MMA's products into the accumulator without
    round-to-nearest, so the error grows linearly with the chain of K/16 steps
    (measured 1.25e-4 rms for one 18944-long chain); 2^-22 per step, at least 1e-4."""
    return max(1e-4, K / 16 * 2.0 ** -22)


# (n, N, K): one token (16-wide tile), ragged token tails, a half 256-row tile,
# split K (including a split that starts in the middle of a scale group), and
# the 7B layer shapes at a 512-token prompt
SHAPES = [(1, 128, 128), (5, 256, 256), (16, 384, 512), (37, 512, 3584), (45, 640, 1152),
          (300, 1024, 640), (257, 256, 1280), (512, 4608, 3584), (512, 3584, 3584), (512, 3584, 18944)]


@pytest.fixture(params=[0, 1], ids=["a_smem", "a_tmem"])
def placement(request, lib):
    """Expanded weights in shared memory (the default) or in TMEM."""
    binding.gemm_tune(request.param)
    yield request.param
    binding.gemm_tune(0)


@pytest.mark.parametrize("n,N,K", SHAPES)
def test_gemm_against_oracle(lib, placement, n, N, K):
    x, packed, scales, codes, sc = _case(n * 7 + N + K, n, N, K)
    y = binding.gemm_w4a16(torch.from_numpy(x).cuda(), packed, scales)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    got = y.cpu().numpy().astype(np.float64)
    ref = ogemv.gemv_ref(x, codes, sc)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.all(np.isfinite(got))
    assert np.abs(got - ref).max() <= 1e-2 * rms
    ref16 = _fp16_weights_ref(x, codes, sc)
    assert np.abs(got - ref16).max() <= _acc_tol(K) * rms


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("n,N,K", [s for s in SHAPES if s[0] < 512])
def test_gemm_tile_heights_against_oracle(lib, rows, n, N, K):
    # 128- and 256-row weight tiles (the automatic choice picks per shape)
    x, packed, scales, codes, sc = _case(n * 5 + N + K + rows, n, N, K)
    binding.gemm_tune_tile_rows(rows)
    try:
        y = binding.gemm_w4a16(torch.from_numpy(x).cuda(), packed, scales)
        torch.cuda.synchronize()
    finally:
        binding.gemm_tune_tile_rows(0)
    assert lib.device_error() == 0
    got = y.cpu().numpy().astype(np.float64)
    ref16 = _fp16_weights_ref(x, codes, sc)
    rms = np.sqrt(np.mean(ref16 ** 2))
    assert np.abs(got - ref16).max() <= _acc_tol(K) * rms


def test_gemm_one_hot_reads_single_weights_exactly(lib, placement):
    # row t of x is one-hot at column k_t: y[t][r] = fp16(q[r][k_t] * s) exactly
    N, K = 384, 1024
    ks = np.array(sorted({0, 1, 2, 7, 8, 15, 16, 63, 64, 65, 127, 128, 200, 255, 256, 511, 777, 1023} |
                         set(range(3, 1024, 37))))
    n = len(ks)
    x = np.zeros((n, K), np.float16)
    x[np.arange(n), ks] = 1.0
    w = synth.gemv_w(11, N, K)
    packed, scales = gmodel.pack_host_matrix(w)
    codes, sc = oquant.quantize_g128(w)
    y = binding.gemm_w4a16(torch.from_numpy(x).cuda(), packed, scales).cpu().numpy()
    want = (codes[:, ks].astype(np.float32) * sc[:, ks // 128].astype(np.float32)).astype(np.float16)
    assert np.array_equal(y, want.T.astype(np.float32))


def test_gemm_is_deterministic(lib, placement):
    x, packed, scales, codes, sc = _case(3, 77, 512, 3584)
    xd = torch.from_numpy(x).cuda()
    a = binding.gemm_w4a16(xd, packed, scales)
    b = binding.gemm_w4a16(xd, packed, scales)
    assert torch.equal(a, b)


def test_gemm_rejects_bad_shapes(lib):
    with pytest.raises(binding.W4Error):
        binding.gemm_tune(2)
    with pytest.raises(binding.W4Error):
        binding.gemm_tune_tile_rows(64)
    x = torch.zeros((4, 256), dtype=torch.float16, device="cuda")
    packed = torch.zeros((200, 32), dtype=torch.int32, device="cuda")
    scales = torch.zeros(200 * 2 + 8, dtype=torch.float16, device="cuda")
    with pytest.raises(binding.W4Error):
        binding.gemm_w4a16(x, packed, scales)   # N = 200 is not a multiple of 128
