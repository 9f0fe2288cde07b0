"""GPU W4A16 GEMM (w4_gemm_w4a16, tcgen05 kernel) against the oracle.

y[t][r] = sum_k x[t][k] q[r][k] s[r][k/128] for n activation rows.  The kernel
multiplies the INT4 codes themselves on the tensor cores (exact products),
sums each 128-column scale group into its own fp32 accumulator and applies the
group's scale in fp32, so against the oracle's float64 product the only error
is fp32 accumulation: checked at 1e-4 * rms (growing with K past 6700, see
_acc_tol) -- a hundred times inside the GEMV bar of 1e-2 * rms, and tight
enough to fail a kernel that rounds each weight to fp16 as q * s.  A one-hot
activation reads single weights back exactly (q * s in fp32), which pins the
operand layout (nibble order, K permutation, 128-byte swizzle, TMEM lanes and
the accumulator of each scale group).
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


def _acc_tol(K):
    """Bound for the fp32 accumulation against the float64 product, per rms: the
    tensor cores add each MMA's products into the accumulator without
    round-to-nearest, so the error grows linearly with the chain of K/16 steps;
    2^-22 per step, at least 1e-4."""
    return max(1e-4, K / 16 * 2.0 ** -22)


# (n, N, K): one token (64-wide tile), ragged token tails, each tile width (64,
# 128, 256), split K (in whole scale groups), stream-K at each tile width (33,
# 100 and 300 rows x 5120 or 2560 x 8192: 40 tiles of 64 groups over 152 CTAs
# of 16-17 groups, up to five pieces a tile, ragged token tails), and the 7B
# layer shapes at a 512-token prompt (down by stream-K, 56 tiles over 152 CTAs),
# and launches whose tiles outnumber the SMs (160 tiles, no split; one with a
# ragged token tail)
SHAPES = [(1, 128, 128), (5, 256, 256), (16, 384, 512), (37, 512, 3584), (45, 640, 1152), (100, 384, 1024),
          (300, 1024, 640), (257, 256, 1280), (33, 5120, 8192), (100, 5120, 8192), (300, 2560, 8192),
          (512, 4608, 3584), (512, 3584, 3584), (512, 3584, 18944), (300, 10240, 1152), (200, 20480, 512)]


@pytest.mark.parametrize("n,N,K", SHAPES)
def test_gemm_against_oracle(lib, n, N, K):
    x, packed, scales, codes, sc = _case(n * 7 + N + K, n, N, K)
    y = binding.gemm_w4a16(torch.from_numpy(x).cuda(), packed, scales)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    got = y.cpu().numpy().astype(np.float64)
    ref = ogemv.gemv_ref(x, codes, sc)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref).max()
    assert err <= 1e-2 * rms
    assert err <= _acc_tol(K) * rms, "max err %.3e rms vs bound %.3e" % (err / rms, _acc_tol(K))


def test_gemm_one_hot_reads_single_weights_exactly(lib):
    # row t of x is one-hot at column k_t: y[t][r] = q[r][k_t] * s (exact in fp32)
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
    want = codes[:, ks].astype(np.float32) * sc[:, ks // 128].astype(np.float32)
    assert np.array_equal(y, want.T)


@pytest.mark.parametrize("n,N,K", [(77, 512, 3584), (300, 2560, 8192)])
def test_gemm_is_deterministic(lib, n, N, K):
    x, packed, scales, codes, sc = _case(3, n, N, K)
    xd = torch.from_numpy(x).cuda()
    a = binding.gemm_w4a16(xd, packed, scales)
    b = binding.gemm_w4a16(xd, packed, scales)
    assert torch.equal(a, b)


def test_gemm_rejects_bad_shapes(lib):
    x = torch.zeros((4, 256), dtype=torch.float16, device="cuda")
    packed = torch.zeros((200, 32), dtype=torch.int32, device="cuda")
    scales = torch.zeros(200 * 2 + 8, dtype=torch.float16, device="cuda")
    with pytest.raises(binding.W4Error):
        binding.gemm_w4a16(x, packed, scales)   # N = 200 is not a multiple of 128
