"""W4A8 GEMV: INT4 weights against activations quantised to INT8 per group.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "How To Build Your Own LLM Runtime From Scratch | daily.dev", the
question on INT8-activation dp4a for Hopper GEMV shapes, and "How to build
your own LLM runtime from scratch (Towards Data Science)", "Two more honest
findings": the builder quantised the activations to INT8 before each GEMV
and multiplied them with the INT4 codes by dp4a; on Hopper that path lost to
fp16 activations.  The pages give no activation quantiser, so this oracle
takes the reading that mirrors the weight rule of ``quant``: per activation
row and 128-group along K, in fp32,

    s = max|x| / 127            (IEEE fp32 division; s = 0 for an all-zero group)
    q = clamp(rint(x / s), -127, 127)       (round half to even)

and the product is computed exactly:

    y[m][n] = sum_g  s_w[n][g] * s_x[m][g] * sum_{k in g} q_w[n][k] * q_x[m][k]

with the inner sums in integers and the rest in float64.  Where floating
point decides an integer (q_x), it is decided in fp32, as the kernel does.
"""

import numpy as np

GROUP = 128


def quantize_activations_g128(x):
    """x: [M][K] fp16 values.  Returns (q int8 [M][K], s float32 [M][K/128])."""
    x32 = np.atleast_2d(np.asarray(x)).astype(np.float16).astype(np.float32)
    m, k = x32.shape
    xg = x32.reshape(m, k // GROUP, GROUP)
    amax = np.max(np.abs(xg), axis=2)
    s = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = np.rint(xg / safe[:, :, None]).astype(np.float32)
    q = np.clip(q, -127, 127)
    q = np.where(s[:, :, None] > 0, q, 0)
    return q.astype(np.int8).reshape(m, k), s


def gemv_w4a8_ref(x, codes, scales):
    """x: [M][K] fp16; codes int8 [N][K] and scales fp16 [N][K/128] as from
    ``quant.quantize_g128``.  Returns float64 [M][N]."""
    q, s = quantize_activations_g128(x)
    m, k = q.shape
    n = codes.shape[0]
    g = k // GROUP
    dots = np.einsum("mgk,ngk->mng", q.reshape(m, g, GROUP).astype(np.int64),
                     np.asarray(codes).reshape(n, g, GROUP).astype(np.int64))
    return np.einsum("mng,ng,mg->mn", dots.astype(np.float64), np.asarray(scales).astype(np.float64),
                     s.astype(np.float64))
