"""W4A16 GEMV, the plain definition: dequantise to float64, then matvec.

Source: "How to build your own LLM runtime from scratch (Towards Data Science)",
section "What it actually builds" (fused GEMVs for the Q/K/V/O projections and
the MLP gate/up/down over INT4 group-128 weights), and "How To Build Your Own
LLM Runtime From Scratch | daily.dev", third question (fp16 activations against
INT4-unpacked weights).

    y[m][n] = sum_k x[m][k] * q[n][k] * s[n][k/128]  (+ bias[n])  (+ residual[m][n])

computed in float64 from the fp16 activations and the codes/scales of
``quant.quantize_g128``.  The result is returned in float64; the GPU writes it
rounded to fp16, and the tests compare with max|err| <= 1e-2 * rms(ref).
"""

import numpy as np

from .quant import dequantize


def gemv_ref(x, codes, scales, bias=None, residual=None):
    """x: [M][K] or [K] (fp16 values); codes int8 [N][K]; scales fp16 [N][K/128].

    Returns float64 [M][N] (or [N] for a 1-D x).
    """
    x = np.asarray(x)
    one_d = x.ndim == 1
    x64 = np.atleast_2d(x).astype(np.float64)
    w64 = dequantize(codes, scales)
    y = x64 @ w64.T
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)[None, :]
    if residual is not None:
        y = y + np.atleast_2d(np.asarray(residual, dtype=np.float64))
    return y[0] if one_d else y


def gemv_rows_ref(x, codes, scales, rows, bias=None):
    """The same definition for a chosen subset of output rows only, so that a
    sample of a very large GEMV (the 152064-row LM head) can be checked one
    row at a time.  x: [K]; returns float64 [len(rows)]."""
    rows = np.asarray(rows)
    x64 = np.asarray(x).astype(np.float64)
    w64 = dequantize(np.asarray(codes)[rows], np.asarray(scales)[rows])
    y = w64 @ x64
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)[rows]
    return y
