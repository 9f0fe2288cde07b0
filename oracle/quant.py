"""Symmetric group-wise INT4 quantisation (group 128) and the packed format.

Source: "How to build your own LLM runtime from scratch (Towards Data Science)",
section "What it actually builds": INT4 weights, symmetric, group-wise with
group size 128.  The pages name the scheme but print no formula; the plain
symmetric reading used here maps the largest magnitude of a group to code 7:

    s = fp16(max|w| / 7)                 one fp16 scale per (row, 128-group)
    q = clamp(rint(w / s), -8, 7)        codes, round half to even

The division uses the fp16-rounded scale widened to fp32, so that the product
q*s used at inference time is exactly what the codes were chosen against; all
of it is done in IEEE fp32 (NumPy float32 division is correctly rounded).  A
group whose scale is 0 (all-zero group, or max/7 below the fp16 range) gets
s = 0 and q = 0.

Packed format (this library's own; the pages' "ValueShuffle" layout is named
but never defined, so it is replaced):

    packed : uint32 [N][K/8], row-major; word j of row n holds k = 8j .. 8j+7
    nibble : u = q + 8  (offset binary, 0..15)
    slots  : element e (0..7) of the word sits in the 4-bit slot
             slot(e) = 4*(e % 2) + e // 2, i.e. bits [4*slot, 4*slot+4)
    scales : float16 [N][K/128], row-major

So elements (0,1) are slots (0,4), (2,3) are (1,5), (4,5) are (2,6) and (6,7)
are (3,7): each even/odd element pair lands in the low nibble of the two
16-bit halves of the word, shifted by 0, 4, 8 or 12 bits.
"""

import numpy as np

GROUP = 128
QMIN, QMAX = -8, 7


def slot_of_element(e):
    """4-bit slot that holds element e (0..7) of an 8-element word."""
    return 4 * (e % 2) + e // 2


class NonFiniteError(ValueError):
    """A weight is NaN/Inf, or a scale does not fit in fp16."""


def quantize_g128(w):
    """Quantise fp32 weights W[N][K] group-wise along K.

    Returns (codes int8 [N][K], scales float16 [N][K/128]).
    Raises NonFiniteError for a NaN/Inf weight or a scale above fp16's range.
    """
    w = np.asarray(w, dtype=np.float32)
    if w.ndim != 2 or w.shape[1] % GROUP != 0:
        raise ValueError("W must be [N][K] with K a multiple of 128")
    if not np.all(np.isfinite(w)):
        raise NonFiniteError("non-finite weight")
    n, k = w.shape
    g = w.reshape(n, k // GROUP, GROUP)
    amax = np.abs(g).max(axis=2)                       # fp32, exact
    s32 = amax / np.float32(7.0)                       # IEEE fp32 division
    with np.errstate(over="ignore"):
        s16 = s32.astype(np.float16)                   # round to nearest even
    if not np.all(np.isfinite(s16)):
        raise NonFiniteError("scale overflows fp16")
    sw = s16.astype(np.float32)[:, :, None]
    safe = np.where(sw == 0, np.float32(1.0), sw)
    q = np.rint(g / safe)                              # fp32 quotient, half-even
    q = np.clip(q, QMIN, QMAX)
    q = np.where(sw == 0, np.float32(0.0), q)
    return q.astype(np.int8).reshape(n, k), s16


def dequantize(codes, scales):
    """W_deq[n][k] = q[n][k] * s[n][k/128], in float64."""
    codes = np.asarray(codes)
    n, k = codes.shape
    s = np.asarray(scales, dtype=np.float64)
    return (codes.astype(np.float64).reshape(n, k // GROUP, GROUP) * s[:, :, None]).reshape(n, k)


def pack(codes):
    """int8 codes [N][K] in [-8, 7]  ->  uint32 words [N][K/8] (format above)."""
    codes = np.asarray(codes)
    n, k = codes.shape
    if k % 8 != 0:
        raise ValueError("K must be a multiple of 8")
    if codes.min(initial=0) < QMIN or codes.max(initial=0) > QMAX:
        raise ValueError("codes outside [-8, 7]")
    u = (codes.astype(np.int64) + 8).reshape(n, k // 8, 8)
    words = np.zeros((n, k // 8), dtype=np.uint64)
    for e in range(8):
        words |= (u[:, :, e].astype(np.uint64) << np.uint64(4 * slot_of_element(e)))
    return words.astype(np.uint32)


def unpack(words):
    """uint32 words [N][K/8]  ->  int8 codes [N][K] (inverse of pack)."""
    words = np.asarray(words, dtype=np.uint32)
    n, kw = words.shape
    out = np.empty((n, kw, 8), dtype=np.int8)
    for e in range(8):
        u = (words >> np.uint32(4 * slot_of_element(e))) & np.uint32(0xF)
        out[:, :, e] = (u.astype(np.int16) - 8).astype(np.int8)
    return out.reshape(n, kw * 8)
