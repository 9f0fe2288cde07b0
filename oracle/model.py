"""One greedy decode step of a Qwen2.5-7B-shaped model, plain float64 definition.

Source for the scope: "How to build your own LLM runtime from scratch (Towards
Data Science)", opening paragraph (decode-only engine for Qwen2.5-Coder-7B,
greedy sampling only) and section "What it actually builds" (INT4 group-128
weights, paged KV cache, fused Q/K/V/O and gate/up/down GEMVs).  The pages name
the model but not its block; the block below is the published Qwen2
architecture, which is the plain reading:

    x = E[token]
    for each layer:
        h = rmsnorm(x) * g1
        q, k, v = Wq h + bq, Wk h + bk, Wv h + bv
        q, k = rope(q, pos), rope(k, pos)          rotate-half, theta = 1e6
        append k, v at pos;  a = attention(q, K[0..pos], V[0..pos])
        x = x + Wo a
        h = rmsnorm(x) * g2
        x = x + Wd (silu(Wg h) * (Wu h))
    logits = Wlm (rmsnorm(x) * gf);  token' = argmax(logits), lowest index on ties

All arithmetic is float64.  Values are rounded to fp16 only where the W4A16
data format stores them as fp16 tensors: the activation fed to every GEMV (h, a
and silu(g)*u), the q/k/v projection outputs, the roped query and the K/V rows
kept in the cache.  The residual stream x and the logits stay float64.
"""

import numpy as np

from .quant import quantize_g128, dequantize
from .paged import attention_contiguous


def f16(a):
    """Round float64 values to the nearest fp16 (ties to even), back as float64."""
    return np.asarray(a, dtype=np.float64).astype(np.float16).astype(np.float64)


def rmsnorm(x, gamma, eps):
    """x / sqrt(mean(x^2) + eps) * gamma."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x) + eps) * np.asarray(gamma, dtype=np.float64)


def rope_inv_freq(head_dim, theta):
    """theta^(-2i/head_dim) for i = 0 .. head_dim/2 - 1."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return theta ** (-2.0 * i / head_dim)


def rope(vecs, pos, theta):
    """Rotate-half RoPE of every head vector in vecs [H][D] at position pos.

    Dimension i pairs with i + D/2 and turns by angle pos * theta^(-2i/D).
    """
    vecs = np.asarray(vecs, dtype=np.float64)
    d = vecs.shape[-1]
    half = d // 2
    ang = float(pos) * rope_inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    a, b = vecs[..., :half], vecs[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


class QuantLinear:
    """Codes and scales of one INT4 matrix, dequantised row-block by row-block.

    Built from the fp32 weights (quantised here), or from codes and scales
    already produced by ``quantize_g128`` (``QuantLinear.from_codes``)."""

    def __init__(self, w_fp32):
        self.codes, self.scales = quantize_g128(w_fp32)

    @classmethod
    def from_codes(cls, codes, scales):
        obj = cls.__new__(cls)
        obj.codes, obj.scales = np.asarray(codes), np.asarray(scales)
        return obj

    def __call__(self, x, row_block=8192):
        x64 = np.asarray(x, dtype=np.float64)
        n = self.codes.shape[0]
        y = np.empty(n, dtype=np.float64)
        for r0 in range(0, n, row_block):
            r1 = min(n, r0 + row_block)
            y[r0:r1] = dequantize(self.codes[r0:r1], self.scales[r0:r1]) @ x64
        return y

    def matmul(self, xs, row_block=4096):
        """Y[i][n] = sum_k xs[i][k] * W_deq[n][k] for every row i of xs [m][K]."""
        x64 = np.asarray(xs, dtype=np.float64)
        n = self.codes.shape[0]
        y = np.empty((x64.shape[0], n), dtype=np.float64)
        for r0 in range(0, n, row_block):
            r1 = min(n, r0 + row_block)
            y[:, r0:r1] = x64 @ dequantize(self.codes[r0:r1], self.scales[r0:r1]).T
        return y


class DecodeModel:
    """Weights in oracle form.  ``weights`` maps names to arrays:

    embed fp16 [V][H]; final_norm fp16 [H]; lm_head fp32 [V][H];
    layers: list of dicts with ln1, ln2 fp16 [H]; wq, wk, wv, wo, wg, wu, wd
    fp32 matrices; bq, bk, bv fp16 vectors.  fp32 matrices are quantised here
    (a matrix given as a QuantLinear is used as it is).
    """

    def __init__(self, cfg, weights):
        self.cfg = cfg
        self.embed = np.asarray(weights["embed"])
        self.final_norm = np.asarray(weights["final_norm"])
        self.lm_head = _linear(weights["lm_head"])
        self.layers = []
        for lw in weights["layers"]:
            layer = {}
            for name in ("ln1", "ln2", "bq", "bk", "bv"):
                layer[name] = np.asarray(lw[name])
            for name in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
                layer[name] = _linear(lw[name])
            self.layers.append(layer)


def _linear(w):
    """An fp32 matrix is quantised here; a QuantLinear is taken as it is."""
    return w if isinstance(w, QuantLinear) else QuantLinear(w)


def decode_step_ref(model, k_cache, v_cache, token, pos):
    """One decode step at position ``pos`` (0-based) for input ``token``.

    k_cache/v_cache: per layer, fp16 arrays [max_len][Hkv][D] holding tokens
    0..pos-1; row pos is written here.  Returns (logits float64 [V], argmax).
    """
    cfg = model.cfg
    hq, hkv, d = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    eps, theta = cfg["rms_eps"], cfg["rope_theta"]
    group = hq // hkv
    x = model.embed[int(token)].astype(np.float64)
    for li, layer in enumerate(model.layers):
        h = f16(rmsnorm(x, layer["ln1"], eps))
        q = f16(layer["wq"](h) + layer["bq"].astype(np.float64))
        k = f16(layer["wk"](h) + layer["bk"].astype(np.float64))
        v = f16(layer["wv"](h) + layer["bv"].astype(np.float64))
        q = f16(rope(q.reshape(hq, d), pos, theta))
        k = f16(rope(k.reshape(hkv, d), pos, theta))
        k_cache[li][pos] = k.astype(np.float16)
        v_cache[li][pos] = v.reshape(hkv, d).astype(np.float16)
        a = np.empty((hq, d), dtype=np.float64)
        for h_i in range(hq):
            g = h_i // group
            a[h_i], _ = attention_contiguous(
                q[h_i], k_cache[li][: pos + 1, g, :], v_cache[li][: pos + 1, g, :], 1.0 / np.sqrt(d))
        x = x + layer["wo"](f16(a.reshape(-1)))
        h = f16(rmsnorm(x, layer["ln2"], eps))
        m = f16(silu(layer["wg"](h)) * layer["wu"](h))
        x = x + layer["wd"](m)
    h = f16(rmsnorm(x, model.final_norm, eps))
    logits = model.lm_head(h)
    return logits, int(np.argmax(logits))


def prefill_ref(model, k_cache, v_cache, tokens, start=0):
    """Run a prompt: the decode step applied to each prompt token in turn.

    "How to build your own LLM runtime from scratch (Towards Data Science)",
    section "What the numbers say" (time to first token).  Prompt token i sits
    at position start + i and sees the cache rows 0 .. start + i, so the
    pass is causal by construction; the next input is always the prompt's
    next token, never a sampled one.  The caches must hold rows 0 .. start-1;
    rows start .. start+n-1 are written.  Returns (logits float64 [V] of the
    last prompt token, their argmax) -- the first generated token.
    """
    tokens = [int(t) for t in tokens]
    if not tokens:
        raise ValueError("prefill_ref: empty prompt")
    logits, tok = None, None
    for i, t in enumerate(tokens):
        logits, tok = decode_step_ref(model, k_cache, v_cache, t, start + i)
    return logits, tok


def rope_rows(vecs, positions, theta):
    """Rotate-half RoPE of vecs [n][H][D], row i at position positions[i]:
    the same rotation as ``rope`` with one angle set per row."""
    vecs = np.asarray(vecs, dtype=np.float64)
    d = vecs.shape[-1]
    half = d // 2
    ang = np.asarray(positions, dtype=np.float64)[:, None, None] * rope_inv_freq(d, theta)[None, None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = vecs[..., :half], vecs[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def rmsnorm_rows(x, gamma, eps):
    """``rmsnorm`` of every row of x [n][H]."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps) * np.asarray(gamma, dtype=np.float64)


def prefill_block_ref(model, k_cache, v_cache, tokens, start=0, logits_rows=None):
    """The prompt pass written as one block instead of a loop over tokens.

    Same definition as ``prefill_ref`` (the decode step of every prompt token,
    with the same fp16 rounding points), organised the way a prompt is
    evaluated at once: each projection is one matrix product over all n
    prompt rows, and attention scores every query row against all keys
    0 .. start+n-1 with an explicit causal mask -- row i, at position
    start + i, sees the keys at positions <= start + i ("How to build your own
    LLM runtime from scratch (Towards Data Science)", section "What the numbers
    say": the time to first token is this pass plus the first greedy token).

    Teacher-forced decode is the same computation: with the input tokens fixed
    in advance, step i of a decode run at positions start.. is row i here.

    k_cache/v_cache: per layer, fp16 [max_len][Hkv][D] holding rows
    0 .. start-1; rows start .. start+n-1 are written.  logits_rows: indices
    of the prompt rows whose logits are wanted (default: the last row).
    Returns (logits float64 [len(logits_rows)][V], argmax of each row, lowest
    index on ties).
    """
    cfg = model.cfg
    hq, hkv, d = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    eps, theta = cfg["rms_eps"], cfg["rope_theta"]
    group = hq // hkv
    tokens = np.asarray(tokens, dtype=np.int64)
    n = tokens.shape[0]
    if n == 0:
        raise ValueError("prefill_block_ref: empty prompt")
    rows = [n - 1] if logits_rows is None else [int(r) for r in logits_rows]
    pos = start + np.arange(n)
    causal = np.arange(start + n)[None, :] <= pos[:, None]            # [n][start + n]
    x = model.embed[tokens].astype(np.float64)                         # [n][H]
    for li, layer in enumerate(model.layers):
        h = f16(rmsnorm_rows(x, layer["ln1"], eps))
        q = f16(layer["wq"].matmul(h) + layer["bq"].astype(np.float64)).reshape(n, hq, d)
        k = f16(layer["wk"].matmul(h) + layer["bk"].astype(np.float64)).reshape(n, hkv, d)
        v = f16(layer["wv"].matmul(h) + layer["bv"].astype(np.float64)).reshape(n, hkv, d)
        q = f16(rope_rows(q, pos, theta))
        k = f16(rope_rows(k, pos, theta))
        k_cache[li][start:start + n] = k.astype(np.float16)
        v_cache[li][start:start + n] = v.astype(np.float16)
        keys = k_cache[li][:start + n].astype(np.float64)             # [start + n][Hkv][D]
        vals = v_cache[li][:start + n].astype(np.float64)
        a = np.empty((n, hq, d), dtype=np.float64)
        for h_i in range(hq):
            g = h_i // group
            scores = (q[:, h_i, :] @ keys[:, g, :].T) * (1.0 / np.sqrt(d))
            scores = np.where(causal, scores, -np.inf)
            e = np.exp(scores - scores.max(axis=1, keepdims=True))   # two passes: max, then exp / sum
            a[:, h_i, :] = (e / e.sum(axis=1, keepdims=True)) @ vals[:, g, :]
        x = x + layer["wo"].matmul(f16(a.reshape(n, hq * d)))
        h = f16(rmsnorm_rows(x, layer["ln2"], eps))
        m = f16(silu(layer["wg"].matmul(h)) * layer["wu"].matmul(h))
        x = x + layer["wd"].matmul(m)
    hf = f16(rmsnorm_rows(x[rows], model.final_norm, eps))
    logits = model.lm_head.matmul(hf)
    return logits, [int(np.argmax(r)) for r in logits]
