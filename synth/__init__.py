"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module draws random numbers and lays them out; it holds none of the
method's arithmetic (no quantisation, packing, GEMV, attention or model math),
so both the CPU oracle's callers and the GPU path's callers may use it.

Every array comes from ``numpy.random.default_rng`` seeded with a list of
integers ``[seed, stream, ...]``, so any one tensor can be regenerated alone
(the full-size model is produced one matrix at a time and never held whole in
host memory).  Distributions follow the workloads the library is measured on:

* activations x ~ N(0, 1) fp16; weights W ~ N(0, 0.02) fp32;
* K/V pool entries and queries ~ N(0, 1) fp16; page tables are slices of one
  seeded permutation of the pool's page ids;
* model: embedding ~ N(0, 0.02) fp16, RMSNorm weights 1 + N(0, 0.02) fp16,
  q/k/v biases ~ N(0, 0.02) fp16, INT4 source weights ~ N(0, 0.02) fp32.

The pages' own workload is Qwen2.5-Coder-7B with trained weights, which are not
available; these seeded tensors of the same shapes stand in for it.
"""

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# stream ids: keep every tensor family on its own random stream
_X, _W, _BIAS, _Q, _KPOOL, _VPOOL, _PERM, _EMBED, _NORM, _KPRE, _VPRE, _TOK = range(12)

PAGE_TOKENS = 16

QWEN25_7B = dict(hidden=3584, ffn=18944, n_layers=28, n_q_heads=28, n_kv_heads=4,
                 head_dim=128, vocab=152064, rms_eps=1e-6, rope_theta=1e6)

# A small model of the same structure for fast end-to-end parity checks.
TINY = dict(hidden=512, ffn=1280, n_layers=2, n_q_heads=4, n_kv_heads=2,
            head_dim=128, vocab=1000, rms_eps=1e-6, rope_theta=1e6)

# The seven projections of one layer, (name, N, K).
LAYER_PROJECTIONS = [("q", 3584, 3584), ("k", 512, 3584), ("v", 512, 3584),
                     ("o", 3584, 3584), ("gate", 18944, 3584), ("up", 18944, 3584),
                     ("down", 3584, 18944)]


def rng(*key):
    return np.random.default_rng([int(k) % (1 << 32) for k in key])


def normal_f32(key, shape, std):
    a = rng(*key).standard_normal(shape, dtype=np.float32)
    a *= np.float32(std)
    return a


def normal_f16(key, shape, std=1.0, mean=0.0):
    a = rng(*key).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if mean != 0.0:
        a += np.float32(mean)
    return a.astype(np.float16)


# --------------------------------------------------------------------------- GEMV

def gemv_x(seed, m, k):
    """Activations x fp16 [M][K] ~ N(0, 1)."""
    return normal_f16((seed, _X, m, k), (m, k))


def gemv_w(seed, n, k, tag=0):
    """Weights W fp32 [N][K] ~ N(0, 0.02)."""
    return normal_f32((seed, _W, tag, n, k), (n, k), 0.02)


def gemv_bias(seed, n, tag=0):
    return normal_f16((seed, _BIAS, tag, n), (n,), 0.02)


# ---------------------------------------------------------------------- attention

def page_table(seed, lens, num_pages, max_pages=None):
    """Disjoint slices of one seeded permutation of 0..num_pages-1.

    Row b holds ceil(lens[b]/16) page ids for sequence b; unused entries are
    padded with the first page of the row (never read)."""
    need = [max(1, math.ceil(int(L) / PAGE_TOKENS)) for L in lens]
    if max_pages is None:
        max_pages = max(need)
    if sum(need) > num_pages:
        raise ValueError("pool too small for these contexts")
    perm = rng(seed, _PERM, num_pages).permutation(num_pages).astype(np.int32)
    pt = np.zeros((len(lens), max_pages), dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[off:off + n]
        pt[b, n:] = perm[off]
        off += n
    return pt


def kv_pool(seed, num_pages, hkv, d=128):
    """K and V pools fp16 [P][Hkv][16][D] ~ N(0, 1)."""
    shape = (num_pages, hkv, PAGE_TOKENS, d)
    return normal_f16((seed, _KPOOL, num_pages), shape), normal_f16((seed, _VPOOL, num_pages), shape)


def queries(seed, b, hq, d=128):
    return normal_f16((seed, _Q, b, hq), (b, hq, d))


# -------------------------------------------------------------------------- model

MATRICES = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def matrix_shape(cfg, name):
    h, f = cfg["hidden"], cfg["ffn"]
    kv = cfg["n_kv_heads"] * cfg["head_dim"]
    return {"wq": (h, h), "wk": (kv, h), "wv": (kv, h), "wo": (h, h),
            "wg": (f, h), "wu": (f, h), "wd": (h, f), "lm_head": (cfg["vocab"], h)}[name]


def model_matrix(seed, cfg, layer, name):
    """One INT4 source matrix (fp32 ~ N(0, 0.02)); layer -1 is the LM head."""
    idx = ("lm_head",) + MATRICES
    shape = matrix_shape(cfg, name)
    return normal_f32((seed, _W, 1000 + layer, idx.index(name)), shape, 0.02)


def model_small_tensors(seed, cfg):
    """Embedding, norms and biases: everything that is not an INT4 matrix."""
    h = cfg["hidden"]
    kv = cfg["n_kv_heads"] * cfg["head_dim"]
    out = {"embed": normal_f16((seed, _EMBED), (cfg["vocab"], h), 0.02),
           "final_norm": normal_f16((seed, _NORM, -1, 0), (h,), 0.02, 1.0),
           "layers": []}
    for li in range(cfg["n_layers"]):
        out["layers"].append({
            "ln1": normal_f16((seed, _NORM, li, 1), (h,), 0.02, 1.0),
            "ln2": normal_f16((seed, _NORM, li, 2), (h,), 0.02, 1.0),
            "bq": normal_f16((seed, _BIAS, 1000 + li, 0), (h,), 0.02),
            "bk": normal_f16((seed, _BIAS, 1000 + li, 1), (kv,), 0.02),
            "bv": normal_f16((seed, _BIAS, 1000 + li, 2), (kv,), 0.02),
        })
    return out


def model_all_matrices(seed, cfg, threads=None):
    """Yield (layer, name, W fp32) for every INT4 matrix, layer -1 = LM head,
    generating a few at a time on worker threads (NumPy releases the GIL)."""
    jobs = [(li, n) for li in range(cfg["n_layers"]) for n in MATRICES] + [(-1, "lm_head")]
    threads = threads or min(16, len(os.sched_getaffinity(0)))
    with ThreadPoolExecutor(threads) as ex:
        window = []
        for job in jobs:
            window.append((job, ex.submit(model_matrix, seed, cfg, job[0], job[1])))
            if len(window) >= threads:
                (li, n), fut = window.pop(0)
                yield li, n, fut.result()
        for (li, n), fut in window:
            yield li, n, fut.result()


def prefill_kv(seed, cfg, layer, length):
    """K and V rows for tokens 0..length-1 of one layer, fp16 [L][Hkv][D] ~ N(0, 1).

    The decode benchmark starts from a cache filled directly with these rows
    rather than from a prompt pass, so its numbers do not depend on one."""
    shape = (length, cfg["n_kv_heads"], cfg["head_dim"])
    return normal_f16((seed, _KPRE, layer, length), shape), normal_f16((seed, _VPRE, layer, length), shape)


def start_token(seed, vocab):
    return int(rng(seed, _TOK, vocab).integers(0, vocab))


def prompt_tokens(seed, n, vocab):
    """A prompt of n token ids, uniform over the vocabulary (int32 [n]).

    The pages time the first token of a coding prompt whose text they do not
    give; uniform random ids of the chosen length stand in for it."""
    return rng(seed, _TOK, vocab, n).integers(0, vocab, size=n).astype(np.int32)
