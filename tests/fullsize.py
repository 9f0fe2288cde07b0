"""The 7B-shaped model for the slow full-size GPU tests.

One pass over the seeded fp32 matrices builds both sides: each matrix is
packed on the GPU by the library (``pack_int4_g128``) and, independently,
quantised on the host by the oracle (``oracle.quant.quantize_g128``, on worker
threads).  Neither side reads the other's codes; the fp32 matrices are dropped
as soon as both have them, so host memory holds only the oracle's int8 codes
(about 7 GB).
"""

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import synth
from int4_weight_only_w4a16_gb300 import model as gmodel
from oracle import model as omodel
from oracle import quant as oquant


def enough_host_memory(gib):
    try:
        return os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE") >= gib * (1 << 30)
    except (ValueError, OSError):
        return False


def build_pair(seed, max_context, num_pages, threads=None):
    """(cfg, GPU Decoder, oracle DecodeModel, page table) of the 7B shape."""
    cfg = dict(synth.QWEN25_7B)
    small = synth.model_small_tensors(seed, cfg)
    pt = synth.page_table(seed, [max_context], num_pages, max_context // 16)[0]
    threads = threads or max(1, min(8, len(os.sched_getaffinity(0)) // 2))
    pool = ThreadPoolExecutor(threads)
    pending, done = [], []

    def matrices():
        for li, name, w in synth.model_all_matrices(seed, cfg):
            pending.append((li, name, pool.submit(oquant.quantize_g128, w)))
            while len(pending) > 2 * threads:   # bound the fp32 matrices held by queued jobs
                done.append(_finish(pending.pop(0)))
            yield li, name, w

    try:
        dec = gmodel.build_decoder(cfg, small, matrices(), pt, num_pages=num_pages, max_context=max_context)
        while pending:
            done.append(_finish(pending.pop(0)))
    finally:
        pool.shutdown(wait=True)
    w = dict(small)
    w["layers"] = [dict(small["layers"][li]) for li in range(cfg["n_layers"])]
    for li, name, ql in done:
        if li < 0:
            w["lm_head"] = ql
        else:
            w["layers"][li][name] = ql
    return cfg, dec, omodel.DecodeModel(cfg, w), pt


def _finish(job):
    li, name, fut = job
    codes, scales = fut.result()
    return li, name, omodel.QuantLinear.from_codes(codes, scales)


def empty_cache(cfg, max_context):
    shape = (max_context, cfg["n_kv_heads"], cfg["head_dim"])
    return ([np.zeros(shape, np.float16) for _ in range(cfg["n_layers"])],
            [np.zeros(shape, np.float16) for _ in range(cfg["n_layers"])])


def rel_err(got, ref):
    """(max |got - ref|, rms of the difference), both relative to rms(ref)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    d = got - ref
    return float(np.abs(d).max() / rms), float(np.sqrt(np.mean(d ** 2)) / rms)
