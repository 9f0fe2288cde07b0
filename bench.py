#!/usr/bin/env python
"""Benchmark: graph-captured single-token decode of a 28-layer Qwen2.5-7B-shaped
model with INT4 group-128 weights (W4A16 GEMVs + paged GQA attention).

One step = one generated token = the whole hot path: embedding, 28 x [RMSNorm +
fused QKV GEMV + bias, RoPE + paged KV append, paged attention, O GEMV +
residual, RMSNorm + gate/up GEMV + SwiGLU, down GEMV + residual], final RMSNorm,
INT4 LM head (vocab 152064), greedy argmax.  The KV cache starts with 512
prefilled tokens; every 256 generated tokens the position is reset to 512, so
the timed tokens cover the 512..767 context range of the workload.

Prints ONE JSON line (rank 0).  `value` = algorithmic HBM bytes per token /
time per token (GB/s); ms_per_step is ms per token.  Weights (3.65 GB per
token) are far larger than the 129 MB L2, so no flush is needed between steps.

--impl reference times the float64 CPU oracle on a bounded sample of the same
workload (it is the only reference available: the pages publish no code).
"""

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "INT4 GEMV & paged-attn achieved HBM GB/s (% of peak); decode ms/token"
PREFILL = 512
RUN_TOKENS = 256
SEED = 2024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the time-to-first-token leg of the default run")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config kernel measurements (C0, C1, C2, C4)")
    ap.add_argument("--profile", action="store_true",
                    help="set up, run --warmup eager steps and one more eager step, then exit (for ncu)")
    ap.add_argument("--profile-layers", type=int, default=0, metavar="L",
                    help="with --profile: a model of the same shape cut to L layers (a small ncu case)")
    ap.add_argument("--profile-gemv", metavar="M,N,K",
                    help="pack one seeded N x K matrix, run --warmup + 1 gemv_w4a16 calls at batch M, exit (for ncu)")
    ap.add_argument("--gemv-variant", type=int, default=0,
                    help="w4_gemv_tune variant for --profile-gemv (0 default, 1 mma.sync kernel at batch 1 too, "
                         "2 W4A8, 3 tcgen05 kernel at every batch)")
    ap.add_argument("--profile-attention", metavar="B,L",
                    help="standalone paged decode attention over B sequences of L tokens (28/4 heads, a 4096-page "
                         "pool per sequence): --warmup untimed and --steps timed calls, exit (for ncu)")
    ap.add_argument("--profile-gemm", metavar="n,N,K",
                    help="pack one seeded N x K matrix, run --warmup untimed and --steps timed gemm_w4a16 calls on n rows")
    ap.add_argument("--prefill-bench", type=int, metavar="N", default=0,
                    help="time the prompt pass (time to first token) for an N-token prompt on the 7B shape")
    ap.add_argument("--container-bench", action="store_true",
                    help="write the full-size model to the own container format, load it back; print timings")
    return ap.parse_args()


# ------------------------------------------------------------------ bytes model

def gemv_bytes(n, k, x_bytes=2, out_bytes=2, extra=0):
    """Algorithmic bytes of one GEMV: packed codes + fp16 scales + input + output."""
    return n * k // 2 + n * (k // 128) * 2 + k * x_bytes + n * out_bytes + extra


def layer_bytes(cfg, ctx):
    h, f = cfg["hidden"], cfg["ffn"]
    kv = cfg["n_kv_heads"] * cfg["head_dim"]
    nqkv = h + 2 * kv
    b = {}
    # fp32 x + gamma in, bias, roped q out, k/v rows into the pools
    b["qkv"] = gemv_bytes(nqkv, h, x_bytes=4 + 2, extra=nqkv * 2)
    b["attention"] = attention_bytes(cfg, ctx)
    b["o"] = gemv_bytes(h, h, out_bytes=8)                                     # fp32 residual r+w
    b["gate_up"] = 2 * (f * h // 2 + f * (h // 128) * 2) + h * 6 + f * 2
    b["down"] = gemv_bytes(h, f, out_bytes=8)
    return b


def attention_bytes(cfg, ctx, batch=1):
    hkv, d, hq = cfg["n_kv_heads"], cfg["head_dim"], cfg["n_q_heads"]
    pages = math.ceil(ctx / 16)
    return batch * (2 * 2 * hkv * d * ctx + 4 * pages + 2 * 2 * hq * d)


def step_bytes(cfg, ctx):
    lb = layer_bytes(cfg, ctx)
    h = cfg["hidden"]
    lm = cfg["vocab"] * h // 2 + cfg["vocab"] * (h // 128) * 2 + h * 6 + 8
    return cfg["n_layers"] * sum(lb.values()) + lm + h * 2 + h * 4


def mean_step_bytes(cfg):
    # tokens at positions 512..767: the context of the token at p is p + 1
    return sum(step_bytes(cfg, PREFILL + i + 1) for i in range(RUN_TOKENS)) / RUN_TOKENS


# ---------------------------------------------------------------------- helpers

def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class Clocks:
    """nvidia-smi sampler running during the timed region."""

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        mx = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("gemv_tma.cuh", "gemv.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "int4_weight_only_w4a16_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch of the gate/up kernel from the committed ncu summary,
    valid only while the kernel source is the one that was profiled."""
    path = os.path.join(ROOT, "profiles", "gate_up_gemv_traffic.txt")
    try:
        vals = {}
        with open(path) as f:
            for line in f:
                if "=" in line and not line.startswith("#"):
                    k, v = line.split("=", 1)
                    vals[k.strip()] = v.strip()
        if vals.get("source_hash") == kernel_source_hash():
            return float(vals["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# -------------------------------------------------------------------- CPU oracle

def oracle_layer_sample(seed, cfg, rows_fraction=1.0):
    """Oracle objects for a bounded sample of the step: decoder layer 0 (its 7
    INT4 projections and paged attention over the 513-token context) plus the LM
    head, restricted to a fraction of each matrix's rows when asked."""
    import numpy as np

    import synth
    from oracle import model as omodel

    c1 = dict(cfg)
    c1["n_layers"] = 1
    small = synth.model_small_tensors(seed, cfg)
    small["layers"] = small["layers"][:1]
    w = dict(small)
    w["layers"] = [dict(small["layers"][0])]
    for name in synth.MATRICES:
        w["layers"][0][name] = synth.model_matrix(seed, cfg, 0, name)
    w["lm_head"] = synth.model_matrix(seed, cfg, -1, "lm_head")
    if rows_fraction < 1.0:
        # keep the shapes consistent: sample rows of the LM head only; the
        # layer's matrices stay whole (their outputs feed each other)
        n = max(1, int(cfg["vocab"] * rows_fraction))
        w["lm_head"] = w["lm_head"][:n]
    om = omodel.DecodeModel(c1, w)
    k, v = synth.prefill_kv(seed, cfg, 0, PREFILL)
    kc = np.zeros((PREFILL + 1, cfg["n_kv_heads"], cfg["head_dim"]), np.float16)
    vc = np.zeros_like(kc)
    kc[:PREFILL], vc[:PREFILL] = k, v
    lm_rows = w["lm_head"].shape[0]
    bytes_ = sum(layer_bytes(cfg, PREFILL + 1).values()) + lm_rows * cfg["hidden"] // 2 + \
        lm_rows * (cfg["hidden"] // 128) * 2
    return om, kc, vc, bytes_


def oracle_timings(seed, cfg):
    """Seconds the float64 oracle takes per call on this host, per workload:
    C0 the k_proj GEMV, C1 each projection of a layer, C2 paged attention at
    each context length, and C3 one decode step, composed from a measured
    decoder layer (its 7 projections and attention at context 513) and the
    measured LM head as 28 layers + 1 LM head (a whole 7B step is a minute of
    CPU work; its layers are identical in cost).  Quantisation is not timed."""
    import numpy as np

    import synth
    from oracle import gemv as ogemv, model as omodel, paged as opaged, quant as oquant

    def best_of(fn, n=2):
        ts = []
        for _ in range(n):
            t0 = time.perf_counter()
            fn()
            ts.append(time.perf_counter() - t0)
        return min(ts)

    out = {}
    x = synth.gemv_x(seed, 1, 3584)[0]
    codes, sc = oquant.quantize_g128(synth.gemv_w(seed, 512, 3584))
    out["c0_k_proj_s"] = best_of(lambda: ogemv.gemv_ref(x, codes, sc))
    c1 = {}
    for i, (name, n, k) in enumerate(synth.LAYER_PROJECTIONS):
        xi = synth.gemv_x(seed + i, 1, k)[0]
        ci, si = oquant.quantize_g128(synth.gemv_w(seed + i, n, k))
        c1[name] = best_of(lambda: ogemv.gemv_ref(xi, ci, si), 1)
        del ci, si
    c1["total"] = sum(c1.values())
    out["c1_layer_s"] = c1
    c2 = {}
    kp, vp = synth.kv_pool(seed, 512, 4)
    for L in (1, 15, 16, 17, 1000, 4096):
        pt = synth.page_table(seed, [L], 512, (L + 15) // 16)
        q = synth.queries(seed, 1, 28)
        c2["L%d" % L] = best_of(lambda: opaged.paged_attention_ref(q, kp, vp, pt, [L], 1.0 / math.sqrt(128)), 1)
    out["c2_attention_s"] = c2
    om, kc, vc, _ = oracle_layer_sample(seed, cfg)
    t_sample = best_of(lambda: omodel.decode_step_ref(om, [kc.copy()], [vc.copy()], 1, PREFILL), 1)
    h = synth.gemv_x(seed, 1, cfg["hidden"])[0]
    t_lm = best_of(lambda: om.lm_head(h), 1)
    out["c3_step_s"] = cfg["n_layers"] * (t_sample - t_lm) + t_lm
    out["c3_layer_s"] = t_sample - t_lm
    out["c3_lm_head_s"] = t_lm
    return out, om, kc, vc


_ONE_THREAD = r"""
import json, os, sys
sys.path.insert(0, %r)
import bench, synth
print("ONE_THREAD_JSON " + json.dumps(bench.oracle_timings(%d, dict(synth.QWEN25_7B))[0]))
"""


def cpu_baseline(seed, cfg):
    """The oracle on this host's cores over a bounded sample of the step
    (decoder layer 0 + the full LM head), plus per-workload oracle timings at
    all cores and at one BLAS thread (a child process started with one-thread
    BLAS settings)."""
    from oracle import model as omodel
    cores = len(os.sched_getaffinity(0))
    timings, om, kc, vc = oracle_timings(seed, cfg)
    nbytes = oracle_layer_sample_bytes(cfg)
    t0 = time.perf_counter()
    omodel.decode_step_ref(om, [kc], [vc], 1, PREFILL)
    dt = time.perf_counter() - t0
    one = None
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, "-c", _ONE_THREAD % (ROOT, seed)], env=env, capture_output=True,
                           text=True, timeout=600)
        for line in r.stdout.splitlines():
            if line.startswith("ONE_THREAD_JSON "):
                one = json.loads(line[len("ONE_THREAD_JSON "):])
    except (subprocess.SubprocessError, ValueError, OSError):
        one = None
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "float64 NumPy oracle: decoder layer 0 (7 INT4 projections + paged attention at "
                      "context 513) + the full 152064-row INT4 LM head, %.2f s per sample" % dt,
            "seconds_per_sample": dt,
            "seconds_per_call": {"threads": cores, **timings},
            "seconds_per_call_1_thread": one}


def oracle_layer_sample_bytes(cfg):
    return sum(layer_bytes(cfg, PREFILL + 1).values()) + cfg["vocab"] * cfg["hidden"] // 2 + \
        cfg["vocab"] * (cfg["hidden"] // 128) * 2


# ----------------------------------------------------------- per-config kernels

def _time_graph(fn, reps, replays=20):
    """Capture `reps` calls of fn() in a CUDA graph, replay it `replays` times
    (each between its own CUDA events on the capturing stream) and return the
    median us per call."""
    import numpy as np
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(replays)]
    for e0, e1 in ev:
        e0.record()
        g.replay()
        e1.record()
    torch.cuda.synchronize()
    return float(np.median([e0.elapsed_time(e1) for e0, e1 in ev])) * 1e3 / reps


def run_configs(dev):
    """The other workloads as kernel measurements (each call's inputs rotate
    through copies that together exceed L2, so bytes come from HBM):
    C0 k_proj GEMV, C1 the seven projections of a layer, C2 paged attention
    over contexts 1..4096, C4 gate/up/down at batch 1..16 and attention over
    8 x 32768 tokens."""
    import numpy as np
    import torch

    import synth
    from int4_weight_only_w4a16_gb300 import binding as bd

    l2 = 129e6
    out = {}

    def gemv_case(n, k, m, seed):
        nbytes_w = n * k // 2 + n * (k // 128) * 2
        copies = int(min(512, max(2, np.ceil(3 * l2 / nbytes_w))))
        mats = []
        for c in range(copies):
            w = torch.randn((n, k), device=dev) * 0.02
            mats.append(bd.pack_int4_g128(w))
            del w
        x = torch.from_numpy(synth.gemv_x(seed, m, k)).to(dev)
        y = torch.empty((m, n), dtype=torch.float16, device=dev)
        ws = bd.gemv_workspace(m, n, k, dev)

        def call(i=0):
            pk, sc = mats[i % copies]
            bd.gemv_w4a16(x, pk, sc, out=y, workspace=ws)
        us = _time_graph(call, copies)
        nb = nbytes_w + 2 * m * k + 2 * m * n
        del mats
        torch.cuda.empty_cache()
        return {"us": round(us, 2), "gbs": round(nb / us / 1e3, 1), "bytes": nb}

    out["c0_k_proj_512x3584"] = gemv_case(512, 3584, 1, 1)
    out["c1_layer"] = {name: gemv_case(n, k, 1, 10 + i) for i, (name, n, k) in enumerate(synth.LAYER_PROJECTIONS)}
    c1 = out["c1_layer"]
    tot_b = sum(v["bytes"] for v in c1.values())
    tot_us = sum(v["us"] for v in c1.values())
    c1["total"] = {"us": round(tot_us, 2), "gbs": round(tot_b / tot_us / 1e3, 1), "bytes": tot_b}

    batch = {}
    for m in (1, 2, 4, 8, 16):
        for name, n, k in (("gate", 18944, 3584), ("down", 3584, 18944)):
            batch["%s_m%d" % (name, m)] = gemv_case(n, k, m, 100 + m)
    out["c4_batched_gemv"] = batch
    # the same shapes on the opt-in tcgen05 kernel (w4_gemv_tune(3)), measured beside the defaults
    bd.gemv_tune(3)
    try:
        tc = {}
        for m in (1, 8, 16):
            for name, n, k in (("gate", 18944, 3584), ("down", 3584, 18944)):
                tc["%s_m%d" % (name, m)] = gemv_case(n, k, m, 100 + m)
        out["c4_batched_gemv_tcgen05"] = tc
    finally:
        bd.gemv_tune(0)

    def attn_case(b, L, num_pages, rot):
        kp, vp = synth.kv_pool(7, num_pages, 4)
        kp, vp = torch.from_numpy(kp).to(dev), torch.from_numpy(vp).to(dev)
        pages = (L + 15) // 16
        perm = torch.from_numpy(synth.page_table(7, [num_pages * 16], num_pages)[0]).to(dev)
        pts = []
        for r in range(rot):   # disjoint page sets per call so no call's pages are still in L2
            base = (r * b * pages) % max(1, num_pages - b * pages + 1)
            pts.append(perm[base:base + b * pages].reshape(b, pages).contiguous())
        q = torch.from_numpy(synth.queries(7, b, 28)).to(dev)
        lens = torch.full((b,), L, dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        ws = bd.attention_workspace(b, 28, 4, L, dev)

        def call(i=0):
            bd.paged_decode_attention(q, kp, vp, pts[i % rot], lens, L, out=o, workspace=ws)
        us = _time_graph(call, rot)
        nb = attention_bytes(synth.QWEN25_7B, L, b)
        return {"us": round(us, 2), "gbs": round(nb / us / 1e3, 1), "bytes": nb}

    out["c2_attention"] = {"L%d" % L: attn_case(1, L, 4096, 16) for L in (1, 15, 16, 17, 1000, 4096)}
    out["c4_attention_b8_L32768"] = attn_case(8, 32768, 16384 + 512, 1)
    return out


# ------------------------------------------------------------------ replicas

def replica_env():
    """(world size, rank, local rank) of a torchrun launch; (1, 0, 0) alone."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x, world, device):
    """The largest of every rank's x: the job's time is its slowest replica's."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_unit, ms_per_unit, world):
    """Whole-job throughput: every replica moves bytes_per_unit per unit, the job
    takes the slowest replica's time."""
    return world * bytes_per_unit / (ms_per_unit * 1e-3) / 1e9


# ------------------------------------------------------------------------ ours

def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import synth
    from int4_weight_only_w4a16_gb300 import binding, build as gbuild, model as gmodel

    world, rank, local = replica_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gbuild.build()

    cfg = dict(synth.QWEN25_7B)
    if args.profile and args.profile_layers > 0:
        cfg["n_layers"] = min(cfg["n_layers"], args.profile_layers)
    max_context = PREFILL + RUN_TOKENS + 16
    max_pages = max_context // 16
    num_pages = 2 * max_pages
    t_setup = time.perf_counter()
    small = synth.model_small_tensors(SEED, cfg)
    pt = synth.page_table(SEED, [max_context], num_pages, max_pages)[0]
    dec = gmodel.build_decoder(cfg, small, synth.model_all_matrices(SEED, cfg), pt, num_pages=num_pages,
                               max_context=max_context, device=dev)
    for li in range(cfg["n_layers"]):
        k, v = synth.prefill_kv(SEED, cfg, li, PREFILL)
        gmodel.fill_kv(dec, li, k, v)
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t_setup
    tok0 = synth.start_token(SEED, cfg["vocab"])
    stream = torch.cuda.current_stream()
    if args.profile:
        dec.set_state(tok0, PREFILL)
        for _ in range(args.warmup + 1):
            dec.step(with_logits=False)
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        print(json.dumps({"profile_run": "ok", "steps": args.warmup + 1, "launches_per_step": dec.launches_per_step,
                          "our_setup_launches": 7 * cfg["n_layers"] + 1 + cfg["n_layers"] + 1}))
        dec.close()
        return

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    dec.set_state(tok0, PREFILL)
    dec.capture(with_logits=False)
    for i in range(args.warmup):
        if i % RUN_TOKENS == 0:
            dec.pos.fill_(PREFILL)
        dec.replay()
    barrier()

    # ---- timed region: K graph-replayed tokens
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.25)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for i in range(args.steps):
        if i % RUN_TOKENS == 0:
            dec.pos.fill_(PREFILL)
        dec.replay()
    e1.record(stream)
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    assert binding.device_error() == 0, "device error during the timed region"
    final_tok = int(dec.token.item())

    bytes_tok = mean_step_bytes(cfg)
    value = job_gbs(bytes_tok, ms, world)
    peak, peak_kind = peaks()

    # ---- e2e: public API with host buffers (token H2D, graph, token D2H, sync)
    host_in = torch.empty(1, dtype=torch.int32, pin_memory=True)
    host_out = torch.empty(1, dtype=torch.int32, pin_memory=True)
    host_in[0] = tok0
    k_e2e = min(args.steps, 256)
    dec.pos.fill_(PREFILL)
    barrier()
    t0 = time.perf_counter()
    for i in range(k_e2e):
        dec.token.copy_(host_in, non_blocking=True)
        dec.replay()
        host_out.copy_(dec.token, non_blocking=True)
        stream.synchronize()
        host_in[0] = host_out[0]
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / k_e2e, world, dev)

    # ---- eager step (same kernels, one launch each) for the launch-overhead comparison
    dec.release_graph()
    dec.pos.fill_(PREFILL)
    for _ in range(3):
        dec.step(with_logits=False)
    barrier()
    e0.record(stream)
    for i in range(32):
        dec.step(with_logits=False)
    e1.record(stream)
    barrier()
    eager_ms = e0.elapsed_time(e1) / 32

    # ---- per-kernel live timing: each kernel's 28 per-layer launches (one per
    # layer, so 28 different weight sets: nothing stays in L2) captured in a
    # CUDA graph and replayed between CUDA events on the launching stream
    kernels = {}
    lb = layer_bytes(cfg, PREFILL + 1)
    lm_bytes = cfg["vocab"] * cfg["hidden"] // 2 + cfg["vocab"] * (cfg["hidden"] // 128) * 2 + cfg["hidden"] * 6
    dec.pos.fill_(PREFILL)
    for name in ("qkv", "attention", "o", "gate_up", "down", "lm_head"):
        layers = [-1] if name == "lm_head" else list(range(cfg["n_layers"]))
        for li in layers:  # eager warm-up, also sets any per-kernel attributes
            dec.launch_kernel(name, li, with_logits=False)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for li in layers:
                dec.launch_kernel(name, li, with_logits=False)
        g.replay()
        reps = 20 if name != "lm_head" else 50
        barrier()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        barrier()
        us = e0.elapsed_time(e1) * 1e3 / (reps * len(layers))
        nb = lm_bytes if name == "lm_head" else lb[name]
        kernels[name] = {"us": round(us, 3), "bytes": nb, "gbs": round(nb / (us * 1e-6) / 1e9, 1)}
        del g
    assert binding.device_error() == 0
    launches = dec.launches_per_step
    prefill = None if args.no_prefill else prefill_measure(dec, cfg, dev, stream)
    dec.close()

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    dom = kernels["gate_up"]
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "ms_per_token": round(ms, 4),
        "tok_per_s": round(world * 1e3 / ms, 1), "pct_of_peak": round(100 * value / world / peak, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int4*f16->f32",
        "data": "synthetic: seeded N(0,0.02) INT4-quantised weights, N(0,1) fp16 KV prefill (trained "
                "Qwen2.5-Coder-7B weights are not available)",
        "config": arm_config(cfg, world, args),
        "roofline": {"bound": "hbm", "kernel": "gate_up GEMV + SwiGLU (2 x 18944x3584 INT4)",
                     "achieved": dom["gbs"], "peak": peak, "peak_kind": peak_kind + " hbm_gbs (burst)",
                     "unit": "GB/s", "frac": round(dom["gbs"] / peak, 3), "traffic": recorded_traffic(),
                     "algorithmic_bytes_per_launch": dom["bytes"], "us_per_launch": dom["us"]},
        "e2e": {"value": round(job_gbs(bytes_tok, e2e_ms, world), 1), "unit": "GB/s",
                "ms_per_token": round(e2e_ms, 4), "h2d_bytes_per_step": 4, "d2h_bytes_per_step": 4},
        "gpu_launches": launches * args.steps,
        "launches_per_step": launches,
        "eager_ms_per_token": round(eager_ms, 4),
        "clocks": clk,
        "kernels": kernels,
        "setup_s": round(setup_s, 1),
        "final_token": final_tok,
    }
    if prefill is not None:
        line["prefill"] = prefill
    if not args.no_configs:
        line["configs"] = run_configs(dev)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(SEED, cfg)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def prefill_measure(dec, cfg, dev, stream, n=512, reps=5):
    """After the decode measurements: time to first token for an n-token prompt
    on an empty cache through the public API (overwrites cache rows 0..n-1), and
    the prompt pass's dominant kernel -- the tcgen05 W4A16 GEMM on the gate+up
    shape -- timed alone with CUDA events against the measured bf16 peak."""
    import torch

    import synth
    from int4_weight_only_w4a16_gb300 import binding

    tokens = torch.from_numpy(synth.prompt_tokens(SEED, n, cfg["vocab"])).to(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        dec.prefill(tokens)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        dec.prefill(tokens)
    e1.record(stream)
    torch.cuda.synchronize()
    ttft = e0.elapsed_time(e1) / reps
    assert binding.device_error() == 0 and int(dec.pos.item()) == n
    h, f = cfg["hidden"], cfg["ffn"]
    w = torch.empty((2 * f, h), dtype=torch.float32, device=dev).normal_(0.0, 0.02,
                                                                         generator=torch.Generator(dev).manual_seed(SEED))
    packed, scales = binding.pack_int4_g128(w)
    del w
    x = torch.empty((n, h), dtype=torch.float32, device=dev).normal_(
        generator=torch.Generator(dev).manual_seed(SEED + 1)).half()
    y = torch.empty((n, 2 * f), dtype=torch.float32, device=dev)
    ws = torch.empty(max(binding.load().w4_gemm_workspace_size(n, 2 * f, h), 16), dtype=torch.uint8, device=dev)
    for _ in range(3):
        binding.gemm_w4a16(x, packed, scales, out=y, workspace=ws)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(20):
        binding.gemm_w4a16(x, packed, scales, out=y, workspace=ws)
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / 20
    tflops = 2.0 * n * 2 * f * h / (us * 1e-6) / 1e12
    peak = bf16_peak()
    return {"workload": "prompt pass, %d synthetic tokens, empty cache, same 28-layer model" % n,
            "ttft_ms": round(ttft, 3), "prompt_tok_s": round(n / ttft * 1e3, 1),
            "dominant_kernel": {"kernel": "tcgen05 W4A16 GEMM, gate+up %dx%d, %d rows" % (2 * f, h, n),
                                "bound": "tensor", "us": round(us, 2), "achieved": round(tflops, 1),
                                "peak": peak[0], "peak_kind": peak[1], "unit": "TFLOP/s",
                                "frac": round(tflops / peak[0], 3)}}


def bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            v = json.load(fh).get("bf16_tflops")
        if v:
            return float(v), "measured bf16_tflops (burst)"
    except (OSError, ValueError):
        pass
    return 1900.0, "fallback bf16 burst"


def arm_config(cfg, world, args):
    """The workload both arms report (the reference arm times a bounded sample of it)."""
    return {"workload": "decode step, 28-layer Qwen2.5-7B shape (hidden 3584, FFN 18944, GQA 28/4, "
                        "head_dim 128, vocab 152064), INT4 g128 W4A16, paged KV 16-token pages, "
                        "prefill 512, 256-token runs, CUDA graph",
            "bytes_per_token": int(mean_step_bytes(cfg)), "l2": "no flush: 3.65 GB of weights per step >> 129 MB L2",
            "seed": SEED, "parallelism": "replicas" if world > 1 else "single GPU"}


# ------------------------------------------------------------------- reference

def run_reference(args):
    world, rank, _ = replica_env()
    if rank != 0:
        return
    import synth
    from oracle import model as omodel
    cfg = dict(synth.QWEN25_7B)
    # each step: decoder layer 0 + a row sample of the LM head, sized so that
    # warmup + steps stay within about two minutes
    budget_s = 120.0
    om, kc, vc, nbytes = oracle_layer_sample(SEED, cfg, rows_fraction=0.02)
    t0 = time.perf_counter()
    omodel.decode_step_ref(om, [kc], [vc], 1, PREFILL)
    one = time.perf_counter() - t0
    n_total = args.warmup + args.steps
    steps = args.steps
    if one * n_total > budget_s:
        steps = max(1, int(budget_s / one) - args.warmup)
    for _ in range(max(0, args.warmup - 1)):
        omodel.decode_step_ref(om, [kc], [vc], 1, PREFILL)
    t0 = time.perf_counter()
    for _ in range(steps):
        omodel.decode_step_ref(om, [kc], [vc], 1, PREFILL)
    dt = (time.perf_counter() - t0) / steps
    value = nbytes / dt / 1e9
    cores = len(os.sched_getaffinity(0))
    sample = ("float64 NumPy oracle: decoder layer 0 (7 INT4 projections + paged attention at context 513) + "
              "2%% of the LM head rows per step; %d of %d requested steps timed" % (steps, args.steps))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": arm_config(cfg, world, args),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def profile_gemv(args):
    """One standalone GEMV shape, called --warmup + 1 times (a small, ncu-friendly workload)."""
    import torch

    import synth
    from int4_weight_only_w4a16_gb300 import binding as bd

    m, n, k = (int(v) for v in args.profile_gemv.split(","))
    bd.load()
    bd.gemv_tune(args.gemv_variant)
    w = torch.from_numpy(synth.gemv_w(SEED, n, k)).cuda()
    packed, scales = bd.pack_int4_g128(w)
    del w
    x = torch.from_numpy(synth.gemv_x(SEED, m, k)).cuda()
    y = torch.empty((m, n), dtype=torch.float16, device="cuda")
    ws = bd.gemv_workspace(m, n, k)
    for _ in range(args.warmup + 1):
        bd.gemv_w4a16(x, packed, scales, out=y, workspace=ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_gemv": [m, n, k], "variant": args.gemv_variant, "calls": args.warmup + 1}))


def profile_attention(args):
    """Standalone paged decode attention, B sequences of L tokens (the C2/C4 inputs):
    --warmup calls, then --steps calls timed with CUDA events (ncu-friendly with small counts)."""
    import torch

    import synth
    from int4_weight_only_w4a16_gb300 import binding as bd

    b, L = (int(v) for v in args.profile_attention.split(","))
    pages = (L + 15) // 16
    num_pages = max(4096, b * pages)
    kp, vp = synth.kv_pool(7, num_pages, 4)
    kp, vp = torch.from_numpy(kp).cuda(), torch.from_numpy(vp).cuda()
    perm = torch.from_numpy(synth.page_table(7, [num_pages * 16], num_pages)[0]).cuda()
    pt = perm[:b * pages].reshape(b, pages).contiguous()
    q = torch.from_numpy(synth.queries(7, b, 28)).cuda()
    lens = torch.full((b,), L, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    ws = bd.attention_workspace(b, 28, 4, L, "cuda")
    for _ in range(args.warmup):
        bd.paged_decode_attention(q, kp, vp, pt, lens, L, out=out, workspace=ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        bd.paged_decode_attention(q, kp, vp, pt, lens, L, out=out, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    assert bd.device_error() == 0
    us = e0.elapsed_time(e1) * 1e3 / max(1, args.steps)
    nb = attention_bytes(synth.QWEN25_7B, L, b)
    print(json.dumps({"profile_attention": [b, L], "warmup": args.warmup, "calls": args.steps, "us": round(us, 2),
                      "gbs": round(nb / us / 1e3, 1)}))


def profile_gemm(args):
    """One standalone prompt-pass GEMM shape: --warmup calls, then --steps calls timed with CUDA events
    (ncu-friendly with small counts)."""
    import torch

    import synth
    from int4_weight_only_w4a16_gb300 import binding as bd

    n, nn, k = (int(v) for v in args.profile_gemm.split(","))
    bd.load()
    w = torch.from_numpy(synth.gemv_w(SEED, nn, k)).cuda()
    packed, scales = bd.pack_int4_g128(w)
    del w
    x = torch.from_numpy(synth.gemv_x(SEED, n, k)).cuda()
    y = torch.empty((n, nn), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(bd.load().w4_gemm_workspace_size(n, nn, k), 16), dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        bd.gemm_w4a16(x, packed, scales, out=y, workspace=ws)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    calls = max(1, args.steps)
    e0.record(stream)
    for _ in range(calls):
        bd.gemm_w4a16(x, packed, scales, out=y, workspace=ws)
    e1.record(stream)
    torch.cuda.synchronize()
    assert bd.device_error() == 0
    us = e0.elapsed_time(e1) * 1e3 / calls
    print(json.dumps({"profile_gemm": [n, nn, k], "warmup": args.warmup, "calls": calls, "us": round(us, 2),
                      "tflops": round(2.0 * n * nn * k / (us * 1e-6) / 1e12, 1)}))


def container_bench(args):
    """Write the 28-layer model's packed weights to a container file and load
    them back through the mapped reader and pinned staging (page cache warm:
    the file was just written)."""
    import shutil

    import torch

    import synth
    from int4_weight_only_w4a16_gb300 import binding, build as gbuild, model as gmodel

    gbuild.build()
    cfg = dict(synth.QWEN25_7B)
    max_context = PREFILL + RUN_TOKENS + 16
    num_pages = 2 * (max_context // 16)
    small = synth.model_small_tensors(SEED, cfg)
    pt = synth.page_table(SEED, [max_context], num_pages, max_context // 16)[0]
    dec = gmodel.build_decoder(cfg, small, synth.model_all_matrices(SEED, cfg), pt, num_pages=num_pages,
                               max_context=max_context)
    torch.cuda.synchronize()
    d = tempfile.mkdtemp()
    path = os.path.join(d, "qwen25_7b_shape.w4c")
    try:
        t0 = time.perf_counter()
        gmodel.save_container(path, dec)
        t_write = time.perf_counter() - t0
        size = os.path.getsize(path)
        ref = [(n, t.clone()) for n, t in gmodel.decoder_tensors(dec)[:4]]
        dec.close()
        del dec
        torch.cuda.empty_cache()
        t0 = time.perf_counter()
        c = binding.Container(path, verify=True)
        t_verify = time.perf_counter() - t0
        c.close()
        t0 = time.perf_counter()
        dec2 = gmodel.load_decoder(path, pt, num_pages=num_pages, max_context=max_context)
        t_load = time.perf_counter() - t0
        same = all(torch.equal(a, b) for (_, a), (_, b) in zip(ref, gmodel.decoder_tensors(dec2)[:4]))
        dec2.close()
    finally:
        shutil.rmtree(d, ignore_errors=True)
    print(json.dumps({"container_bench": {
        "file_bytes": size, "tensors": 4 + 13 * cfg["n_layers"],
        "write_s": round(t_write, 2), "write_gbs": round(size / t_write / 1e9, 2),
        "open_verify_crc_s": round(t_verify, 2), "open_verify_gbs": round(size / t_verify / 1e9, 2),
        "load_to_device_s": round(t_load, 2), "load_gbs": round(size / t_load / 1e9, 2),
        "first_tensors_bitwise_equal": same,
        "note": "page cache warm (file just written); load = mmap + pinned staging + cudaMemcpyAsync, no verify"}}))


def prefill_bench(args):
    """Time to first token: one prompt pass of N synthetic tokens through the
    28-layer 7B shape (prompt rows at positions 0..N-1, empty cache), ending in
    the first greedy token.  Timed with CUDA events over --steps passes after
    --warmup, and once more end to end through the public API (prompt copied
    from pinned host memory, token read back)."""
    import torch

    import synth
    from int4_weight_only_w4a16_gb300 import binding, build as gbuild, model as gmodel

    gbuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n = args.prefill_bench
    cfg = dict(synth.QWEN25_7B)
    max_context = max(1024, (n + 16 + 15) // 16 * 16)
    num_pages = max_context // 16 + 8
    small = synth.model_small_tensors(SEED, cfg)
    pt = synth.page_table(SEED, [max_context], num_pages, max_context // 16)[0]
    dec = gmodel.build_decoder(cfg, small, synth.model_all_matrices(SEED, cfg), pt, num_pages=num_pages,
                               max_context=max_context, device=dev)
    tokens = torch.from_numpy(synth.prompt_tokens(SEED, n, cfg["vocab"])).to(dev)
    stream = torch.cuda.current_stream()
    if args.profile:   # warm passes, then one pass inside cudaProfilerStart/Stop (ncu --profile-from-start off)
        for _ in range(args.warmup):
            dec.prefill(tokens)
        torch.cuda.synchronize()
        torch.cuda.profiler.start()
        dec.prefill(tokens)
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
        assert binding.device_error() == 0
        print(json.dumps({"prefill_profile_run": "ok", "prompt_tokens": n, "warmup": args.warmup}))
        dec.close()
        return
    for _ in range(args.warmup):
        dec.prefill(tokens)
    torch.cuda.synchronize()
    clocks = Clocks(0)
    clocks.start()
    time.sleep(0.25)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        dec.prefill(tokens)
    e1.record(stream)
    torch.cuda.synchronize()
    ms, clk, tok = e0.elapsed_time(e1) / args.steps, clocks.stop(), int(dec.token.item())
    assert binding.device_error() == 0, "device error during the prompt pass"
    assert int(dec.pos.item()) == n
    # e2e: prompt copied from pinned host memory, first token read back, per pass
    host_tok = torch.from_numpy(synth.prompt_tokens(SEED, n, cfg["vocab"])).pin_memory()
    host_out = torch.empty(1, dtype=torch.int32, pin_memory=True)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        tokens.copy_(host_tok, non_blocking=True)
        dec.prefill(tokens)
        host_out.copy_(dec.token, non_blocking=True)
        stream.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    h, f = cfg["hidden"], cfg["ffn"]
    kv = cfg["n_kv_heads"] * cfg["head_dim"]
    w_layer = (h + 2 * kv) * h + h * h + 2 * f * h + h * f
    flops = 2.0 * n * w_layer * cfg["n_layers"] + 2.0 * cfg["vocab"] * h
    print(json.dumps({"prefill_bench": {
        "workload": "Qwen2.5-7B shape, random INT4 weights, prompt of %d synthetic tokens, empty cache" % n,
        "prompt_tokens": n, "steps": args.steps, "warmup": args.warmup,
        "ttft_ms": round(ms, 3), "prompt_tok_s": round(n / ms * 1e3, 1),
        "gemm_tflops_effective": round(flops / (ms * 1e-3) / 1e12, 1),
        "e2e_ttft_ms": round(e2e_ms, 3), "h2d_bytes": 4 * n, "d2h_bytes": 4,
        "first_token": tok,
        "clocks": clk}}))
    dec.close()


def main():
    args = parse()
    if args.prefill_bench:
        prefill_bench(args)
        return
    if args.container_bench:
        container_bench(args)
        return
    if args.profile_gemv:
        profile_gemv(args)
        return
    if args.profile_gemm:
        profile_gemm(args)
        return
    if args.profile_attention:
        profile_attention(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
