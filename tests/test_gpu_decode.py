"""GPU decode step (eager and CUDA graph) against the oracle's decode step.

Logits must match within 2e-2 * rms(ref).  With random weights nearby logits
can be close, so the check is teacher-forced: every step feeds the oracle's
token to both sides, and a differing argmax is accepted only when the
oracle's top-2 gap is inside that tolerance.
"""

import numpy as np
import pytest
import torch

import fullsize
import synth
from int4_weight_only_w4a16_gb300 import model as gmodel
from oracle import model as omodel

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _weights(seed, cfg):
    small = synth.model_small_tensors(seed, cfg)
    mats = [(li, n, synth.model_matrix(seed, cfg, li, n)) for li in range(cfg["n_layers"]) for n in synth.MATRICES]
    mats.append((-1, "lm_head", synth.model_matrix(seed, cfg, -1, "lm_head")))
    return small, mats


def _oracle_model(cfg, small, mats):
    w = dict(small)
    w["layers"] = [dict(small["layers"][li]) for li in range(cfg["n_layers"])]
    for li, n, m in mats:
        if li < 0:
            w["lm_head"] = m
        else:
            w["layers"][li][n] = m
    return omodel.DecodeModel(cfg, w)


def _setup(cfg, seed, prefill, max_context, num_pages):
    small, mats = _weights(seed, cfg)
    max_pages = max_context // 16
    pt = synth.page_table(seed, [max_context], num_pages, max_pages)[0]
    dec = gmodel.build_decoder(cfg, small, mats, pt, num_pages=num_pages, max_context=max_context)
    kc, vc = [], []
    for li in range(cfg["n_layers"]):
        k, v = synth.prefill_kv(seed, cfg, li, prefill)
        gmodel.fill_kv(dec, li, k, v)
        kk = np.zeros((max_context, cfg["n_kv_heads"], cfg["head_dim"]), np.float16)
        vv = np.zeros_like(kk)
        kk[:prefill], vv[:prefill] = k, v
        kc.append(kk)
        vc.append(vv)
    torch.cuda.synchronize()
    return dec, _oracle_model(cfg, small, mats), kc, vc


def _compare(got, ref, tok_gpu, tok_ref):
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref).max()
    assert np.all(np.isfinite(got))
    assert err <= TOL * rms, "logits max err %.3e > %.1e * rms %.3e" % (err, TOL, rms)
    if tok_gpu != tok_ref:
        assert ref[tok_ref] - ref[tok_gpu] <= TOL * rms


def _teacher_forced(dec, om, kc, vc, tok, pos0, steps, use_graph):
    if use_graph:
        dec.capture()
    for s in range(steps):
        pos = pos0 + s
        dec.token.fill_(tok)
        if use_graph:
            dec.replay()
        else:
            dec.step()
        torch.cuda.synchronize()
        got = dec.logits.cpu().numpy().astype(np.float64)
        tok_gpu = int(dec.token.item())
        assert int(dec.pos.item()) == pos + 1
        ref, tok_ref = omodel.decode_step_ref(om, kc, vc, tok, pos)
        _compare(got, ref, tok_gpu, tok_ref)
        tok = tok_ref


@pytest.fixture(scope="module")
def tiny(lib):
    cfg = dict(synth.TINY)
    dec, om, kc, vc = _setup(cfg, 9, prefill=8, max_context=128, num_pages=32)
    yield cfg, dec, om, kc, vc
    dec.close()


def test_tiny_eager_steps_cross_page_boundaries(lib, tiny):
    cfg, dec, om, kc, vc = tiny
    dec.set_state(3, 8)
    _teacher_forced(dec, om, kc, vc, 3, 8, 20, use_graph=False)
    assert lib.device_error() == 0


def test_tiny_graph_equals_eager_bitwise(lib, tiny):
    cfg, dec, om, kc, vc = tiny
    seq = {}
    for mode in ("eager", "graph"):
        dec.set_state(5, 40)
        if mode == "graph":
            dec.capture()
        toks, logits = [], []
        for _ in range(6):
            dec.replay() if mode == "graph" else dec.step()
            toks.append(int(dec.token.item()))
            logits.append(dec.logits.clone())
        seq[mode] = (toks, torch.stack(logits))
        assert int(dec.pos.item()) == 46
    assert seq["eager"][0] == seq["graph"][0]
    assert torch.equal(seq["eager"][1], seq["graph"][1])
    dec.release_graph()


def test_tiny_graph_teacher_forced_against_oracle(lib, tiny):
    cfg, dec, om, kc, vc = tiny
    # positions 8..27 were written by the eager test with the same tokens; rewrite from 28 on
    dec.set_state(7, 60)
    kc2 = [k.copy() for k in kc]
    vc2 = [v.copy() for v in vc]
    # the oracle's cache rows 8..59 must hold what the GPU cache holds: replay them eagerly
    # through the oracle with the GPU's own tokens is not allowed, so refill that range fresh:
    for li in range(cfg["n_layers"]):
        k, v = synth.prefill_kv(99, cfg, li, 60)
        gmodel.fill_kv(dec, li, k, v)
        kc2[li][:60], vc2[li][:60] = k, v
    torch.cuda.synchronize()
    _teacher_forced(dec, om, kc2, vc2, 7, 60, 8, use_graph=True)
    dec.release_graph()


@pytest.mark.parametrize("max_context,prefill", [(560, 500), (784, 700), (1408, 1300), (3072, 2990)])
def test_tiny_long_context_cluster_attention(lib, max_context, prefill):
    # capacities of 33 to 64 pages (35, 49: one page per warp in clusters of 9 and 13
    # CTAs, the full-size decode's plan) and past 64 pages (the decode attention's
    # splits form one cluster of up to 16 CTAs; 88 pages: two-page rings; 192 pages:
    # three pages per warp in four-page rings), with every page but the one receiving
    # the new row loaded while the QKV kernel runs; teacher-forced across page
    # boundaries, eager and graph
    cfg = dict(synth.TINY)
    dec, om, kc, vc = _setup(cfg, 31, prefill=prefill, max_context=max_context, num_pages=max_context // 16 + 24)
    try:
        dec.set_state(5, prefill)
        _teacher_forced(dec, om, kc, vc, 5, prefill, 10, use_graph=False)
        kc2 = [k.copy() for k in kc]
        vc2 = [v.copy() for v in vc]
        for li in range(cfg["n_layers"]):
            k, v = synth.prefill_kv(32, cfg, li, prefill + 10)
            gmodel.fill_kv(dec, li, k, v)
            kc2[li][:prefill + 10], vc2[li][:prefill + 10] = k, v
        torch.cuda.synchronize()
        dec.set_state(9, prefill + 10)
        _teacher_forced(dec, om, kc2, vc2, 9, prefill + 10, 10, use_graph=True)
        assert lib.device_error() == 0
    finally:
        dec.release_graph()
        dec.close()


def test_launch_count(lib, tiny):
    cfg, dec, *_ = tiny
    assert dec.launches_per_step == 5 * cfg["n_layers"] + 2


def test_two_sequences_share_one_model(lib, tiny):
    # one weight set, two caches (w4_kv handles) with their own pools, page tables
    # and positions: the same prompt gives bitwise the same logits in both, and
    # steps interleaved across the two follow the oracle, each on its own cache
    cfg, dec, om, kc, vc = tiny
    pt2 = torch.from_numpy(synth.page_table(77, [128], 40, 8)[0]).cuda()
    seq = dec.new_sequence(pt2, num_pages=40, max_context=128)
    try:
        prompt = torch.from_numpy(synth.prompt_tokens(21, 30, cfg["vocab"])).cuda()
        dec.prefill(prompt)
        seq.prefill(prompt)
        torch.cuda.synchronize()
        assert torch.equal(dec.logits, seq.logits) and int(dec.token.item()) == int(seq.token.item())
        assert int(dec.pos.item()) == int(seq.pos.item()) == 30
        shape = (128, cfg["n_kv_heads"], cfg["head_dim"])
        caches = []
        for _ in range(2):
            k = [np.zeros(shape, np.float16) for _ in range(cfg["n_layers"])]
            v = [np.zeros(shape, np.float16) for _ in range(cfg["n_layers"])]
            omodel.prefill_ref(om, k, v, prompt.cpu().numpy(), 0)
            caches.append((k, v))
        toks = [(3, 900), (17, 5), (250, 250)]
        for s_i, (ta, tb) in enumerate(toks):
            for which, (obj, t) in enumerate(((dec, ta), (seq, tb))):
                obj.token.fill_(t)
                obj.step()
                torch.cuda.synchronize()
                assert int(obj.pos.item()) == 31 + s_i
                ref, tref = omodel.decode_step_ref(om, caches[which][0], caches[which][1], t, 30 + s_i)
                _compare(obj.logits.cpu().numpy().astype(np.float64), ref, int(obj.token.item()), tref)
        assert lib.device_error() == 0
    finally:
        seq.close()


def _decoder_with_lm_head(lm_fp32, seed=41):
    """The tiny model with a chosen fp32 LM head, an 8-row cache, and the oracle beside it."""
    cfg = dict(synth.TINY)
    small, mats = _weights(seed, cfg)
    mats = [m for m in mats if m[0] >= 0] + [(-1, "lm_head", lm_fp32)]
    pt = synth.page_table(seed, [64], 8, 4)[0]
    dec = gmodel.build_decoder(cfg, small, mats, pt, num_pages=8, max_context=64)
    kc, vc = [], []
    for li in range(cfg["n_layers"]):
        k, v = synth.prefill_kv(seed, cfg, li, 8)
        gmodel.fill_kv(dec, li, k, v)
        kk = np.zeros((64, cfg["n_kv_heads"], cfg["head_dim"]), np.float16)
        vv = np.zeros_like(kk)
        kk[:8], vv[:8] = k, v
        kc.append(kk)
        vc.append(vv)
    torch.cuda.synchronize()
    return cfg, dec, _oracle_model(cfg, small, mats), kc, vc


def _one_step(dec, tok, pos):
    dec.set_state(tok, pos)
    dec.step()
    torch.cuda.synchronize()
    return dec.logits.cpu().numpy(), int(dec.token.item())


def test_greedy_ties_go_to_the_lowest_index(lib):
    # greedy sampling takes the lowest index among equal maximal logits
    cfg = dict(synth.TINY)
    v, h = cfg["vocab"], cfg["hidden"]
    row = synth.gemv_w(41, 1, h)[0]
    # every row the same: all logits bitwise equal, so the token is 0
    cfg, dec, om, kc, vc = _decoder_with_lm_head(np.tile(row, (v, 1)))
    try:
        logits, tok = _one_step(dec, 3, 8)
        assert lib.device_error() == 0
        assert np.all(logits == logits[0]) and tok == 0
    finally:
        dec.close()
    # rows 0..9 zero (logit 0, whatever the sign of the zero), rows 10.. one
    # repeated row (logit z): the token is 10 when z > 0 and 0 otherwise
    lm = np.tile(row, (v, 1))
    lm[:10] = 0.0
    cfg, dec, om, kc, vc = _decoder_with_lm_head(lm)
    try:
        logits, tok = _one_step(dec, 5, 8)
        assert lib.device_error() == 0
        ref, tok_ref = omodel.decode_step_ref(om, kc, vc, 5, 8)
        assert np.all(logits[:10] == 0) and np.all(logits[10:] == logits[10])
        z = ref[10]
        assert abs(z) > 1e-3 * np.sqrt(np.mean(ref ** 2))   # the sign is not a near-tie
        assert tok == tok_ref == (10 if z > 0 else 0)
        # the same with the zero rows' logits forced to -0 against +0 cannot
        # change the token: the key of -0 equals the key of +0
        assert np.sign(logits[10]) == np.sign(z)
    finally:
        dec.close()


def test_nan_logit_never_wins_and_is_flagged(lib):
    # a NaN scale in one LM-head row makes its logit NaN: the step flags
    # W4_DEVERR_NAN_LOGIT and the token is the argmax of the other rows
    cfg = dict(synth.TINY)
    lm = synth.model_matrix(43, cfg, -1, "lm_head")
    cfg, dec, om, kc, vc = _decoder_with_lm_head(lm, seed=43)
    try:
        bad = 7
        dec.w["lm_head"][1][bad, 0] = float("nan")
        scales = dec.w["lm_head"][1].cpu().numpy()
        om.lm_head = omodel.QuantLinear.from_codes(om.lm_head.codes, scales)
        logits, tok = _one_step(dec, 9, 8)
        assert lib.device_error() & 0x80
        ref, _ = omodel.decode_step_ref(om, kc, vc, 9, 8)
        assert np.isnan(logits[bad]) and np.isnan(ref[bad])
        ref[bad] = -np.inf
        keep = np.arange(cfg["vocab"]) != bad
        assert np.abs(logits[keep] - ref[keep]).max() <= TOL * np.sqrt(np.mean(ref[keep] ** 2))
        tok_ref = int(np.argmax(ref))
        if tok != tok_ref:
            assert ref[tok_ref] - ref[tok] <= TOL * np.sqrt(np.mean(ref[keep] ** 2))
        assert tok != bad
    finally:
        dec.close()


CHECKED_STEPS = (0, 1, 2, 127, 255)


@pytest.mark.slow
def test_full_size_decode_256_steps(lib):
    """28-layer Qwen2.5-7B shape, KV cache prefilled with 512 random rows, 256
    graph-replayed steps at positions 512..767.  The input token of every step
    is fixed in advance (teacher-forced: both sides consume the same inputs),
    so step i is row i of the oracle's block form over those tokens; the
    logits and greedy token of steps 0, 1, 2, 127 and 255 are checked."""
    if not fullsize.enough_host_memory(24):
        pytest.skip("the full-size oracle needs ~24 GiB of free host memory")
    ctx, pages, prefill, steps = 1024, 128, 512, 256
    cfg, dec, om, pt = fullsize.build_pair(2024, ctx, pages)
    kc, vc = fullsize.empty_cache(cfg, ctx)
    try:
        for li in range(cfg["n_layers"]):
            k, v = synth.prefill_kv(2024, cfg, li, prefill)
            gmodel.fill_kv(dec, li, k, v)
            kc[li][:prefill], vc[li][:prefill] = k, v
        tokens = synth.prompt_tokens(2024, steps, cfg["vocab"])
        dec.set_state(int(tokens[0]), prefill)
        dec.capture()
        got = {}
        for s in range(steps):
            dec.token.fill_(int(tokens[s]))
            dec.replay()
            if s in CHECKED_STEPS:
                torch.cuda.synchronize()
                got[s] = (dec.logits.cpu().numpy().astype(np.float64), int(dec.token.item()))
        torch.cuda.synchronize()
        assert int(dec.pos.item()) == prefill + steps
        assert lib.device_error() == 0
        pools = {li: (dec.w["layers"][li]["k_pool"].cpu().numpy(), dec.w["layers"][li]["v_pool"].cpu().numpy())
                 for li in (0, 13, cfg["n_layers"] - 1)}
    finally:
        dec.close()
    ref, toks = omodel.prefill_block_ref(om, kc, vc, tokens, prefill, logits_rows=CHECKED_STEPS)
    for r, s in enumerate(CHECKED_STEPS):
        print("step %d (position %d): logits max %.3e rms %.3e (x rms)"
              % ((s, prefill + s) + fullsize.rel_err(got[s][0], ref[r])))
    # the K/V rows the 256 steps appended: layer 0's come from one projection of the
    # embedding (the per-op bar), deeper layers' from the composition of the layers
    # below (the model bar)
    p_ = np.arange(prefill, prefill + steps)
    for li, (kp, vp) in pools.items():
        for which, pool, ref_c in (("k", kp, kc), ("v", vp, vc)):
            e = fullsize.rel_err(pool[pt[p_ // 16], :, p_ % 16, :], ref_c[li][prefill:prefill + steps])
            print("layer %d %s rows: max %.3e rms %.3e (x rms)" % ((li, which) + e))
            assert e[0] <= (1e-2 if li == 0 else TOL), (li, which, e)
    for r, s in enumerate(CHECKED_STEPS):
        _compare(got[s][0], ref[r], got[s][1], toks[r])


@pytest.mark.slow
def test_full_size_decode_repeats_bitwise(lib):
    """7B shape: a 512-token prompt pass and 24 graph-replayed decode steps, twice
    from the same state, give the same tokens and bitwise the same logits (the
    step's kernels run as programmatic dependents of each other; every merge adds
    in a fixed order)."""
    cfg = dict(synth.QWEN25_7B)
    small = synth.model_small_tensors(2025, cfg)
    pt = synth.page_table(2025, [1024], 80, 64)[0]
    dec = gmodel.build_decoder(cfg, small, synth.model_all_matrices(2025, cfg), pt, num_pages=80, max_context=1024)
    try:
        tokens = torch.from_numpy(synth.prompt_tokens(2025, 512, cfg["vocab"])).cuda()
        runs = []
        for r in range(2):
            dec.prefill(tokens, start_pos=0)
            torch.cuda.synchronize()
            if r == 0:
                dec.capture()
            toks, lg = [], []
            for _ in range(24):
                dec.replay()
                toks.append(int(dec.token.item()))
                lg.append(dec.logits.clone())
            runs.append((toks, torch.stack(lg).cpu()))
        assert lib.device_error() == 0
        assert runs[0][0] == runs[1][0]
        assert torch.equal(runs[0][1], runs[1][1])
        dec.release_graph()
    finally:
        dec.close()
