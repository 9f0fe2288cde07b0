"""GPU prompt pass (w4_prefill) against the oracle's prompt pass.

The oracle runs its decode step over every prompt token in turn (and, at full
size, its block form of the same pass); the GPU runs all prompt rows at once
(W4A16 GEMMs on tcgen05 with exact INT4 codes, causal paged attention, the
decode step's LM head for the last row).  Checked:
the last row's logits within 2e-2 * rms (argmax equal, or a near-tie inside
that tolerance), every K/V row written into the paged pools within 1e-2 * rms
of the oracle's cache, the stream state (token, pos) the decode step continues
from, and prompts that span several pages with a ragged tail.
"""

import numpy as np
import pytest
import torch

import fullsize
import synth
from int4_weight_only_w4a16_gb300 import binding
from int4_weight_only_w4a16_gb300 import model as gmodel
from oracle import model as omodel

pytestmark = pytest.mark.gpu

TOL_LOGITS = 2e-2
TOL_KV = 1e-2
MAX_CONTEXT = 256
NUM_PAGES = 40


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


@pytest.fixture(scope="module")
def tiny(lib):
    cfg = dict(synth.TINY)
    small, mats = _weights(21, cfg)
    pt = synth.page_table(21, [MAX_CONTEXT], NUM_PAGES, MAX_CONTEXT // 16)[0]
    dec = gmodel.build_decoder(cfg, small, mats, pt, num_pages=NUM_PAGES, max_context=MAX_CONTEXT)
    om = _oracle_model(cfg, small, mats)
    yield cfg, dec, om, pt
    dec.close()


def _empty_cache(cfg):
    shape = (MAX_CONTEXT, cfg["n_kv_heads"], cfg["head_dim"])
    return ([np.zeros(shape, np.float16) for _ in range(cfg["n_layers"])],
            [np.zeros(shape, np.float16) for _ in range(cfg["n_layers"])])


def _gpu_rows(dec, pt, layer, which, p0, p1):
    """Cache rows p0..p1-1 of one layer gathered through the page table, [n][Hkv][D]."""
    pool = dec.w["layers"][layer][which].cpu().numpy()
    pos = np.arange(p0, p1)
    return pool[pt[pos // 16], :, pos % 16, :]


def _check_logits(got, ref, tok_gpu, tok_ref):
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref).max()
    assert err <= TOL_LOGITS * rms, "logits max err %.3e > %.0e * rms %.3e" % (err, TOL_LOGITS, rms)
    if tok_gpu != tok_ref:
        assert ref[tok_ref] - ref[tok_gpu] <= TOL_LOGITS * rms


def _check_cache(cfg, dec, pt, kc, vc, p0, p1):
    for li in range(cfg["n_layers"]):
        for which, ref_c in (("k_pool", kc), ("v_pool", vc)):
            got = _gpu_rows(dec, pt, li, which, p0, p1).astype(np.float64)
            ref = ref_c[li][p0:p1].astype(np.float64)
            rms = np.sqrt(np.mean(ref ** 2))
            err = np.abs(got - ref).max()
            assert err <= TOL_KV * rms, "layer %d %s rows %d..%d: err %.3e > %.0e * rms %.3e" % (
                li, which, p0, p1, err, TOL_KV, rms)


def _run(dec, tokens, start):
    dec.prefill(torch.from_numpy(tokens).cuda(), start_pos=start)
    torch.cuda.synchronize()
    return dec.logits.cpu().numpy().astype(np.float64), int(dec.token.item()), int(dec.pos.item())


@pytest.mark.parametrize("n", [1, 16, 37])
def test_prefill_against_oracle(lib, tiny, n):
    # one page exactly, a single token, and three pages with a ragged tail of 5
    cfg, dec, om, pt = tiny
    tokens = synth.prompt_tokens(5, n, cfg["vocab"])
    got, tok, pos = _run(dec, tokens, 0)
    assert lib.device_error() == 0
    assert pos == n
    kc, vc = _empty_cache(cfg)
    ref, tok_ref = omodel.prefill_ref(om, kc, vc, tokens, 0)
    _check_logits(got, ref, tok, tok_ref)
    _check_cache(cfg, dec, pt, kc, vc, 0, n)


def test_prefill_in_two_passes_and_decode_after(lib, tiny):
    # 20 tokens, then 25 more at start 20 (attending to the first pass's rows),
    # then three teacher-forced decode steps from the state the prompt left
    cfg, dec, om, pt = tiny
    tokens = synth.prompt_tokens(6, 45, cfg["vocab"])
    _run(dec, tokens[:20], 0)
    got, tok, pos = _run(dec, tokens[20:], 20)
    assert lib.device_error() == 0 and pos == 45
    kc, vc = _empty_cache(cfg)
    ref, tok_ref = omodel.prefill_ref(om, kc, vc, tokens, 0)
    _check_logits(got, ref, tok, tok_ref)
    _check_cache(cfg, dec, pt, kc, vc, 0, 45)
    t = tok_ref
    for s in range(3):
        dec.token.fill_(t)
        dec.step()
        torch.cuda.synchronize()
        assert int(dec.pos.item()) == 46 + s
        r, tr = omodel.decode_step_ref(om, kc, vc, t, 45 + s)
        _check_logits(dec.logits.cpu().numpy().astype(np.float64), r, int(dec.token.item()), tr)
        t = tr


def test_prefill_long_prompt_many_attention_splits(lib, tiny):
    # a long cached context and a short prompt: each query's attention is split
    # across CTAs and merged by the last one
    cfg, dec, om, pt = tiny
    tokens = synth.prompt_tokens(8, 200, cfg["vocab"])
    _run(dec, tokens[:197], 0)
    got, tok, pos = _run(dec, tokens[197:], 197)
    assert lib.device_error() == 0 and pos == 200
    kc, vc = _empty_cache(cfg)
    ref, tok_ref = omodel.prefill_ref(om, kc, vc, tokens, 0)
    _check_logits(got, ref, tok, tok_ref)
    _check_cache(cfg, dec, pt, kc, vc, 190, 200)


def test_prefill_rejects_bad_arguments(lib, tiny):
    cfg, dec, om, pt = tiny
    with pytest.raises(binding.W4Error):
        dec.prefill(torch.zeros(10, dtype=torch.int32, device="cuda"), start_pos=MAX_CONTEXT - 5)
    with pytest.raises(binding.W4Error):
        dec.prefill(torch.zeros(3, dtype=torch.int32, device="cuda"), start_pos=-1)
    with pytest.raises(binding.W4Error):
        dec.prefill(torch.zeros(0, dtype=torch.int32, device="cuda"))
    # an out-of-range token is recorded on the device, not read
    bad = torch.tensor([1, cfg["vocab"], 2], dtype=torch.int32, device="cuda")
    dec.prefill(bad)
    torch.cuda.synchronize()
    assert lib.device_error() & 0x40


def test_prefill_ignores_stale_nan_slots(lib, tiny):
    # every cache slot starts as NaN: the slots past the prompt in its last page
    # (and every unused page) must not reach the output
    cfg, dec, om, pt = tiny
    for lw in dec.w["layers"]:
        lw["k_pool"].fill_(float("nan"))
        lw["v_pool"].fill_(float("nan"))
    try:
        tokens = synth.prompt_tokens(9, 37, cfg["vocab"])
        got, tok, pos = _run(dec, tokens, 0)
        assert lib.device_error() == 0 and pos == 37
        kc, vc = _empty_cache(cfg)
        ref, tok_ref = omodel.prefill_ref(om, kc, vc, tokens, 0)
        _check_logits(got, ref, tok, tok_ref)
        _check_cache(cfg, dec, pt, kc, vc, 0, 37)
    finally:
        for lw in dec.w["layers"]:
            lw["k_pool"].zero_()
            lw["v_pool"].zero_()


def test_prefill_unaligned_start_across_key_splits(lib, tiny):
    # 5 cached tokens, then 150 prompt rows: the 16-row blocks straddle pages and
    # the key range is split across CTAs, so some rows see no key in a later split
    cfg, dec, om, pt = tiny
    tokens = synth.prompt_tokens(10, 155, cfg["vocab"])
    _run(dec, tokens[:5], 0)
    got, tok, pos = _run(dec, tokens[5:], 5)
    assert lib.device_error() == 0 and pos == 155
    kc, vc = _empty_cache(cfg)
    ref, tok_ref = omodel.prefill_ref(om, kc, vc, tokens, 0)
    _check_logits(got, ref, tok, tok_ref)
    _check_cache(cfg, dec, pt, kc, vc, 140, 155)


def test_prefill_whole_context_capacity(lib, tiny):
    # a prompt that fills the whole context capacity (every page of the table)
    cfg, dec, om, pt = tiny
    tokens = synth.prompt_tokens(11, MAX_CONTEXT, cfg["vocab"])
    got, tok, pos = _run(dec, tokens, 0)
    assert lib.device_error() == 0 and pos == MAX_CONTEXT
    kc, vc = _empty_cache(cfg)
    ref, tok_ref = omodel.prefill_ref(om, kc, vc, tokens, 0)
    _check_logits(got, ref, tok, tok_ref)
    _check_cache(cfg, dec, pt, kc, vc, MAX_CONTEXT - 20, MAX_CONTEXT)


MID = dict(hidden=1024, ffn=2048, n_layers=2, n_q_heads=8, n_kv_heads=2, head_dim=128, vocab=1000,
           rms_eps=1e-6, rope_theta=1e6)


def _pools(dec, cfg, layers):
    return {(li, w): dec.w["layers"][li][w].cpu().numpy() for li in layers for w in ("k_pool", "v_pool")}


def _assert_same_pass(dec, cfg, tokens, layers):
    """Run the same prompt pass again: logits, next token and the K/V pools must
    repeat bit for bit (every split and merge adds in a fixed order, and the
    kernels of the pass, launched as programmatic dependents, wait for their
    predecessors before touching their outputs)."""
    got0, tok0, pos0 = _run(dec, tokens, 0)
    pools0 = _pools(dec, cfg, layers)
    got1, tok1, pos1 = _run(dec, tokens, 0)
    pools1 = _pools(dec, cfg, layers)
    assert np.array_equal(got0, got1) and tok0 == tok1 and pos0 == pos1
    for key in pools0:
        assert np.array_equal(pools0[key], pools1[key]), key


def test_prefill_is_bitwise_reproducible(lib, tiny):
    cfg, dec, om, pt = tiny
    _assert_same_pass(dec, cfg, synth.prompt_tokens(9, 37, cfg["vocab"]), range(cfg["n_layers"]))
    assert lib.device_error() == 0


@pytest.mark.parametrize("n", [40, 300])
def test_prefill_split_k_merges_against_oracle(lib, n):
    # hidden 1024 / ffn 2048: every prompt-pass GEMM splits K (QKV and O partials added by
    # the RoPE kernel and the RMSNorm after O, down partials by the next RMSNorm and the
    # tail, gate/up by its SwiGLU merge kernel)
    cfg = dict(MID)
    small, mats = _weights(31, cfg)
    ctx = 320
    pt = synth.page_table(31, [ctx], 24, ctx // 16)[0]
    dec = gmodel.build_decoder(cfg, small, mats, pt, num_pages=24, max_context=ctx)
    try:
        om = _oracle_model(cfg, small, mats)
        tokens = synth.prompt_tokens(13, n, cfg["vocab"])
        got, tok, pos = _run(dec, tokens, 0)
        assert lib.device_error() == 0 and pos == n
        shape = (ctx, cfg["n_kv_heads"], cfg["head_dim"])
        kc = [np.zeros(shape, np.float16) for _ in range(cfg["n_layers"])]
        vc = [np.zeros(shape, np.float16) for _ in range(cfg["n_layers"])]
        ref, tok_ref = omodel.prefill_ref(om, kc, vc, tokens, 0)
        _check_logits(got, ref, tok, tok_ref)
        for li in range(cfg["n_layers"]):
            for which, ref_c in (("k_pool", kc), ("v_pool", vc)):
                pool = dec.w["layers"][li][which].cpu().numpy()
                p_ = np.arange(n)
                g = pool[pt[p_ // 16], :, p_ % 16, :].astype(np.float64)
                r = ref_c[li][:n].astype(np.float64)
                assert np.abs(g - r).max() <= TOL_KV * np.sqrt(np.mean(r ** 2))
        _assert_same_pass(dec, cfg, tokens, range(cfg["n_layers"]))
    finally:
        dec.close()


def test_prefill_decode_prefill_interleaved(lib, tiny):
    # a 20-token prompt, three decode steps, then 10 more prompt tokens at the
    # position the decode steps reached: the cache and logits follow the oracle
    cfg, dec, om, pt = tiny
    first = synth.prompt_tokens(14, 20, cfg["vocab"])
    more = synth.prompt_tokens(15, 10, cfg["vocab"])
    kc, vc = _empty_cache(cfg)
    _run(dec, first, 0)
    ref, tok_ref = omodel.prefill_ref(om, kc, vc, first, 0)
    t = tok_ref
    for s in range(3):
        dec.token.fill_(t)
        dec.step()
        torch.cuda.synchronize()
        r, t = omodel.decode_step_ref(om, kc, vc, t, 20 + s)
    assert int(dec.pos.item()) == 23
    got, tok, pos = _run(dec, more, 23)
    assert lib.device_error() == 0 and pos == 33
    ref, tok_ref = omodel.prefill_ref(om, kc, vc, more, 23)
    _check_logits(got, ref, tok, tok_ref)
    _check_cache(cfg, dec, pt, kc, vc, 0, 33)


@pytest.mark.slow
def test_full_size_prefill_against_oracle(lib):
    """7B shape, a 512-token prompt on an empty cache (the time-to-first-token
    workload) against the oracle's prompt pass in block form: the last row's
    logits within 2e-2 * rms; every K/V row of layer 0 (one projection of the
    embedding) within the per-op 1e-2 * rms, and of layers 13 and 27 (the
    composition of the layers below) within the model's 2e-2 * rms."""
    if not fullsize.enough_host_memory(24):
        pytest.skip("the full-size oracle needs ~24 GiB of free host memory")
    n, ctx, pages = 512, 1024, 80
    cfg, dec, om, pt = fullsize.build_pair(2025, ctx, pages)
    try:
        tokens = synth.prompt_tokens(2025, n, cfg["vocab"])
        got, tok, pos = _run(dec, tokens, 0)
        assert lib.device_error() == 0 and pos == n
        pools = {li: (dec.w["layers"][li]["k_pool"].cpu().numpy(), dec.w["layers"][li]["v_pool"].cpu().numpy())
                 for li in (0, 13, cfg["n_layers"] - 1)}
        _assert_same_pass(dec, cfg, tokens, (0, 13, cfg["n_layers"] - 1))
    finally:
        dec.close()
    kc, vc = fullsize.empty_cache(cfg, ctx)
    ref, toks = omodel.prefill_block_ref(om, kc, vc, tokens, 0)
    mx, rm = fullsize.rel_err(got, ref[0])
    print("full-size prompt pass vs oracle: logits max %.3e rms %.3e (x rms)" % (mx, rm))
    p_ = np.arange(n)
    errs = {}
    for li, (kp, vp) in pools.items():
        for which, pool, ref_c in (("k", kp, kc), ("v", vp, vc)):
            errs[(li, which)] = fullsize.rel_err(pool[pt[p_ // 16], :, p_ % 16, :], ref_c[li][:n])
            print("layer %d %s rows: max %.3e rms %.3e (x rms)" % ((li, which) + errs[(li, which)]))
    _check_logits(got, ref[0], tok, toks[0])
    for key, (e, _) in errs.items():
        tol = TOL_KV if key[0] == 0 else TOL_LOGITS
        assert e <= tol, "%s rows: max err %.3e > %.0e * rms" % (key, e, tol)
