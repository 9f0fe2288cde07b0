"""Pins for oracle.model (CPU only): per-op closed forms and invariants.

The composed decode step has no published values to compare with (the pages
print no logits and the trained weights are not available).  Beyond the ops
pinned here it is pinned by two symmetries (relabelled hidden groups, and
relabelled KV heads with their query groups), which a misrouted, transposed
or misgrouped projection breaks; by an identity: layers whose output and down
projections are zero leave the embedding -> final norm -> LM head path (a
dropped residual or a lost norm breaks it); by a closed gate: a gate column of
-1000 silences the MLP exactly (gate and up swapped breaks it); and by a
cancellation: attention built to add exactly -x0 zeroes every logit (a
residual with the wrong sign, or dropped, breaks it).  Each of these mistakes,
planted in a scratch copy of the oracle, fails at least one pin.
"""

import math

import numpy as np

import synth
from oracle import model


def test_rmsnorm_unit_rms_and_gamma():
    r = np.random.default_rng(1)
    x = r.standard_normal(512) * 7.0
    y = model.rmsnorm(x, np.ones(512), 0.0)
    assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 1e-14
    g = r.standard_normal(512)
    assert np.allclose(model.rmsnorm(x, g, 0.0), y * g, rtol=1e-15, atol=0)
    # eps enters under the root: a zero vector stays finite and zero
    assert np.all(model.rmsnorm(np.zeros(8), np.ones(8), 1e-6) == 0)


def test_rope_position_zero_is_identity():
    r = np.random.default_rng(2)
    v = r.standard_normal((3, 128))
    assert np.array_equal(model.rope(v, 0, 1e6), v)


def test_rope_rotate_half_pairs_and_frequencies():
    # unit vector at dim i turns into (cos, sin) at dims (i, i + 64) with angle
    # pos * theta^(-2i/128); dims i+1 and the rest stay zero
    pos, theta = 37, 1e6
    for i in (0, 1, 17, 63):
        e = np.zeros((1, 128))
        e[0, i] = 1.0
        out = model.rope(e, pos, theta)[0]
        ang = pos * theta ** (-2.0 * i / 128)
        want = np.zeros(128)
        want[i] = math.cos(ang)
        want[i + 64] = math.sin(ang)
        assert np.allclose(out, want, rtol=0, atol=1e-15)
        # and the partner dimension rotates the other way
        e2 = np.zeros((1, 128))
        e2[0, i + 64] = 1.0
        out2 = model.rope(e2, pos, theta)[0]
        want2 = np.zeros(128)
        want2[i] = -math.sin(ang)
        want2[i + 64] = math.cos(ang)
        assert np.allclose(out2, want2, rtol=0, atol=1e-15)


def test_rope_norm_preserving_and_relative():
    r = np.random.default_rng(3)
    q = r.standard_normal((1, 128))
    k = r.standard_normal((1, 128))
    for p in (1, 100, 4095):
        assert abs(np.linalg.norm(model.rope(q, p, 1e6)) - np.linalg.norm(q)) < 1e-12
    d1 = float(model.rope(q, 50, 1e6)[0] @ model.rope(k, 20, 1e6)[0])
    d2 = float(model.rope(q, 530, 1e6)[0] @ model.rope(k, 500, 1e6)[0])
    assert abs(d1 - d2) < 1e-11


def test_silu_values():
    assert model.silu(0.0) == 0.0
    assert abs(model.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(model.silu(40.0) - 40.0) < 1e-12
    assert abs(model.silu(-40.0)) < 1e-15


def test_f16_rounding_is_nearest_even():
    # 1 + 2^-11 is halfway between 1 and 1 + 2^-10: ties go to the even 1.0
    assert model.f16(1.0 + 2.0 ** -11) == 1.0
    assert model.f16(1.0 + 3 * 2.0 ** -11) == 1.0 + 2 * 2.0 ** -10


def test_argmax_ties_take_lowest_index():
    logits = np.array([0.5, 2.0, -1.0, 2.0])
    assert int(np.argmax(logits)) == 1


def _tiny(seed=5):
    cfg = dict(synth.TINY)
    w = synth.model_small_tensors(seed, cfg)
    for li in range(cfg["n_layers"]):
        for name in synth.MATRICES:
            w["layers"][li][name] = synth.model_matrix(seed, cfg, li, name)
    w["lm_head"] = synth.model_matrix(seed, cfg, -1, "lm_head")
    return cfg, model.DecodeModel(cfg, w)


def test_decode_step_first_token_attends_to_itself():
    # at position 0 the context is the token itself: the attention output of
    # every query head equals the (fp16) v row of its KV head
    cfg, m = _tiny()
    hkv, d = cfg["n_kv_heads"], cfg["head_dim"]
    kc = [np.zeros((4, hkv, d), np.float16) for _ in range(cfg["n_layers"])]
    vc = [np.zeros((4, hkv, d), np.float16) for _ in range(cfg["n_layers"])]
    logits, tok = model.decode_step_ref(m, kc, vc, 3, 0)
    assert logits.shape == (cfg["vocab"],) and 0 <= tok < cfg["vocab"]
    assert tok == int(np.argmax(logits))
    # the cache row written at position 0 is finite and v is the un-roped projection
    layer0 = m.layers[0]
    x = m.embed[3].astype(np.float64)
    h = model.f16(model.rmsnorm(x, layer0["ln1"], cfg["rms_eps"]))
    v = model.f16(layer0["wv"](h) + layer0["bv"].astype(np.float64))
    assert np.array_equal(vc[0][0].astype(np.float64).reshape(-1), v)


def test_decode_step_is_deterministic_and_uses_the_cache():
    cfg, m = _tiny()
    hkv, d = cfg["n_kv_heads"], cfg["head_dim"]

    def run(prefill_seed):
        kc, vc = [], []
        for li in range(cfg["n_layers"]):
            k, v = synth.prefill_kv(prefill_seed, cfg, li, 8)
            kk = np.zeros((9, hkv, d), np.float16)
            vv = np.zeros_like(kk)
            kk[:8], vv[:8] = k, v
            kc.append(kk)
            vc.append(vv)
        return model.decode_step_ref(m, kc, vc, 11, 8)[0]

    a, b, c = run(1), run(1), run(2)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c)


def test_prefill_matches_causal_masked_block_form():
    # the loop definition (decode step per token) against the block form (all
    # rows through each projection at once, explicit causal mask over the
    # cached and prompt keys), after 5 cached rows: same logits up to float64
    # summation order.  A wrong position offset or a causality leak moves the
    # logits by a large fraction of their rms.
    cfg, m = _tiny()
    hkv, d = cfg["n_kv_heads"], cfg["head_dim"]
    start, tokens = 5, [7, 1, 300, 42, 42, 9, 100, 3, 250, 17, 0, 64, 511, 8, 8, 2, 77, 19, 33]
    kc, vc = [], []
    for li in range(cfg["n_layers"]):
        k, v = synth.prefill_kv(4, cfg, li, start)
        kk = np.zeros((start + len(tokens), hkv, d), np.float16)
        vv = np.zeros_like(kk)
        kk[:start], vv[:start] = k, v
        kc.append(kk)
        vc.append(vv)
    kc0, vc0 = [c.copy() for c in kc], [c.copy() for c in vc]
    logits, tok = model.prefill_ref(m, kc, vc, tokens, start)
    want, toks = model.prefill_block_ref(m, kc0, vc0, tokens, start)
    rms = np.sqrt(np.mean(want[0] ** 2))
    # fp16 rounding points can flip on a summation-order difference: allow a few
    assert np.max(np.abs(logits - want[0])) <= 1e-6 * rms
    assert tok == toks[0] == int(np.argmax(logits))
    # every cache row written by the loop is the block form's, rows before start untouched
    for li in range(cfg["n_layers"]):
        assert np.mean(kc[li] == kc0[li]) > 0.99 and np.mean(vc[li] == vc0[li]) > 0.99
        assert np.array_equal(kc0[li][:start], synth.prefill_kv(4, cfg, li, start)[0])


def test_block_form_logits_of_several_rows_are_teacher_forced_decode_steps():
    # row i of the block form is decode step i with the input tokens fixed in
    # advance: logits of chosen rows equal the loop's steps at those positions
    cfg, m = _tiny(6)
    hkv, d = cfg["n_kv_heads"], cfg["head_dim"]
    start, tokens = 17, list(synth.prompt_tokens(3, 23, cfg["vocab"]))
    kc, vc = [], []
    for li in range(cfg["n_layers"]):
        k, v = synth.prefill_kv(8, cfg, li, start)
        kk = np.zeros((start + len(tokens), hkv, d), np.float16)
        vv = np.zeros_like(kk)
        kk[:start], vv[:start] = k, v
        kc.append(kk)
        vc.append(vv)
    kc0, vc0 = [c.copy() for c in kc], [c.copy() for c in vc]
    rows = [0, 1, 2, 15, 22]
    want, toks = model.prefill_block_ref(m, kc0, vc0, tokens, start, logits_rows=rows)
    assert want.shape == (len(rows), cfg["vocab"])
    for i, t in enumerate(tokens):
        got, tok = model.decode_step_ref(m, kc, vc, t, start + i)
        if i in rows:
            r = rows.index(i)
            assert np.max(np.abs(got - want[r])) <= 1e-6 * np.sqrt(np.mean(want[r] ** 2))
            assert tok == toks[r]


def test_rope_rows_and_rmsnorm_rows_are_the_per_row_functions():
    r = np.random.default_rng(9)
    v = r.standard_normal((5, 3, 128))
    pos = np.array([0, 1, 16, 511, 4095])
    got = model.rope_rows(v, pos, 1e6)
    for i in range(5):
        assert np.allclose(got[i], model.rope(v[i], pos[i], 1e6), rtol=0, atol=1e-14)
    x = r.standard_normal((4, 256)) * 3
    g = 1 + 0.1 * r.standard_normal(256)
    got = model.rmsnorm_rows(x, g, 1e-6)
    for i in range(4):
        assert np.allclose(got[i], model.rmsnorm(x[i], g, 1e-6), rtol=1e-15, atol=0)


def test_quant_linear_matmul_is_matvec_per_row_and_from_codes():
    w = synth.gemv_w(3, 300, 256)
    ql = model.QuantLinear(w)
    xs = synth.gemv_x(3, 3, 256)
    y = ql.matmul(xs, row_block=128)
    for i in range(3):
        assert np.allclose(y[i], ql(xs[i]), rtol=1e-13, atol=1e-13)
    q2 = model.QuantLinear.from_codes(ql.codes, ql.scales)
    assert np.array_equal(q2.matmul(xs), ql.matmul(xs))


def test_prefill_of_one_token_is_one_decode_step_and_splits_compose():
    cfg, m = _tiny()
    hkv, d = cfg["n_kv_heads"], cfg["head_dim"]
    L = cfg["n_layers"]
    z = lambda: [np.zeros((12, hkv, d), np.float16) for _ in range(L)]  # noqa: E731
    k1, v1, k2, v2 = z(), z(), z(), z()
    a = model.prefill_ref(m, k1, v1, [5], 0)
    b = model.decode_step_ref(m, k2, v2, 5, 0)
    assert np.array_equal(a[0], b[0]) and a[1] == b[1]
    # a prompt split in two passes leaves the same cache and logits as one pass
    toks = [3, 1, 4, 1, 5, 9, 2, 6, 5, 3]
    k3, v3, k4, v4 = z(), z(), z(), z()
    one = model.prefill_ref(m, k3, v3, toks, 0)
    model.prefill_ref(m, k4, v4, toks[:6], 0)
    two = model.prefill_ref(m, k4, v4, toks[6:], 6)
    assert np.array_equal(one[0], two[0])
    assert all(np.array_equal(k3[i], k4[i]) and np.array_equal(v3[i], v4[i]) for i in range(L))
    try:
        model.prefill_ref(m, k3, v3, [], 0)
        raise AssertionError("empty prompt accepted")
    except ValueError:
        pass


# ---------------------------------------------------------------- symmetries of the composed step
# The decode step is a fixed composition: relabelling hidden units, or KV heads
# together with their query-head groups, consistently in every weight must leave
# the logits unchanged.  Both relabellings move whole 128-column scale groups
# (head_dim = 128), so the quantised model is the same function, and only float64
# summation order differs.  A wrong head-to-group mapping, a transposed or
# misrouted projection, or a norm weight on the wrong axis breaks the equality.

def _ql(codes, scales):
    return model.QuantLinear.from_codes(np.ascontiguousarray(codes), np.ascontiguousarray(scales))


def _relabelled(m, cfg, hidden_groups=None, kv_heads=None, skip=()):
    """A copy of oracle model m with hidden groups and/or KV heads relabelled.
    hidden_groups[g]: the old group that becomes group g; kv_heads[j] likewise.
    Names in `skip` keep their old layout (to plant an inconsistency)."""
    H, d = cfg["hidden"], cfg["head_dim"]
    hq, hkv = cfg["n_q_heads"], cfg["n_kv_heads"]
    grp = hq // hkv
    gh = np.arange(H // 128) if hidden_groups is None else np.asarray(hidden_groups)
    cols = (gh[:, None] * 128 + np.arange(128)).ravel()
    kvp = np.arange(hkv) if kv_heads is None else np.asarray(kv_heads)
    qheads = (kvp[:, None] * grp + np.arange(grp)).ravel()          # new q head -> old q head
    qrows = (qheads[:, None] * d + np.arange(d)).ravel()
    kvrows = (kvp[:, None] * d + np.arange(d)).ravel()

    def reads_hidden(ql, name):
        return ql if name in skip else _ql(ql.codes[:, cols], ql.scales[:, gh])

    def rows(ql, r, name):
        return ql if name in skip else _ql(ql.codes[r], ql.scales[r])

    w = {"embed": m.embed[:, cols], "final_norm": m.final_norm[cols], "lm_head": reads_hidden(m.lm_head, "lm_head"),
         "layers": []}
    for L in m.layers:
        wq, wk, wv = (reads_hidden(L[n], n) for n in ("wq", "wk", "wv"))
        wo = L["wo"]
        wo = wo if "wo" in skip else _ql(wo.codes[cols][:, qrows], wo.scales[cols][:, qheads])
        wd = L["wd"]
        wd = wd if "wd" in skip else _ql(wd.codes[cols], wd.scales[cols])
        w["layers"].append({
            "ln1": L["ln1"][cols], "ln2": L["ln2"][cols],
            "wq": rows(wq, qrows, "wq_rows"), "bq": L["bq"][qrows],
            "wk": rows(wk, kvrows, "wk_rows"), "bk": L["bk"][kvrows],
            "wv": rows(wv, kvrows, "wv_rows"), "bv": L["bv"][kvrows],
            "wo": wo, "wg": reads_hidden(L["wg"], "wg"), "wu": reads_hidden(L["wu"], "wu"), "wd": wd})
    return model.DecodeModel(cfg, w)


def _decode_logits(m, cfg, tokens):
    hkv, d = cfg["n_kv_heads"], cfg["head_dim"]
    kc = [np.zeros((len(tokens), hkv, d), np.float16) for _ in range(cfg["n_layers"])]
    vc = [np.zeros((len(tokens), hkv, d), np.float16) for _ in range(cfg["n_layers"])]
    return np.stack([model.decode_step_ref(m, kc, vc, t, p)[0] for p, t in enumerate(tokens)])


def _rel(a, b):
    return np.abs(a - b).max() / np.sqrt(np.mean(b ** 2))


def test_decode_step_is_invariant_under_relabelled_hidden_groups():
    cfg, m = _tiny()
    tokens = [3, 141, 59, 265]
    ref = _decode_logits(m, cfg, tokens)
    perm = [2, 0, 3, 1]                                   # the hidden size 512 is four scale groups
    assert _rel(_decode_logits(_relabelled(m, cfg, hidden_groups=perm), cfg, tokens), ref) < 1e-9
    # planted: the down projection keeps its old output order
    assert _rel(_decode_logits(_relabelled(m, cfg, hidden_groups=perm, skip=("wd",)), cfg, tokens), ref) > 0.1


def test_decode_step_is_invariant_under_relabelled_kv_heads():
    cfg, m = _tiny()
    tokens = [7, 77, 700, 70]
    ref = _decode_logits(m, cfg, tokens)
    perm = [1, 0]                                          # two KV heads, two query heads each
    assert _rel(_decode_logits(_relabelled(m, cfg, kv_heads=perm), cfg, tokens), ref) < 1e-9
    # planted: the K rows keep their old head order (queries meet the other group's keys)
    assert _rel(_decode_logits(_relabelled(m, cfg, kv_heads=perm, skip=("wk_rows",)), cfg, tokens), ref) > 0.1
    # planted: the output projection keeps its old input order
    assert _rel(_decode_logits(_relabelled(m, cfg, kv_heads=perm, skip=("wo",)), cfg, tokens), ref) > 0.1


def test_layers_adding_nothing_leave_the_embedding_path():
    # with every layer's output and down projections zero, each layer adds nothing to
    # the residual stream: the step equals the step of the same model without layers
    # (embedding -> final RMSNorm -> LM head).  A step that replaced the residual
    # instead of adding to it, or lost the final norm, fails this.
    cfg, m = _tiny()
    hkv, d = cfg["n_kv_heads"], cfg["head_dim"]
    zero = lambda ql: model.QuantLinear.from_codes(np.zeros_like(ql.codes), ql.scales)
    w = {"embed": m.embed, "final_norm": m.final_norm, "lm_head": m.lm_head, "layers": []}
    for L in m.layers:
        lw = dict(L)
        lw["wo"], lw["wd"] = zero(L["wo"]), zero(L["wd"])
        w["layers"].append(lw)
    quiet = model.DecodeModel(cfg, w)
    bare = model.DecodeModel(cfg, {"embed": m.embed, "final_norm": m.final_norm, "lm_head": m.lm_head, "layers": []})
    for p, t in enumerate([5, 500, 50]):
        kc = [np.zeros((3, hkv, d), np.float16) for _ in range(cfg["n_layers"])]
        vc = [np.zeros((3, hkv, d), np.float16) for _ in range(cfg["n_layers"])]
        a = model.decode_step_ref(quiet, kc, vc, t, p)[0]
        b = model.decode_step_ref(bare, [], [], t, p)[0]
        assert np.array_equal(a, b)
    # and the layers do matter when they add something
    kc = [np.zeros((1, hkv, d), np.float16) for _ in range(cfg["n_layers"])]
    vc = [np.zeros((1, hkv, d), np.float16) for _ in range(cfg["n_layers"])]
    full = model.decode_step_ref(m, kc, vc, 5, 0)[0]
    assert _rel(full, model.decode_step_ref(bare, [], [], 5, 0)[0]) > 0.1


def test_a_closed_gate_silences_the_mlp():
    # One layer at position 0 whose attention adds nothing (zero output projection).
    # The second norm keeps one coordinate j, where the token's embedding is large
    # and positive, so the MLP input is c * e_j with c of order one; the gate's
    # column j is -1000 in every row (its other columns zero).
    # Every gate pre-activation is then about -1000 c: SiLU gives exactly 0 and the
    # MLP adds nothing, so the step equals the step with a zero down projection.
    # Gate and up swapped would give SiLU(up) * (-1000 c) instead: far from zero.
    cfg, m = _tiny()
    cfg = dict(cfg, n_layers=1)
    hkv, d, H = cfg["n_kv_heads"], cfg["head_dim"], cfg["hidden"]
    tok = 5
    x0 = m.embed[tok].astype(np.float64)
    j = int(np.argmax(x0))
    assert x0[j] > 0.5 * np.sqrt(np.mean(x0 ** 2))
    L = dict(m.layers[0])
    L["wo"] = model.QuantLinear.from_codes(np.zeros_like(L["wo"].codes), L["wo"].scales)
    ln2 = np.zeros(H, np.float16)
    ln2[j] = 1.0
    L["ln2"] = ln2
    codes = np.zeros_like(L["wg"].codes)
    codes[:, j] = -8
    scales = np.zeros_like(L["wg"].scales)
    scales[:, j // 128] = 125.0                                # -8 * 125 = -1000
    L["wg"] = model.QuantLinear.from_codes(codes, scales)
    silent = dict(L, wd=model.QuantLinear.from_codes(np.zeros_like(L["wd"].codes), L["wd"].scales))
    outs = []
    for layer in (L, silent):
        mm = model.DecodeModel(cfg, {"embed": m.embed, "final_norm": m.final_norm, "lm_head": m.lm_head,
                                     "layers": [layer]})
        kc, vc = [np.zeros((1, hkv, d), np.float16)], [np.zeros((1, hkv, d), np.float16)]
        with np.errstate(over="ignore"):   # exp(+2800) in SiLU's denominator: SiLU = -0
            outs.append(model.decode_step_ref(mm, kc, vc, tok, 0)[0])
    assert np.array_equal(outs[0], outs[1])


def test_attention_that_adds_minus_the_embedding_cancels_the_residual():
    # One layer at position 0.  A zero V projection with bias 1 in dimension 0 of
    # every KV head makes each query head's attention output the unit vector e_0
    # (softmax over one key is 1).  The output projection's column 0 is -1 times
    # the token's embedding (code -1, scale = the fp16 embedding value; every other
    # code zero), so attention adds exactly -x0: the residual cancels, the MLP
    # sees RMSNorm(0) = 0 and adds 0, and every logit is exactly 0.  A residual
    # with the wrong sign leaves 2 x0, a dropped one -x0: nonzero logits.
    cfg, m = _tiny()
    cfg = dict(cfg, n_layers=1)
    hkv, d = cfg["n_kv_heads"], cfg["head_dim"]
    tok = 11
    x0 = m.embed[tok].astype(np.float16)
    L = dict(m.layers[0])
    L["wv"] = model.QuantLinear.from_codes(np.zeros_like(L["wv"].codes), L["wv"].scales)
    bv = np.zeros(hkv * d, np.float16)
    bv[::d] = 1.0
    L["bv"] = bv
    codes = np.zeros_like(L["wo"].codes)
    codes[:, 0] = -1
    scales = np.zeros_like(L["wo"].scales)
    scales[:, 0] = x0
    L["wo"] = model.QuantLinear.from_codes(codes, scales)
    mm = model.DecodeModel(cfg, {"embed": m.embed, "final_norm": m.final_norm, "lm_head": m.lm_head, "layers": [L]})
    kc, vc = [np.zeros((1, hkv, d), np.float16)], [np.zeros((1, hkv, d), np.float16)]
    logits = model.decode_step_ref(mm, kc, vc, tok, 0)[0]
    assert np.all(logits == 0.0)
