"""Pins for oracle.paged (CPU only): closed forms, brute force, invariants."""

import math
import os

import numpy as np
import pytest

from oracle import paged

T = paged.PAGE_TOKENS


def _scatter_dict(k_rows, v_rows, pt_row):
    """Reference placement through a dict (page, slot) -> row, independent of
    kv_append_ref's arithmetic."""
    place = {}
    for t in range(k_rows.shape[0]):
        place[(int(pt_row[t // T]), t % T)] = t
    return place


def _make(rng, L, hkv=2, d=128, pages=None):
    pages = pages or (math.ceil(L / T) + 3)
    k_pool = rng.standard_normal((pages, hkv, T, d)).astype(np.float16)
    v_pool = rng.standard_normal((pages, hkv, T, d)).astype(np.float16)
    pt = rng.permutation(pages).astype(np.int32)[None, :]
    return k_pool, v_pool, pt


def test_append_matches_dict_scatter():
    r = np.random.default_rng(1)
    hkv, d, L = 2, 128, 37
    k_pool = np.zeros((8, hkv, T, d), dtype=np.float16)
    v_pool = np.zeros_like(k_pool)
    pt = r.permutation(8).astype(np.int32)[None, :]
    k_rows = r.standard_normal((L, hkv, d)).astype(np.float16)
    v_rows = r.standard_normal((L, hkv, d)).astype(np.float16)
    for t in range(L):
        paged.kv_append_ref(k_pool, v_pool, pt, k_rows[t:t + 1], v_rows[t:t + 1], [t])
    place = _scatter_dict(k_rows, v_rows, pt[0])
    for p in range(8):
        for s in range(T):
            if (p, s) in place:
                t = place[(p, s)]
                assert np.array_equal(k_pool[p, :, s], k_rows[t])
                assert np.array_equal(v_pool[p, :, s], v_rows[t])
            else:
                assert not k_pool[p, :, s].any() and not v_pool[p, :, s].any()


def _kv_golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "kv_placement.txt")
    tables, places = {}, []
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("table"):
            head, vals = line.split("=")
            tables[int(head.split()[1])] = [int(v) for v in vals.split()]
        else:
            places.append(tuple(int(v) for v in line.split()))
    return tables, places


def test_append_places_tokens_at_hand_worked_pages_and_slots():
    # literal (sequence, token, page, slot) placements worked by hand from the page
    # layout: a wrong page index (t % 16, t // 15), slot (t // 16, (t + 1) % 16), head
    # axis or per-sequence table fails here, whatever arithmetic the oracle uses
    tables, places = _kv_golden()
    hkv, d, pages = 2, 128, 8
    k_pool = np.zeros((pages, hkv, T, d), dtype=np.float16)
    v_pool = np.zeros_like(k_pool)
    width = max(len(tb) for tb in tables.values())
    pt = np.full((2, width), -1, dtype=np.int32)
    for b, tb in tables.items():
        pt[b, :len(tb)] = tb

    def marker(b, t, h, kv):   # distinct, exactly representable in fp16
        return (1 + b) * 1000 + t * 4 + h * 2 + kv

    tokens = {0: [t for b, t, _, _ in places if b == 0], 1: [t for b, t, _, _ in places if b == 1]}
    for i in range(max(len(v) for v in tokens.values())):
        # one batched append per step: sequence b writes its i-th listed token (the
        # other sequence repeats its last one when it has fewer)
        pos = [tokens[b][min(i, len(tokens[b]) - 1)] for b in (0, 1)]
        k = np.stack([np.stack([np.full(d, marker(b, pos[b], h, 0)) for h in range(hkv)]) for b in (0, 1)])
        v = np.stack([np.stack([np.full(d, marker(b, pos[b], h, 1)) for h in range(hkv)]) for b in (0, 1)])
        paged.kv_append_ref(k_pool, v_pool, pt, k.astype(np.float16), v.astype(np.float16), pos)
    seen = set()
    for b, t, page, slot in places:
        for h in range(hkv):
            assert np.all(k_pool[page, h, slot] == marker(b, t, h, 0)), (b, t, h)
            assert np.all(v_pool[page, h, slot] == marker(b, t, h, 1)), (b, t, h)
        seen.add((page, slot))
    for page in range(pages):
        for slot in range(T):
            if (page, slot) not in seen:
                assert not k_pool[page, :, slot].any() and not v_pool[page, :, slot].any(), (page, slot)


def test_length_one_returns_first_value():
    r = np.random.default_rng(2)
    k_pool, v_pool, pt = _make(r, 1)
    q = r.standard_normal((1, 4, 128)).astype(np.float16)
    out = paged.paged_attention_ref(q, k_pool, v_pool, pt, [1], 1 / math.sqrt(128))
    for h in range(4):
        assert np.array_equal(out[0, h], v_pool[pt[0, 0], h // 2, 0].astype(np.float64))


def test_equal_keys_give_mean_of_values():
    r = np.random.default_rng(3)
    L = 23
    k_pool, v_pool, pt = _make(r, L, hkv=1)
    k_pool[:] = k_pool[0, 0, 0]
    q = r.standard_normal((1, 2, 128)).astype(np.float16)
    out = paged.paged_attention_ref(q, k_pool, v_pool, pt, [L], 0.1)
    v_c = paged.gather_contiguous(v_pool, pt[0], 0, L).astype(np.float64)
    assert np.allclose(out[0, 0], v_c.mean(axis=0), rtol=0, atol=1e-12)


def test_one_dominant_key_selects_its_value():
    r = np.random.default_rng(4)
    L = 40
    k_pool, v_pool, pt = _make(r, L, hkv=1)
    k_pool[:] = 0
    t_hot = 29
    k_pool[pt[0, t_hot // T], 0, t_hot % T, 0] = 100.0
    q = np.zeros((1, 1, 128), dtype=np.float16)
    q[0, 0, 0] = 100.0
    out = paged.paged_attention_ref(q, k_pool, v_pool, pt, [L], 1.0)
    assert np.array_equal(out[0, 0], v_pool[pt[0, t_hot // T], 0, t_hot % T].astype(np.float64))


def test_softmax_weights_sum_to_one_and_match_scalar_loop():
    r = np.random.default_rng(5)
    L = 17
    q = r.standard_normal(128)
    k_c = r.standard_normal((L, 128))
    v_c = r.standard_normal((L, 128))
    out, p = paged.attention_contiguous(q, k_c, v_c, 0.125)
    assert abs(p.sum() - 1.0) < 1e-14
    # brute force with scalar math, no max-subtraction
    s = [math.exp(0.125 * sum(q[i] * k_c[t, i] for i in range(128))) for t in range(L)]
    tot = sum(s)
    want = [sum(s[t] / tot * v_c[t, j] for t in range(L)) for j in range(128)]
    assert np.allclose(out, want, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("L", [1, 15, 16, 17, 31, 32, 33, 1000, 4096])
def test_paged_equals_contiguous(L):
    r = np.random.default_rng(100 + L)
    hkv, hq = 2, 4
    k_rows = r.standard_normal((L, hkv, 128)).astype(np.float16)
    v_rows = r.standard_normal((L, hkv, 128)).astype(np.float16)
    pages = math.ceil(L / T) + 2
    pt = r.permutation(pages).astype(np.int32)[None, :]
    k_pool = np.full((pages, hkv, T, 128), np.nan, dtype=np.float16)  # unused slots poisoned
    v_pool = np.full_like(k_pool, np.nan)
    for t in range(L):
        k_pool[pt[0, t // T], :, t % T] = k_rows[t]
        v_pool[pt[0, t // T], :, t % T] = v_rows[t]
    q = r.standard_normal((1, hq, 128)).astype(np.float16)
    scale = 1 / math.sqrt(128)
    out = paged.paged_attention_ref(q, k_pool, v_pool, pt, [L], scale)
    assert np.all(np.isfinite(out))
    for h in range(hq):
        want, _ = paged.attention_contiguous(q[0, h], k_rows[:, h // 2], v_rows[:, h // 2], scale)
        assert np.array_equal(out[0, h], want)


def test_page_permutation_invariance():
    r = np.random.default_rng(7)
    L, pages = 50, 6
    k_pool, v_pool, pt = _make(r, L, pages=pages)
    q = r.standard_normal((1, 4, 128)).astype(np.float16)
    a = paged.paged_attention_ref(q, k_pool, v_pool, pt, [L], 0.09)
    perm = r.permutation(pages)           # new id of old page p is perm[p]
    k2 = np.empty_like(k_pool)
    v2 = np.empty_like(v_pool)
    k2[perm] = k_pool
    v2[perm] = v_pool
    pt2 = perm[pt].astype(np.int32)
    b = paged.paged_attention_ref(q, k2, v2, pt2, [L], 0.09)
    assert np.array_equal(a, b)


def test_zero_length_rejected():
    r = np.random.default_rng(8)
    k_pool, v_pool, pt = _make(r, 1)
    with pytest.raises(ValueError):
        paged.paged_attention_ref(np.zeros((1, 2, 128), np.float16), k_pool, v_pool, pt, [0], 1.0)
