"""CPU checks of the paged decode attention's work division
(w4_attention_plan with the SM count and cluster limit given: host only).

A (sequence, KV head) takes `splits` CTAs of four warps, each warp `ppw`
pages of the capacity in order.  So the splits must cover every page of the
capacity, and none may start past it.  Clustered splits merge in
distributed shared memory, so a cluster must fit what the GPU co-schedules (8
CTAs, or 16 where non-portable clusters fit), and the clusters of up to 16
CTAs that need several of them resident at once must all fit on the GPU.
Unclustered splits merge through the workspace: at most 256 of them, with at
least two pages per warp.  Four-page rings only where a warp has more than two
pages.
"""

import random

import pytest

from int4_weight_only_w4a16_gb300 import binding

WARPS, PAGE = 4, 16


@pytest.fixture(scope="module")
def lib():
    from int4_weight_only_w4a16_gb300 import build
    build.build()
    return binding


def _check(b, hq, hkv, ctx, sms, cmax):
    p = binding.attention_plan(b, hq, hkv, ctx, sms, cmax)
    pages = (ctx + PAGE - 1) // PAGE
    per_cta = WARPS * p["ppw"]
    assert p["grid"] == (p["splits"], hkv, b)
    assert p["ppw"] >= 1 and p["splits"] >= 1
    assert p["splits"] * per_cta >= pages > (p["splits"] - 1) * per_cta
    assert p["stages"] in (2, 4) and (p["stages"] == 2 or (p["cluster"] and p["ppw"] > 2))
    if p["cluster"]:
        assert p["splits"] <= cmax and pages > 2 * WARPS
        if p["splits"] > 8 and pages > 16 * WARPS:   # long contexts: every cluster resident at once
            assert b * hkv * p["splits"] <= sms
    else:
        assert p["splits"] <= 256 and p["ppw"] >= 2
    assert p["ws_bytes"] >= b * hq * p["splits"] * (128 + 2) * 4
    return p


def test_plans_of_the_decode_step(lib):
    # the 7B decode step plans for its cache's capacity: 784 tokens, 49 pages -> 13 CTAs, one page a warp
    p = _check(1, 28, 4, 784, 152, 16)
    assert p["cluster"] == 1 and p["splits"] == 13 and p["ppw"] == 1
    assert _check(1, 28, 4, 784, 152, 8)["splits"] == 7   # without 16-CTA clusters: two pages a warp
    # the long contexts of the standalone calls
    assert _check(1, 28, 4, 8192, 152, 16)["cluster"] == 1
    assert _check(8, 28, 4, 32768, 152, 16)["cluster"] == 0


@pytest.mark.parametrize("sms,cmax", [(152, 16), (152, 8), (148, 16), (132, 8)])
def test_plans_cover_the_capacity(lib, sms, cmax):
    rng = random.Random(sms * 100 + cmax)
    cases = [(b, 28, hkv, ctx) for b in (1, 2, 8) for hkv in (1, 4, 8)
             for ctx in (1, 15, 16, 17, 128, 129, 512, 513, 1000, 1024, 1025, 4096, 8192, 8193, 32768)]
    cases += [(rng.choice((1, 2, 3, 8, 33)), 28, rng.choice((1, 2, 4, 7, 14, 28)), rng.randrange(1, 70000))
              for _ in range(300)]
    kinds = set()
    for b, hq, hkv, ctx in cases:
        if hq % hkv:
            continue
        p = _check(b, hq, hkv, ctx, sms, cmax)
        kinds.add((p["cluster"], p["stages"]))
    assert {(0, 2), (1, 2), (1, 4)} <= kinds


def test_plan_rejects_bad_arguments(lib):
    for args in ((0, 28, 4, 100, 152, 16), (1, 28, 3, 100, 152, 16), (1, 28, 4, 0, 152, 16),
                 (1, 28, 4, 100, -1, 16), (1, 28, 4, 100, 152, 12)):
        with pytest.raises(binding.W4Error):
            binding.attention_plan(*args)
