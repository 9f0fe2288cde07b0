"""CPU checks of the prompt GEMM's work division (w4_gemm_plan, host only).

The kernel gives each CTA a run of (tile, scale group) units and writes a
piece's partial sums to a slot of [splits][n][N]; the next kernel adds all
`splits` slots of every tile.  So the plan must (1) cover every unit exactly
once, (2) give each CTA at least one unit, (3) keep every slot below
`splits` (the workspace holds no more), (4) fill every slot of every tile
exactly once, by a piece or by the zero-fill of the CTA holding the tile's
first piece (stream-K), and (5) give whole tiles to every CTA when there is
one slot (split K of one, and the persistent walk), since those CTAs write
final results.  The unit rules below restate the kernel's, for the planner's
output to be checked against.
"""

import random

import numpy as np
import pytest

from int4_weight_only_w4a16_gb300 import binding


@pytest.fixture(scope="module")
def lib():
    from int4_weight_only_w4a16_gb300 import build
    build.build()
    return binding


def _cta_of(u, units, ctas):
    return ((u + 1) * ctas + units - 1) // units - 1


def _ranges(p, gt):
    tiles = p["tok_tiles"] * p["row_tiles"]
    units, ctas = tiles * gt, p["ctas"]
    c = np.arange(ctas, dtype=np.int64)
    if p["mode"] == 2:
        return (c * tiles // ctas) * gt, ((c + 1) * tiles // ctas) * gt
    if p["mode"] == 1:
        return c * units // ctas, (c + 1) * units // ctas
    gps = p["kb_per_split"] // 2
    split, tile = c // tiles, c % tiles
    u0 = tile * gt + split * gps
    return u0, np.minimum(tile * gt + gt, u0 + gps)


def _check(epi, n, N, K, sms):
    p = binding.gemm_plan(epi, n, N, K, sms)
    gt = K // 128
    tiles = p["tok_tiles"] * p["row_tiles"]
    units = tiles * gt
    assert p["bn"] in (64, 128, 256) and p["tok_tiles"] * p["bn"] >= n > (p["tok_tiles"] - 1) * p["bn"]
    assert p["row_tiles"] * (64 if epi == 2 else 128) == N
    assert 1 <= p["stages"] <= 4 and p["splits"] >= 1
    u0, u1 = _ranges(p, gt)
    assert np.all(u1 > u0), "a CTA without work"
    order = np.argsort(u0, kind="stable")
    assert u0[order][0] == 0 and u1[order][-1] == units and np.all(u0[order][1:] == u1[order][:-1])
    if p["mode"] in (1, 2):
        assert p["ctas"] <= sms
    filled = np.zeros((tiles, p["splits"]), np.int32)
    for c in range(p["ctas"]):
        u = int(u0[c])
        while u < u1[c]:
            t = u // gt
            end = min(int(u1[c]), t * gt + gt)
            if p["splits"] == 1:
                assert u == t * gt and end == t * gt + gt, "a piece short of a whole tile with one slot"
                filled[t, 0] += 1
            else:
                if p["mode"] == 1:
                    first = _cta_of(t * gt, units, p["ctas"])
                    slot = c - first
                    if slot == 0:   # the zero-fill of the slots this tile leaves unused
                        pieces = _cta_of(t * gt + gt - 1, units, p["ctas"]) - first + 1
                        filled[t, pieces:] += 1
                else:
                    slot = c // tiles
                assert 0 <= slot < p["splits"]
                filled[t, slot] += 1
            u = end
    assert np.all(filled == 1), "slots filled %s times" % sorted(set(filled.ravel().tolist()))
    return p


def test_plans_of_the_7b_prompt_pass(lib):
    # 512 tokens: QKV and O split K in two, gate/up persistent, down stream-K
    assert _check(0, 512, 4608, 3584, 152)["mode"] == 0
    assert _check(1, 512, 3584, 3584, 152)["splits"] == 2
    gu = _check(2, 512, 18944, 3584, 152)
    assert gu["mode"] == 2 and gu["ctas"] == 152 and gu["splits"] == 1
    down = _check(1, 512, 3584, 18944, 152)
    assert down["mode"] == 1 and down["ctas"] == 152 and down["splits"] == 4


@pytest.mark.parametrize("sms", [152, 148, 132])
def test_plans_cover_every_unit_and_slot(lib, sms):
    rng = random.Random(sms)
    shapes = [(e, n, N, K) for e in (0, 1, 2) for n in (1, 64, 65, 300, 512) for N in (128, 3584, 18944)
              for K in (128, 1152, 3584, 18944)]
    shapes += [(rng.randrange(3), rng.choice([1, 17, 64, 100, 129, 256, 257, 700, 1024, 2048]),
                128 * rng.randrange(1, 160), 128 * rng.randrange(1, 160)) for _ in range(150)]
    modes = set()
    for e, n, N, K in shapes:
        modes.add(_check(e, n, N, K, sms)["mode"])
    assert modes == {0, 1, 2}


def test_plan_rejects_bad_shapes(lib):
    with pytest.raises(binding.W4Error):
        binding.gemm_plan(0, 4, 200, 128, 152)
    with pytest.raises(binding.W4Error):
        binding.gemm_plan(3, 4, 128, 128, 152)
    with pytest.raises(binding.W4Error):
        binding.gemm_plan(0, 4, 128, 128, 0)
