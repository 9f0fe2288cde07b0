"""CPU checks of the batch-1 streaming GEMV's plan (w4_gemv_plan, host only;
without a GPU it plans for 148 SMs).

Each CTA streams its row groups through a ring of ns stages of gs groups;
unit u (of NU = 2 cw / hpr) owns groups u, u + NU, ... of its CTA, so its
successive groups lie st = NU / gs stages apart.  A unit waits on a stage's
`full` barrier by phase parity, so a slot must never be two fills ahead of a
waiter: either ns is a multiple of st (the slot a unit waits on last held that
unit's own previous group), or no slot is reused at all (every unit owns at
most one group of its CTA and the ring holds them all).  The ring and the
staged input must fit the shared memory the plan may use.  Rows too long for
that (k above 21632 for one matrix, 11264 for a gate/up pair) get no plan, and
the GEMV hands them to the tensor-core kernel.
"""

import random

import pytest

from int4_weight_only_w4a16_gb300 import binding

SMEM_MAX = 220 * 1024
RING_MAX = 176 * 1024


@pytest.fixture(scope="module")
def lib():
    from int4_weight_only_w4a16_gb300 import build
    build.build()
    return binding


def _check(nm, n, k):
    p = binding.gemv_plan(nm, n, k)
    if p["grid"] == 0:
        return p
    assert p["grid"] == min(n, 148)
    assert p["cw"] in (8, 12) and p["hpr"] in (1, 2) and p["rg"] in (1, 2)
    nu = 2 * p["cw"] // p["hpr"]
    assert nu % p["gs"] == 0
    st = nu // p["gs"]
    groups = (n + p["rg"] - 1) // p["rg"]
    per_cta = (groups + p["grid"] - 1) // p["grid"]
    assert 1 <= p["ns"] <= 8
    assert p["ns"] % st == 0 or (per_cta <= nu and p["ns"] * p["gs"] >= per_cta), p
    assert p["wbytes"] == p["gs"] * p["rg"] * k // 2
    assert p["sbytes"] >= p["gs"] * p["rg"] * (k // 128) * 2 + 16
    assert p["ns"] * nm * p["wbytes"] <= RING_MAX and p["smem"] <= SMEM_MAX
    return p


def test_plan_invariants(lib):
    rng = random.Random(7)
    shapes = [(nm, n, k) for nm in (1, 2) for n in (1, 2, 7, 100, 148, 149, 512, 3584, 4608, 18944, 152064)
              for k in (128, 640, 3584, 9344, 18944)]
    shapes += [(rng.choice((1, 2)), rng.randrange(1, 200000), 128 * rng.randrange(1, 190)) for _ in range(400)]
    planned = sum(_check(*s)["grid"] > 0 for s in shapes)
    assert planned > len(shapes) // 2


def test_long_rows_leave_the_streaming_kernel(lib):
    for n in (1, 149, 3584, 152064):
        assert _check(1, n, 21632)["grid"] > 0 and _check(1, n, 21760)["grid"] == 0
        assert _check(2, n, 11264)["grid"] > 0 and _check(2, n, 11392)["grid"] == 0


def test_plan_rejects_bad_arguments(lib):
    for args in ((3, 16, 128), (1, 0, 128), (1, 16, 100), (1, 16, 0)):
        with pytest.raises(binding.W4Error):
            binding.gemv_plan(*args)
