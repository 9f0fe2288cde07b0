"""The allocation-free attention entry point.

w4_paged_decode_attention_noalloc serves callers that cannot allocate device
memory at the point where they run attention -- a process that reserved its
whole device-memory budget up front, an allocator-less host or plugin, a
caller holding only borrowed buffers: its split-merge scratch is a fixed
array inside the library.  Its output is checked against the plain oracle
(oracle.paged) and against the workspace entry point, on two calls in a row
that share that array.  This file is collected last on purpose; it must pass
alone in a fresh process and after every other test.
"""

import math

import numpy as np
import pytest
import torch

import synth
from oracle import paged as opaged

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _inputs(seed, lens, hq=28, hkv=4, num_pages=2048):
    max_context = max(lens)
    k_pool, v_pool = synth.kv_pool(seed, num_pages, hkv)
    pt = synth.page_table(seed, lens, num_pages, max_pages=math.ceil(max_context / 16))
    q = synth.queries(seed, len(lens), hq)
    dev = "cuda"
    return (torch.from_numpy(q).to(dev), torch.from_numpy(k_pool).to(dev), torch.from_numpy(v_pool).to(dev),
            torch.from_numpy(pt).to(dev), torch.tensor(lens, dtype=torch.int32, device=dev), max_context)


def _close(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    rms = np.sqrt(np.mean(b ** 2))
    assert np.all(np.isfinite(a))
    assert np.abs(a - b).max() <= TOL * rms


def test_noalloc_matches_oracle_and_workspace_entry_point_twice(lib):
    # two different calls in a row reuse the shared scratch array; outputs and
    # every buffer are allocated before the first call, and the device's free
    # memory does not move across the calls
    cases = []
    for seed, lens in ((31, [1000, 17, 4096]), (32, [513, 1, 2000])):
        q, kp, vp, pt, lens_t, max_context = _inputs(seed, lens)
        ref = lib.paged_decode_attention(q, kp, vp, pt, lens_t, max_context)
        cases.append((seed, lens, q, kp, vp, pt, lens_t, max_context, ref, torch.empty_like(q)))
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for seed, lens, q, kp, vp, pt, lens_t, max_context, ref, out in cases:
        lib.paged_decode_attention_noalloc(q, kp, vp, pt, lens_t, max_context, out=out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free0 - (1 << 20)
    for seed, lens, q, kp, vp, pt, lens_t, max_context, ref, out in cases:
        _close(out, ref)
        want = opaged.paged_attention_ref(q.cpu().numpy(), kp.cpu().numpy(), vp.cpu().numpy(), pt.cpu().numpy(),
                                          lens, 1.0 / math.sqrt(128))
        _close(out, torch.from_numpy(want))
    assert lib.device_error() == 0


def test_noalloc_rejects_a_batch_beyond_its_scratch(lib):
    limit = lib.load().w4_paged_decode_attention_noalloc_max_scratch()
    assert limit == 8 << 20
    # 1024 one-page sequences x 28 heads need ~15 MB of split partials, more
    # than the fixed array holds: refused on the host, nothing launched
    b = 1024
    q = torch.zeros((b, 28, 128), dtype=torch.float16, device="cuda")
    kp = torch.zeros((16, 4, 16, 128), dtype=torch.float16, device="cuda")
    pt = torch.zeros((b, 1), dtype=torch.int32, device="cuda")
    lens_t = torch.full((b,), 16, dtype=torch.int32, device="cuda")
    assert lib.load().w4_attention_workspace_size(b, 28, 4, 16) > limit
    with pytest.raises(lib.W4Error) as e:
        lib.paged_decode_attention_noalloc(q, kp, kp, pt, lens_t, 16)
    assert e.value.status == 5  # W4_ERR_CAPACITY
