"""GPU paged_kv_append (bit-exact) and paged_decode_attention (1e-2 * rms)
against the oracle, including partial tail pages poisoned with NaN."""

import math

import numpy as np
import pytest
import torch

import synth
from oracle import paged as opaged

pytestmark = pytest.mark.gpu

T = 16
TOL = 1e-2


def _poison_unused(k_pool, v_pool, pt, lens):
    """NaN in every slot of every page that no sequence uses at a position < L."""
    used = np.zeros(k_pool.shape[0] * T, dtype=bool)
    for b, L in enumerate(lens):
        for t in range(int(L)):
            used[pt[b, t // T] * T + t % T] = True
    mask = ~used.reshape(k_pool.shape[0], T)
    k_pool[mask[:, None, :, None].repeat(k_pool.shape[1], 1).repeat(k_pool.shape[3], 3)] = np.nan
    v_pool[mask[:, None, :, None].repeat(v_pool.shape[1], 1).repeat(v_pool.shape[3], 3)] = np.nan


def _run(lib, seed, lens, hq=28, hkv=4, num_pages=4096, poison=True, max_context=None):
    k_pool, v_pool = synth.kv_pool(seed, num_pages, hkv)
    max_context = max_context or max(lens)
    pt = synth.page_table(seed, lens, num_pages, max_pages=math.ceil(max_context / T))
    if poison:
        _poison_unused(k_pool, v_pool, pt, lens)
    q = synth.queries(seed, len(lens), hq)
    dev = "cuda"
    out = lib.paged_decode_attention(torch.from_numpy(q).to(dev), torch.from_numpy(k_pool).to(dev),
                                     torch.from_numpy(v_pool).to(dev), torch.from_numpy(pt).to(dev),
                                     torch.tensor(lens, dtype=torch.int32, device=dev), max_context)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), (q, k_pool, v_pool, pt)


def _check(got, ref, tol=TOL):
    assert np.all(np.isfinite(got))
    for b in range(ref.shape[0]):
        rms = np.sqrt(np.mean(ref[b] ** 2))
        err = np.abs(got[b] - ref[b]).max()
        assert err <= tol * rms, "seq %d: max err %.3e > %.1e * rms %.3e" % (b, err, tol, rms)


# 1..128 pages in one cluster of at most 8 CTAs; 69 / 128 / 188 / 256 / 512 pages in one
# cluster of up to 16 CTAs (two-page rings up to two pages per warp, four-page rings
# beyond); 513 pages merge through the workspace
@pytest.mark.parametrize("L", [1, 15, 16, 17, 31, 32, 33, 1000, 1100, 2048, 3000, 4096, 8192, 8193])
def test_single_sequence_contexts(lib, L):
    got, (q, kp, vp, pt) = _run(lib, 10 + L, [L])
    ref = opaged.paged_attention_ref(q, kp, vp, pt, [L], 1 / math.sqrt(128))
    _check(got, ref)
    assert lib.device_error() == 0


def test_length_one_returns_v_exactly(lib):
    got, (q, kp, vp, pt) = _run(lib, 3, [1])
    for h in range(28):
        assert np.array_equal(got[0, h], vp[pt[0, 0], h // 7, 0].astype(np.float64))


def test_mixed_batch(lib):
    lens = [1, 17, 1000, 4096, 33, 16, 250, 15]
    got, (q, kp, vp, pt) = _run(lib, 77, lens)
    _check(got, opaged.paged_attention_ref(q, kp, vp, pt, lens, 1 / math.sqrt(128)))


@pytest.mark.parametrize("hq,hkv", [(4, 4), (4, 2), (28, 4), (32, 2)])
def test_gqa_group_sizes(lib, hq, hkv):
    lens = [37, 300, 2000]
    got, (q, kp, vp, pt) = _run(lib, 90 + hq, lens, hq=hq, hkv=hkv, num_pages=320)
    _check(got, opaged.paged_attention_ref(q, kp, vp, pt, lens, 1 / math.sqrt(128)))


def test_grid_bound_above_context(lib):
    # the grid is sized for 4096 tokens, the sequences are shorter: idle CTAs exit
    lens = [40, 1]
    got, (q, kp, vp, pt) = _run(lib, 5, lens, max_context=4096)
    _check(got, opaged.paged_attention_ref(q, kp, vp, pt, lens, 1 / math.sqrt(128)))


def test_page_permutation_invariance_bitwise(lib):
    lens = [777]
    _, (q, kp, vp, pt) = _run(lib, 8, lens, num_pages=128, poison=False)
    dev = "cuda"
    outs = []
    for perm in (np.arange(128), np.random.default_rng(2).permutation(128)):
        k2 = np.empty_like(kp)
        v2 = np.empty_like(vp)
        k2[perm] = kp
        v2[perm] = vp
        pt2 = perm[pt].astype(np.int32)
        out = lib.paged_decode_attention(torch.from_numpy(q).to(dev), torch.from_numpy(k2).to(dev),
                                         torch.from_numpy(v2).to(dev), torch.from_numpy(pt2).to(dev),
                                         torch.tensor(lens, dtype=torch.int32, device=dev), 777)
        outs.append(out.cpu())
    assert torch.equal(outs[0], outs[1])


def test_batch8_context_32768_shared_pool(lib):
    lens = [32768] * 8
    got, (q, kp, vp, pt) = _run(lib, 4242, lens, num_pages=16384 + 512, poison=False)
    ref = opaged.paged_attention_ref(q, kp, vp, pt, lens, 1 / math.sqrt(128))
    _check(got, ref)


def test_kv_append_bit_exact_including_untouched_bytes(lib):
    r = np.random.default_rng(12)
    hkv, num_pages, max_pages, B = 4, 64, 8, 5
    k_pool, v_pool = synth.kv_pool(12, num_pages, hkv)
    pt = synth.page_table(12, [max_pages * T] * B, num_pages, max_pages)
    k = r.standard_normal((B, hkv, 128)).astype(np.float16)
    v = r.standard_normal((B, hkv, 128)).astype(np.float16)
    pos = np.array([0, 15, 16, 17, 127], dtype=np.int32)
    kg, vg = torch.from_numpy(k_pool.copy()).cuda(), torch.from_numpy(v_pool.copy()).cuda()
    lib.paged_kv_append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), kg, vg, torch.from_numpy(pt).cuda(),
                        torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    opaged.kv_append_ref(k_pool, v_pool, pt, k, v, pos)
    assert np.array_equal(kg.cpu().numpy().view(np.uint16), k_pool.view(np.uint16))
    assert np.array_equal(vg.cpu().numpy().view(np.uint16), v_pool.view(np.uint16))


def test_device_checks_record_errors_without_faulting(lib):
    dev = "cuda"
    k_pool, v_pool = synth.kv_pool(1, 16, 4)
    kg, vg = torch.from_numpy(k_pool).to(dev), torch.from_numpy(v_pool).to(dev)
    q = torch.from_numpy(synth.queries(1, 1, 28)).to(dev)
    lib.device_error(clear=True)
    # context length 0 and above the launch bound
    for L in (0, 65):
        lib.paged_decode_attention(q, kg, vg, torch.zeros((1, 4), dtype=torch.int32, device=dev),
                                   torch.tensor([L], dtype=torch.int32, device=dev), 64)
        torch.cuda.synchronize()
        assert lib.device_error(clear=True) & lib.DEVERR["CONTEXT"]
    # a page id outside the pool
    pt = torch.tensor([[0, 99, 1, 2]], dtype=torch.int32, device=dev)
    lib.paged_decode_attention(q, kg, vg, pt, torch.tensor([40], dtype=torch.int32, device=dev), 64)
    torch.cuda.synchronize()
    assert lib.device_error(clear=True) & lib.DEVERR["PAGE_ID"]
    # append at a position beyond the page table, and through a bad page id
    kk = torch.zeros((1, 4, 128), dtype=torch.float16, device=dev)
    lib.paged_kv_append(kk, kk, kg, vg, torch.zeros((1, 4), dtype=torch.int32, device=dev),
                        torch.tensor([64], dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    assert lib.device_error(clear=True) & lib.DEVERR["POSITION"]
    lib.paged_kv_append(kk, kk, kg, vg, pt, torch.tensor([20], dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    assert lib.device_error(clear=True) & lib.DEVERR["PAGE_ID"]
    # the context is still usable
    got, (q2, kp, vp, pt2) = _run(lib, 2, [20], num_pages=16)
    _check(got, opaged.paged_attention_ref(q2, kp, vp, pt2, [20], 1 / math.sqrt(128)))
