"""A decoder written to the model container and loaded back decodes exactly
like the one built in memory: every uploaded weight is bitwise equal, and
the same prefill + teacher-forced steps give bitwise equal logits and tokens."""

import numpy as np
import pytest
import torch

import synth
from int4_weight_only_w4a16_gb300 import model as gmodel

pytestmark = pytest.mark.gpu


def _build(cfg, seed, max_context, num_pages):
    small = synth.model_small_tensors(seed, cfg)
    mats = [(li, n, synth.model_matrix(seed, cfg, li, n)) for li in range(cfg["n_layers"]) for n in synth.MATRICES]
    mats.append((-1, "lm_head", synth.model_matrix(seed, cfg, -1, "lm_head")))
    pt = synth.page_table(seed, [max_context], num_pages, max_context // 16)[0]
    return gmodel.build_decoder(cfg, small, mats, pt, num_pages=num_pages, max_context=max_context), pt


def _prefill(dec, cfg, seed, n):
    for li in range(cfg["n_layers"]):
        k, v = synth.prefill_kv(seed, cfg, li, n)
        gmodel.fill_kv(dec, li, k, v)


def test_container_round_trip_decodes_identically(lib, tmp_path):
    cfg = dict(synth.TINY)
    a, pt = _build(cfg, 21, 128, 32)
    path = str(tmp_path / "tiny.w4c")
    gmodel.save_container(path, a)
    b = gmodel.load_decoder(path, pt, num_pages=32, max_context=128, verify=True)
    try:
        ta, tb = gmodel.decoder_tensors(a), gmodel.decoder_tensors(b)
        assert [n for n, _ in ta] == [n for n, _ in tb]
        for (n, x), (_, y) in zip(ta, tb):
            assert x.dtype == y.dtype and x.shape == y.shape, n
            assert torch.equal(x.view(torch.uint8) if x.dtype != torch.int32 else x,
                               y.view(torch.uint8) if y.dtype != torch.int32 else y), n
        for dec in (a, b):
            _prefill(dec, cfg, 22, 40)
        torch.cuda.synchronize()
        seq = []
        for dec in (a, b):
            dec.set_state(7, 40)
            toks, logits = [], []
            for _ in range(5):
                dec.step()
                toks.append(int(dec.token.item()))
                logits.append(dec.logits.clone())
            seq.append((toks, torch.stack(logits)))
        assert seq[0][0] == seq[1][0]
        assert torch.equal(seq[0][1], seq[1][1])
        assert lib.device_error() == 0
    finally:
        a.close()
        b.close()
