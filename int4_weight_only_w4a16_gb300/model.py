"""Build a decode stream on the GPU from fp32/fp16 host tensors.

Every INT4 matrix is quantised and packed on the device by
``pack_int4_g128``; q/k/v rows are packed into one fused QKV matrix.  The
paged KV cache is a pool of ``num_pages`` pages per layer reached through one
page table (a permutation of the pool, so consecutive blocks of a sequence are
scattered), and it can be prefilled with given K/V rows through
``paged_kv_append``.  Host tensors come from the caller (the seeded generators
in ``synth`` for tests and benchmarks).
"""

import numpy as np
import torch

from . import binding

PAGE_TOKENS = 16


def rope_pair_order(n_heads, head_dim=128):
    """Row order that puts each rotate-half RoPE pair (dims i, i + head_dim/2)
    of every head in adjacent rows 2i, 2i+1 -- the q/k row order the fused
    QKV kernel expects (see w4_layer_weights in include/w4a16.h)."""
    half = head_dim // 2
    j = np.arange(head_dim)
    within = (j // 2) + half * (j % 2)
    return (np.arange(n_heads)[:, None] * head_dim + within[None, :]).reshape(-1)


def pack_host_matrix(w_fp32, device="cuda", flags=None):
    """Quantise + pack one fp32 host matrix on the GPU; returns (packed, scales)."""
    w = torch.from_numpy(np.ascontiguousarray(w_fp32)).to(device)
    out = binding.pack_int4_g128(w, flags=flags)
    del w
    return out


def build_decoder(cfg, small, matrices, page_table, num_pages, max_context, device="cuda", pdl=True):
    """small: dict from ``synth.model_small_tensors``; matrices: iterable of
    (layer, name, fp32 W) with layer -1 for the LM head; page_table: int32
    host array [max_pages].  Returns a ``binding.Decoder``."""
    dev = torch.device(device)
    nl = cfg["n_layers"]
    hkv, d = cfg["n_kv_heads"], cfg["head_dim"]
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    packed = [dict() for _ in range(nl)]
    lm = None
    qperm = rope_pair_order(cfg["n_q_heads"], d)
    kperm = rope_pair_order(hkv, d)
    for li, name, w in matrices:
        if name == "wq":
            w = w[qperm]
        elif name == "wk":
            w = w[kperm]
        pw = pack_host_matrix(w, dev, flags)
        if li < 0:
            lm = pw
        else:
            packed[li][name] = pw
    torch.cuda.synchronize(dev)
    if int(flags.item()) != 0:
        raise binding.W4Error(6, "pack_int4_g128 reported non-finite weights or scale overflow")
    layers = []
    for li in range(nl):
        p = packed[li]
        wqkv = (torch.cat([p["wq"][0], p["wk"][0], p["wv"][0]]).contiguous(),
                binding.padded_scales(torch.cat([p["wq"][1], p["wk"][1], p["wv"][1]])))
        sl = small["layers"][li]
        bqkv = np.concatenate([sl["bq"][qperm], sl["bk"][kperm], sl["bv"]])
        layers.append({
            "ln1": torch.from_numpy(sl["ln1"]).to(dev), "ln2": torch.from_numpy(sl["ln2"]).to(dev),
            "bqkv": torch.from_numpy(bqkv).to(dev), "wqkv": wqkv, "wo": p["wo"], "wgate": p["wg"],
            "wup": p["wu"], "wdown": p["wd"],
            "k_pool": torch.zeros((num_pages, hkv, PAGE_TOKENS, d), dtype=torch.float16, device=dev),
            "v_pool": torch.zeros((num_pages, hkv, PAGE_TOKENS, d), dtype=torch.float16, device=dev),
        })
        del packed[li]["wq"], packed[li]["wk"], packed[li]["wv"]
    weights = {"embed": torch.from_numpy(small["embed"]).to(dev),
               "final_norm": torch.from_numpy(small["final_norm"]).to(dev),
               "lm_head": lm, "layers": layers}
    pt = torch.from_numpy(np.ascontiguousarray(page_table, dtype=np.int32)).to(dev)
    return binding.Decoder(cfg, weights, pt, max_context, pdl=pdl)


def prefill(decoder, layer, k_rows, v_rows):
    """Write fp16 K/V rows [L][Hkv][D] for positions 0..L-1 of one layer through
    paged_kv_append (one entry per token, all on the decoder's page table)."""
    dev = decoder.page_table.device
    L = k_rows.shape[0]
    k = torch.from_numpy(np.ascontiguousarray(k_rows)).to(dev)
    v = torch.from_numpy(np.ascontiguousarray(v_rows)).to(dev)
    pt = decoder.page_table.reshape(1, -1).expand(L, -1).contiguous()
    pos = torch.arange(L, dtype=torch.int32, device=dev)
    lw = decoder.w["layers"][layer]
    binding.paged_kv_append(k, v, lw["k_pool"], lw["v_pool"], pt, pos)
