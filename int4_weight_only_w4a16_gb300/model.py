"""Build a decode stream on the GPU from fp32/fp16 host tensors.

Every INT4 matrix is quantised and packed on the device by
``pack_int4_g128``; q/k/v rows are packed into one fused QKV matrix.  The
paged KV cache is a pool of ``num_pages`` pages per layer reached through one
page table (a permutation of the pool, so consecutive blocks of a sequence are
scattered), and it can be filled with given K/V rows through
``paged_kv_append`` (``fill_kv``).  Host tensors come from the caller (the seeded generators
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


def fill_kv(decoder, layer, k_rows, v_rows):
    """Write given fp16 K/V rows [L][Hkv][D] for positions 0..L-1 of one layer
    straight into the paged cache through paged_kv_append (one entry per token,
    all on the decoder's page table) -- a cache filled without running a prompt
    (the prompt pass itself is Decoder.prefill)."""
    dev = decoder.page_table.device
    L = k_rows.shape[0]
    k = torch.from_numpy(np.ascontiguousarray(k_rows)).to(dev)
    v = torch.from_numpy(np.ascontiguousarray(v_rows)).to(dev)
    pt = decoder.page_table.reshape(1, -1).expand(L, -1).contiguous()
    pos = torch.arange(L, dtype=torch.int32, device=dev)
    lw = decoder.w["layers"][layer]
    binding.paged_kv_append(k, v, lw["k_pool"], lw["v_pool"], pt, pos)


# ---------------------------------------------------------------- container

_FIELDS = ("ln1", "ln2", "bqkv")
_MATS = ("wqkv", "wo", "wgate", "wup", "wdown")


def _scales_2d(scales, n, k):
    return scales.reshape(-1)[: n * (k // 128)].view(n, k // 128)


def decoder_tensors(dec):
    """The packed weights of a Decoder as (name, device tensor) pairs, in file order."""
    cfg = dec.cfg
    h, ffn = cfg["hidden"], cfg["ffn"]
    nqkv = h + 2 * cfg["n_kv_heads"] * cfg["head_dim"]
    shapes = {"wqkv": (nqkv, h), "wo": (h, h), "wgate": (ffn, h), "wup": (ffn, h), "wdown": (h, ffn)}
    w = dec.w
    out = [("embed", w["embed"]), ("final_norm", w["final_norm"]),
           ("lm_head.packed", w["lm_head"][0]),
           ("lm_head.scales", _scales_2d(w["lm_head"][1], cfg["vocab"], h))]
    for i, lw in enumerate(w["layers"]):
        for f in _FIELDS:
            out.append(("layers.%d.%s" % (i, f), lw[f]))
        for f in _MATS:
            n, k = shapes[f]
            out.append(("layers.%d.%s.packed" % (i, f), lw[f][0]))
            out.append(("layers.%d.%s.scales" % (i, f), _scales_2d(lw[f][1], n, k)))
    return out


def save_container(path, dec):
    """Write a Decoder's packed weights (QKV rows already in the RoPE pair order)
    to a container file."""
    tensors = []
    for name, t in decoder_tensors(dec):
        a = t.detach().cpu().numpy()
        if a.dtype == np.int32 and name.endswith(".packed"):
            a = a.view(np.uint32)
        tensors.append((name, a))
    binding.container_write(path, dec.cfg, tensors)


def load_decoder(path, page_table, num_pages, max_context, device="cuda", verify=False, pdl=True):
    """Open a container written by save_container, upload every tensor into
    device memory (scales into 16-byte padded buffers) and return a Decoder with
    an empty paged KV cache of num_pages pages per layer."""
    dev = torch.device(device)
    c = binding.Container(path, verify=verify)
    try:
        cfg = dict(c.config)
        hkv, d = cfg["n_kv_heads"], cfg["head_dim"]

        def up(name, dtype=None):
            shape = c.shape(name)
            if name.endswith(".scales"):
                t = binding.scales_buffer(shape[0], shape[1] * 128, dev)
                c.upload(name, _flat_storage(t))
                return t
            t = torch.empty(shape, dtype=dtype or _torch_dtype(c, name), device=dev)
            c.upload(name, t)
            return t

        def mat(prefix):
            return (up(prefix + ".packed", torch.int32), up(prefix + ".scales"))

        layers = []
        for i in range(cfg["n_layers"]):
            p = "layers.%d." % i
            lw = {f: up(p + f) for f in _FIELDS}
            for f in _MATS:
                lw[f] = mat(p + f)
            lw["k_pool"] = torch.zeros((num_pages, hkv, PAGE_TOKENS, d), dtype=torch.float16, device=dev)
            lw["v_pool"] = torch.zeros((num_pages, hkv, PAGE_TOKENS, d), dtype=torch.float16, device=dev)
            layers.append(lw)
        weights = {"embed": up("embed"), "final_norm": up("final_norm"), "lm_head": mat("lm_head"),
                   "layers": layers}
        torch.cuda.synchronize(dev)
    finally:
        c.close()
    pt = torch.from_numpy(np.ascontiguousarray(page_table, dtype=np.int32)).to(dev)
    return binding.Decoder(cfg, weights, pt, max_context, pdl=pdl)


def _torch_dtype(c, name):
    dt = c.array(name).dtype
    return {np.dtype(np.float16): torch.float16, np.dtype(np.float32): torch.float32,
            np.dtype(np.int32): torch.int32, np.dtype(np.uint32): torch.int32}[dt]


def _flat_storage(view):
    """The padded flat buffer behind a scales_buffer view (same data pointer)."""
    n = view.untyped_storage().nbytes() // view.element_size()
    return torch.as_strided(view, (n,), (1,), view.storage_offset())
