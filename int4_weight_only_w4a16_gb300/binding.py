"""Thin Python binding over the C ABI in ``include/w4a16.h`` (ctypes).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  There is no
fallback: if ``libw4a16.so`` is missing or a call fails, an exception is raised.
"""

import ctypes
import math
import os

import numpy as np

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4a16.so")

W4_OK = 0
STATUS_NAMES = {0: "OK", 1: "ERR_NULL", 2: "ERR_SHAPE", 3: "ERR_ALIGN", 4: "ERR_RANGE", 5: "ERR_CAPACITY",
                6: "ERR_NONFINITE", 7: "ERR_CUDA", 8: "ERR_DEVICE_CHECK", 9: "ERR_STATE", 10: "ERR_IO"}
DEVERR = {"PAGE_ID": 0x1, "POSITION": 0x2, "CONTEXT": 0x4, "TIMEOUT": 0x8, "NONFINITE": 0x10,
          "SCALE_OVF": 0x20, "TOKEN": 0x40, "NAN_LOGIT": 0x80}

_vp, _i32, _i64, _sz, _f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float


class W4Error(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), msg))
        self.status = status


class ModelConfig(ctypes.Structure):
    _fields_ = [("hidden", _i32), ("ffn", _i32), ("n_layers", _i32), ("n_q_heads", _i32), ("n_kv_heads", _i32),
                ("head_dim", _i32), ("vocab", _i32), ("rms_eps", _f32), ("rope_theta", _f32)]


class KVConfig(ctypes.Structure):
    _fields_ = [("max_context", _i32), ("num_pages", _i32), ("max_pages", _i32)]


class QMatrix(ctypes.Structure):
    _fields_ = [("packed", _vp), ("scales", _vp)]


class TensorDesc(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("dtype", _i32), ("ndim", _i32), ("dims", _i64 * 2), ("data", _vp),
                ("bytes", _sz)]


# container dtypes (W4_DT_*) <-> numpy
DT_NUMPY = {1: np.uint32, 2: np.float16, 3: np.float32, 4: np.int32}


class LayerWeights(ctypes.Structure):
    _fields_ = [("ln1", _vp), ("ln2", _vp), ("wqkv", QMatrix), ("bqkv", _vp), ("wo", QMatrix),
                ("wgate", QMatrix), ("wup", QMatrix), ("wdown", QMatrix)]


class KVLayer(ctypes.Structure):
    _fields_ = [("k_pool", _vp), ("v_pool", _vp)]


_SIGS = {
    "w4_last_error": (ctypes.c_char_p, []),
    "w4_device_error": (_i32, [ctypes.POINTER(ctypes.c_int32), _i32]),
    "w4_sm_count": (_i32, []),
    "w4_pack_int4_g128": (_i32, [_vp, _i64, _i64, _vp, _vp, _vp, _vp]),
    "w4_gemv_workspace_size": (_sz, [_i32, _i64, _i64]),
    "w4_gemv_w4a16": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "w4_gemv_tune": (_i32, [_i32]),
    "w4_paged_kv_append": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _vp, _i32, _vp, _vp]),
    "w4_attention_workspace_size": (_sz, [_i32, _i32, _i32, _i32]),
    "w4_paged_decode_attention": (_i32, [_vp, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _i32, _vp, _i32, _vp, _i32,
                                         _vp, _vp, _sz, _vp]),
    "w4_paged_decode_attention_noalloc_max_scratch": (_sz, []),
    "w4_paged_decode_attention_noalloc": (_i32, [_vp, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _i32, _vp, _i32, _vp,
                                                 _i32, _vp, _vp]),
    "w4_model_create": (_i32, [ctypes.POINTER(ModelConfig), ctypes.POINTER(LayerWeights), _vp, _vp, QMatrix,
                               ctypes.POINTER(_vp)]),
    "w4_kv_workspace_size": (_sz, [_vp, ctypes.POINTER(KVConfig)]),
    "w4_kv_create": (_i32, [_vp, ctypes.POINTER(KVConfig), ctypes.POINTER(KVLayer), _vp, _vp, _vp, _sz, _vp,
                            ctypes.POINTER(_vp)]),
    "w4_kv_destroy": (None, [_vp]),
    "w4_model_destroy": (None, [_vp]),
    "w4_model_set_pdl": (_i32, [_vp, _i32]),
    "w4_container_write": (_i32, [ctypes.c_char_p, ctypes.POINTER(ModelConfig), ctypes.POINTER(TensorDesc), _i32]),
    "w4_container_open": (_i32, [ctypes.c_char_p, _i32, ctypes.POINTER(_vp)]),
    "w4_container_close": (None, [_vp]),
    "w4_container_config": (_i32, [_vp, ctypes.POINTER(ModelConfig)]),
    "w4_container_count": (_i32, [_vp]),
    "w4_container_tensor": (_i32, [_vp, _i32, ctypes.POINTER(TensorDesc)]),
    "w4_container_find": (_i32, [_vp, ctypes.c_char_p, ctypes.POINTER(_i32)]),
    "w4_container_upload": (_i32, [_vp, _i32, _vp, _sz, _vp]),
    "w4_decode_step": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp]),
    "w4_decode_graph_create": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.POINTER(_vp)]),
    "w4_decode_graph_launch": (_i32, [_vp, _vp]),
    "w4_decode_graph_destroy": (None, [_vp]),
    "w4_decode_launches_per_step": (_i32, [_vp]),
    "w4_decode_launch_kernel": (_i32, [_vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp]),
    "w4_prefill_workspace_size": (_sz, [_vp, _vp, _i32]),
    "w4_prefill": (_i32, [_vp, _vp, _vp, _sz, _vp, _i32, _i32, _vp, _vp, _vp]),
    "w4_gemm_workspace_size": (_sz, [_i32, _i32, _i32]),
    "w4_gemm_plan": (_i32, [_i32, _i32, _i32, _i32, _i32, _vp]),
    "w4_gemv_plan": (_i32, [_i32, ctypes.c_int64, ctypes.c_int64, _vp]),
    "w4_attention_plan": (_i32, [_i32, _i32, _i32, _i32, _i32, _i32, _vp]),
    "w4_gemm_w4a16": (_i32, [_vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
}

KERNELS = {"embed": 0, "qkv": 1, "attention": 2, "o": 3, "gate_up": 4, "down": 5, "lm_head": 6}

_lib = None


def load(path=LIB_PATH):
    """Load libw4a16.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError("libw4a16.so not found at %s: run __graft_entry__.build() first" % path)
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status):
    if status != W4_OK:
        raise W4Error(status, load().w4_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(t, dtype, name):
    if t.device.type != "cuda" or t.dtype != dtype or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dtype))
    return t


def device_error(clear=True):
    """OR of W4_DEVERR_* codes recorded by kernels (synchronous)."""
    v = ctypes.c_int32(0)
    _check(load().w4_device_error(ctypes.byref(v), 1 if clear else 0))
    return v.value


def sm_count():
    return load().w4_sm_count()


# ---------------------------------------------------------------------- pack

def scales_buffer(n, k, device):
    """fp16 [n][k/128] view over storage padded to a multiple of 16 bytes (the
    GEMV reads the scales in whole 16-byte blocks)."""
    count = n * max(1, k // 128)
    flat = torch.zeros(((count + 7) // 8) * 8, dtype=torch.float16, device=device)
    return flat[:count].view(n, max(1, k // 128))


def padded_scales(t):
    """Copy of a [rows][groups] fp16 scale tensor into 16-byte padded storage."""
    out = scales_buffer(t.shape[0], t.shape[1] * 128, t.device)
    out.copy_(t)
    return out


def pack_int4_g128(w, flags=None, stream=None):
    """fp32 W [N][K] on the GPU -> (packed int32 [N][K/8] holding uint32 words, scales fp16 [N][K/128])."""
    _cuda(w, torch.float32, "w")
    n, k = w.shape
    packed = torch.empty((n, k // 8), dtype=torch.int32, device=w.device)
    scales = scales_buffer(n, k, w.device)
    _check(load().w4_pack_int4_g128(_ptr(w), n, k, _ptr(packed), _ptr(scales), _ptr(flags), _stream(stream)))
    return packed, scales


# ---------------------------------------------------------------------- GEMV

def gemv_workspace(m, n, k, device="cuda"):
    nbytes = load().w4_gemv_workspace_size(m, n, k)
    if nbytes == 0:
        raise W4Error(2, "gemv_workspace: bad shape")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def gemv_tune(variant=0):
    """GEMV variant: 0 default, 1 mma.sync kernel at every batch, 2 W4A8 at batch 1, 3 tcgen05 kernel at
    every batch (see w4_gemv_tune)."""
    _check(load().w4_gemv_tune(variant))


def gemv_w4a16(x, packed, scales, bias=None, residual=None, out=None, workspace=None, stream=None):
    """y = W_deq x (+ bias) (+ residual); x fp16 [M][K] (or [K]), returns fp16 [M][N] (or [N])."""
    one_d = x.dim() == 1
    x2 = x.reshape(1, -1) if one_d else x
    _cuda(x2, torch.float16, "x")
    m, k = x2.shape
    n = packed.shape[0]
    if out is None:
        out = torch.empty((m, n), dtype=torch.float16, device=x.device)
    if workspace is None:
        workspace = gemv_workspace(m, n, k, x.device)
    _check(load().w4_gemv_w4a16(_ptr(x2), m, n, k, _ptr(packed), _ptr(scales), _ptr(bias), _ptr(residual),
                                _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out.reshape(-1) if one_d else out


def gemm_w4a16(x, packed, scales, out=None, workspace=None, stream=None):
    """y = x W_deq^T for n activation rows: x fp16 [n][K] -> fp32 [n][N] (tcgen05 kernel, exact INT4 codes,
    each scale group's sum scaled in fp32)."""
    _cuda(x, torch.float16, "x")
    n, k = x.shape
    nrows = packed.shape[0]
    if out is None:
        out = torch.empty((n, nrows), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(max(load().w4_gemm_workspace_size(n, nrows, k), 16), dtype=torch.uint8,
                                device=x.device)
    _check(load().w4_gemm_w4a16(_ptr(x), n, nrows, k, _ptr(packed), _ptr(scales), _ptr(out), _ptr(workspace),
                                workspace.numel(), _stream(stream)))
    return out


def attention_plan(b, hq, hkv, max_context, sms, max_cluster):
    """How the paged decode attention divides its work (host only when sms and
    max_cluster are given): a dict of cluster, ppw, stages, splits, grid (x, y, z)
    and workspace bytes."""
    out = (ctypes.c_int64 * 8)()
    _check(load().w4_attention_plan(b, hq, hkv, max_context, sms, max_cluster, ctypes.cast(out, ctypes.c_void_p)))
    v = list(out)
    return {"cluster": v[0], "ppw": v[1], "stages": v[2], "splits": v[3], "grid": tuple(v[4:7]), "ws_bytes": v[7]}


def gemv_plan(matrices, n, k):
    """How the batch-1 streaming GEMV lays out `matrices` (1, or 2 for gate/up)
    matrices of n x k (host only): a dict of grid, cw, hpr, rg, gs, ns, wbytes,
    sbytes, smem; grid 0 when the rows are too long for its ring."""
    out = (ctypes.c_int32 * 9)()
    _check(load().w4_gemv_plan(matrices, n, k, ctypes.cast(out, ctypes.c_void_p)))
    keys = ("grid", "cw", "hpr", "rg", "gs", "ns", "wbytes", "sbytes", "smem")
    return dict(zip(keys, list(out)))


def gemm_plan(epilogue, n, N, K, sms):
    """How the GEMM divides n x N x K among CTAs on `sms` SMs (host only): a dict of
    bn, tok_tiles, row_tiles, kb_per_split, splits, mode (0 split K, 1 stream-K,
    2 persistent), ctas, stages."""
    out = (ctypes.c_int32 * 8)()
    _check(load().w4_gemm_plan(epilogue, n, N, K, sms, ctypes.cast(out, ctypes.c_void_p)))
    keys = ("bn", "tok_tiles", "row_tiles", "kb_per_split", "splits", "mode", "ctas", "stages")
    return dict(zip(keys, list(out)))


# ------------------------------------------------------------------ paged KV

def paged_kv_append(k, v, k_pool, v_pool, page_table, positions, stream=None):
    """k, v fp16 [B][Hkv][128]; pools fp16 [P][Hkv][16][128]; page_table int32 [B][max_pages]; positions int32 [B]."""
    b, hkv, d = k.shape
    _check(load().w4_paged_kv_append(_ptr(k), _ptr(v), b, hkv, d, _ptr(k_pool), _ptr(v_pool), k_pool.shape[0],
                                     _ptr(page_table), page_table.shape[1], _ptr(positions), _stream(stream)))


def attention_workspace(b, hq, hkv, max_context, device="cuda"):
    nbytes = load().w4_attention_workspace_size(b, hq, hkv, max_context)
    return torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=device)


def paged_decode_attention(q, k_pool, v_pool, page_table, context_lens, max_context, scale=None, out=None,
                           workspace=None, stream=None):
    """q fp16 [B][Hq][128] -> out fp16 [B][Hq][128] over the paged cache."""
    b, hq, d = q.shape
    hkv = k_pool.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = attention_workspace(b, hq, hkv, max_context, q.device)
    _check(load().w4_paged_decode_attention(_ptr(q), b, hq, hkv, d, scale, _ptr(k_pool), _ptr(v_pool),
                                            k_pool.shape[0], _ptr(page_table), page_table.shape[1],
                                            _ptr(context_lens), max_context, _ptr(out), _ptr(workspace),
                                            workspace.numel(), _stream(stream)))
    return out


def paged_decode_attention_noalloc(q, k_pool, v_pool, page_table, context_lens, max_context, scale=None, out=None,
                                   stream=None):
    """paged_decode_attention for callers that cannot allocate: the library's
    fixed scratch array replaces the workspace (calls must not overlap)."""
    b, hq, d = q.shape
    hkv = k_pool.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _check(load().w4_paged_decode_attention_noalloc(_ptr(q), b, hq, hkv, d, scale, _ptr(k_pool), _ptr(v_pool),
                                                    k_pool.shape[0], _ptr(page_table), page_table.shape[1],
                                                    _ptr(context_lens), max_context, _ptr(out), _stream(stream)))
    return out


# -------------------------------------------------------------------- decode

class Model:
    """The weights of one model (w4_model): shared, read-only, by every
    Sequence run over them.

    ``weights`` holds torch CUDA tensors: ``embed`` fp16 [V][H], ``final_norm``
    fp16 [H], ``lm_head`` (packed, scales) and ``layers``: a list of dicts with
    ln1, ln2, bqkv (fp16), wqkv, wo, wgate, wup, wdown ((packed, scales)
    pairs); other keys are ignored.
    """

    def __init__(self, cfg, weights, pdl=True):
        self.cfg = dict(cfg)
        self.w = weights  # keeps the tensors alive
        lib = load()
        c = ModelConfig(cfg["hidden"], cfg["ffn"], cfg["n_layers"], cfg["n_q_heads"], cfg["n_kv_heads"],
                        cfg["head_dim"], cfg["vocab"], cfg["rms_eps"], cfg["rope_theta"])
        arr = (LayerWeights * cfg["n_layers"])()
        for i, lw in enumerate(weights["layers"]):
            q = lambda pair: QMatrix(pair[0].data_ptr(), pair[1].data_ptr())  # noqa: E731
            arr[i] = LayerWeights(lw["ln1"].data_ptr(), lw["ln2"].data_ptr(), q(lw["wqkv"]), lw["bqkv"].data_ptr(),
                                  q(lw["wo"]), q(lw["wgate"]), q(lw["wup"]), q(lw["wdown"]))
        lm = QMatrix(weights["lm_head"][0].data_ptr(), weights["lm_head"][1].data_ptr())
        h = ctypes.c_void_p()
        _check(lib.w4_model_create(ctypes.byref(c), arr, _ptr(weights["embed"]), _ptr(weights["final_norm"]), lm,
                                   ctypes.byref(h)))
        self.handle = h
        _check(lib.w4_model_set_pdl(h, 1 if pdl else 0))
        self.launches_per_step = lib.w4_decode_launches_per_step(h)

    def close(self):
        if getattr(self, "handle", None) is not None:
            load().w4_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Sequence:
    """One sequence's paged KV cache and decode state (w4_kv) over a Model.

    ``pools``: per layer a (k_pool, v_pool) pair of fp16 CUDA tensors
    [num_pages][Hkv][16][128]; ``page_table``: int32 CUDA tensor [max_pages]
    (shared by all layers).  The sequence owns its position, greedy token and
    logits buffers (``pos``, ``token``, ``logits``) and its decode workspace.
    """

    def __init__(self, model, pools, page_table, max_context):
        self.model = model
        self.cfg = model.cfg
        self.pools = pools
        self.page_table = page_table
        lib = load()
        dev = page_table.device
        kc = KVConfig(int(max_context), pools[0][0].shape[0], page_table.shape[0])
        arr = (KVLayer * len(pools))()
        for i, (kp, vp) in enumerate(pools):
            arr[i] = KVLayer(kp.data_ptr(), vp.data_ptr())
        nbytes = lib.w4_kv_workspace_size(model.handle, ctypes.byref(kc))
        if nbytes == 0:
            raise W4Error(4, "Sequence: bad cache sizes (max_context %d, %d pages, %d table entries)"
                          % (kc.max_context, kc.num_pages, kc.max_pages))
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.token = torch.zeros(1, dtype=torch.int32, device=dev)
        self.pos = torch.zeros(1, dtype=torch.int32, device=dev)
        self.logits = torch.zeros(self.cfg["vocab"], dtype=torch.float32, device=dev)
        h = ctypes.c_void_p()
        _check(lib.w4_kv_create(model.handle, ctypes.byref(kc), arr, _ptr(page_table), _ptr(self.pos),
                                _ptr(self.workspace), self.workspace.numel(), _stream(), ctypes.byref(h)))
        self.kv = h
        self.graph = None
        self.launches_per_step = model.launches_per_step

    def prefill(self, tokens, start_pos=0, with_logits=True, stream=None):
        """Run the prompt ``tokens`` (int32 CUDA tensor [n]) at positions start_pos ..
        start_pos + n - 1 in one pass; afterwards self.token holds the greedy next
        token and self.pos = start_pos + n, ready for step()/replay()."""
        if tokens.dtype != torch.int32 or not tokens.is_cuda or tokens.dim() != 1:
            raise W4Error(2, "prefill: tokens must be a 1-D int32 CUDA tensor")
        tokens = tokens.contiguous()
        lib = load()
        need = lib.w4_prefill_workspace_size(self.model.handle, self.kv, tokens.numel())
        ws = getattr(self, "prefill_workspace", None)
        if ws is None or ws.numel() < need:
            self.prefill_workspace = ws = torch.empty(max(need, 16), dtype=torch.uint8, device=tokens.device)
        _check(lib.w4_prefill(self.model.handle, self.kv, _ptr(ws), ws.numel(), _ptr(tokens), tokens.numel(),
                              int(start_pos), _ptr(self.token), _ptr(self.logits) if with_logits else None,
                              _stream(stream)))

    def set_state(self, token, pos):
        self.token.fill_(int(token))
        self.pos.fill_(int(pos))

    def step(self, with_logits=True, stream=None):
        """One eager decode step: token <- argmax, pos += 1 (all on the device)."""
        _check(load().w4_decode_step(self.model.handle, self.kv, _ptr(self.token), _ptr(self.token),
                                     _ptr(self.logits) if with_logits else None, _stream(stream)))

    def capture(self, with_logits=True, stream=None):
        """Capture one step as a CUDA graph on a side stream (replaces any previous graph)."""
        self.release_graph()
        s = stream or torch.cuda.Stream(device=self.token.device)
        g = ctypes.c_void_p()
        _check(load().w4_decode_graph_create(self.model.handle, self.kv, _ptr(self.token), _ptr(self.token),
                                             _ptr(self.logits) if with_logits else None,
                                             ctypes.c_void_p(s.cuda_stream), ctypes.byref(g)))
        self.graph = g

    def launch_kernel(self, name, layer=0, with_logits=True, stream=None):
        """Launch one kernel of the step alone (profiling): see KERNELS."""
        _check(load().w4_decode_launch_kernel(self.model.handle, self.kv, KERNELS[name], layer, _ptr(self.token),
                                              _ptr(self.token), _ptr(self.logits) if with_logits else None,
                                              _stream(stream)))

    def replay(self, stream=None):
        _check(load().w4_decode_graph_launch(self.graph, _stream(stream)))

    def release_graph(self):
        if self.graph is not None:
            load().w4_decode_graph_destroy(self.graph)
            self.graph = None

    def close(self):
        self.release_graph()
        if getattr(self, "kv", None) is not None:
            load().w4_kv_destroy(self.kv)
            self.kv = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Decoder(Sequence):
    """A Model and one Sequence over it, built from one weights dict whose layer
    dicts also hold that sequence's ``k_pool`` and ``v_pool``; more sequences
    over the same weights come from ``new_sequence``."""

    def __init__(self, cfg, weights, page_table, max_context, pdl=True):
        self.w = weights
        model = Model(cfg, weights, pdl=pdl)
        super().__init__(model, [(lw["k_pool"], lw["v_pool"]) for lw in weights["layers"]], page_table, max_context)

    def new_sequence(self, page_table, num_pages, max_context):
        """Another sequence over the same weights, with zeroed pools of its own."""
        hkv, d = self.cfg["n_kv_heads"], self.cfg["head_dim"]
        dev = page_table.device
        pools = [(torch.zeros((num_pages, hkv, 16, d), dtype=torch.float16, device=dev),
                  torch.zeros((num_pages, hkv, 16, d), dtype=torch.float16, device=dev))
                 for _ in range(self.cfg["n_layers"])]
        return Sequence(self.model, pools, page_table, max_context)

    def close(self):
        super().close()
        self.model.close()


# ------------------------------------------------------------------ container

_NP_DT = {np.dtype(np.uint32): 1, np.dtype(np.float16): 2, np.dtype(np.float32): 3, np.dtype(np.int32): 4}


def _config_struct(cfg):
    return ModelConfig(cfg["hidden"], cfg["ffn"], cfg["n_layers"], cfg["n_q_heads"], cfg["n_kv_heads"],
                       cfg["head_dim"], cfg["vocab"], cfg["rms_eps"], cfg["rope_theta"])


def container_write(path, cfg, tensors):
    """Write a container: tensors is a list of (name, 1-D or 2-D host numpy array of
    uint32 / float16 / float32 / int32)."""
    arrays = [(n, np.ascontiguousarray(a)) for n, a in tensors]
    descs = (TensorDesc * len(arrays))()
    names = [n.encode() for n, _ in arrays]
    for i, (n, a) in enumerate(arrays):
        if a.dtype not in _NP_DT or a.ndim not in (1, 2):
            raise W4Error(2, "container_write: %s is %s with %d dims" % (n, a.dtype, a.ndim))
        dims = (_i64 * 2)(a.shape[0], a.shape[1] if a.ndim == 2 else 0)
        descs[i] = TensorDesc(names[i], _NP_DT[a.dtype], a.ndim, dims, a.ctypes.data, a.nbytes)
    c = _config_struct(cfg)
    _check(load().w4_container_write(os.fsencode(path), ctypes.byref(c), descs, len(arrays)))


class Container:
    """A mapped container file: config, tensors as read-only numpy views of the
    mapping, and device uploads."""

    def __init__(self, path, verify=False):
        h = _vp()
        _check(load().w4_container_open(os.fsencode(path), 1 if verify else 0, ctypes.byref(h)))
        self.handle = h
        c = ModelConfig()
        _check(load().w4_container_config(h, ctypes.byref(c)))
        self.config = {f: getattr(c, f) for f, _ in ModelConfig._fields_}
        self.names = []
        for i in range(load().w4_container_count(h)):
            d = TensorDesc()
            _check(load().w4_container_tensor(h, i, ctypes.byref(d)))
            self.names.append(d.name.decode())

    def _desc(self, name):
        idx = _i32()
        _check(load().w4_container_find(self.handle, name.encode(), ctypes.byref(idx)))
        d = TensorDesc()
        _check(load().w4_container_tensor(self.handle, idx.value, ctypes.byref(d)))
        return idx.value, d

    def shape(self, name):
        _, d = self._desc(name)
        return (d.dims[0],) if d.ndim == 1 else (d.dims[0], d.dims[1])

    def array(self, name):
        """Read-only numpy view of a tensor (valid while the container is open)."""
        _, d = self._desc(name)
        raw = (ctypes.c_uint8 * d.bytes).from_address(d.data)
        a = np.frombuffer(raw, dtype=DT_NUMPY[d.dtype])
        return a.reshape(self.shape(name))

    def upload(self, name, dst, stream=None):
        """Copy a tensor into the device tensor dst (at least as many bytes)."""
        idx, d = self._desc(name)
        if not dst.is_cuda or not dst.is_contiguous():
            raise W4Error(2, "upload: %s needs a contiguous CUDA destination" % name)
        _check(load().w4_container_upload(self.handle, idx, _ptr(dst), dst.numel() * dst.element_size(),
                                          _stream(stream)))

    def close(self):
        if getattr(self, "handle", None) is not None:
            load().w4_container_close(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
