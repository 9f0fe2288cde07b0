"""CPU checks of the C ABI: the library builds, loads, exports every function
declared in include/w4a16.h, and host-side validation rejects bad arguments
before anything is launched (no GPU needed: these calls return before any
kernel launch or device access)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def clib():
    from int4_weight_only_w4a16_gb300 import build, binding
    build.build()
    return binding.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(w4_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("w4_pack_int4_g128", "w4_gemv_w4a16", "w4_paged_kv_append", "w4_paged_decode_attention",
              "w4_decode_step"):
        assert n in names


def test_every_declared_function_is_exported(clib):
    for n in _declared_functions():
        assert hasattr(clib, n), n


def test_binding_signatures_cover_the_header():
    from int4_weight_only_w4a16_gb300 import binding
    assert set(_declared_functions()) <= set(binding._SIGS)


# fake, never-dereferenced device addresses for host-validation tests
A = ctypes.c_void_p(0x10000)      # 16-byte aligned
B = ctypes.c_void_p(0x20000)
ODD = ctypes.c_void_p(0x10008)    # 8-byte aligned only


def test_pack_host_validation(clib):
    assert clib.w4_pack_int4_g128(None, 4, 128, A, B, None, None) == 1          # NULL
    assert clib.w4_pack_int4_g128(A, 4, 100, B, A, None, None) == 2            # K % 128
    assert b"multiple of 128" in clib.w4_last_error()
    assert clib.w4_pack_int4_g128(A, 0, 128, B, A, None, None) == 2            # N = 0
    assert clib.w4_pack_int4_g128(ODD, 4, 128, B, A, None, None) == 3          # misaligned


def test_gemv_host_validation(clib):
    ws = ctypes.c_void_p(0x40000)
    big = 1 << 30
    assert clib.w4_gemv_w4a16(None, 1, 16, 128, A, B, None, None, B, ws, big, None) == 1
    assert clib.w4_gemv_w4a16(A, 0, 16, 128, A, B, None, None, B, ws, big, None) == 2    # m = 0
    assert clib.w4_gemv_w4a16(A, 17, 16, 128, A, B, None, None, B, ws, big, None) == 2   # m > 16
    assert clib.w4_gemv_w4a16(A, 1, 16, 130, A, B, None, None, B, ws, big, None) == 2    # K % 128
    assert clib.w4_gemv_w4a16(ODD, 1, 16, 128, A, B, None, None, B, ws, big, None) == 3  # alignment
    assert clib.w4_gemv_w4a16(A, 1, 16, 128, A, B, None, None, A, ws, big, None) == 4    # y aliases x
    assert clib.w4_gemv_w4a16(A, 1, 16, 128, A, B, None, None, B, ws, 0, None) == 5      # workspace
    assert clib.w4_gemv_workspace_size(0, 16, 128) == 0
    assert clib.w4_gemv_workspace_size(1, 16, 128) > 0


def test_attention_host_validation(clib):
    ws = ctypes.c_void_p(0x40000)
    big = 1 << 30
    args = lambda **kw: [kw.get("q", A), kw.get("b", 1), kw.get("hq", 28), kw.get("hkv", 4), kw.get("d", 128),  # noqa: E731
                         ctypes.c_float(kw.get("scale", 0.088)), kw.get("kp", A), kw.get("vp", B), 64, A, 8,
                         B, kw.get("maxctx", 128), kw.get("out", B), ws, kw.get("wsb", big), None]
    f = clib.w4_paged_decode_attention
    assert f(*args(q=None)) == 1
    assert f(*args(d=64)) == 2
    assert f(*args(hq=30)) == 2              # hq % hkv != 0
    assert f(*args(hq=68)) == 2              # group > 16
    assert f(*args(maxctx=129)) == 4         # beyond 16 * max_pages
    assert f(*args(kp=ODD)) == 3
    assert f(*args(wsb=0)) == 5
    assert f(*args(scale=float("nan"))) == 4


def test_kv_append_host_validation(clib):
    f = clib.w4_paged_kv_append
    assert f(None, B, 1, 4, 128, A, B, 64, A, 8, B, None) == 1
    assert f(A, B, 1, 4, 64, A, B, 64, A, 8, B, None) == 2
    assert f(A, B, 0, 4, 128, A, B, 64, A, 8, B, None) == 2
    assert f(ODD, B, 1, 4, 128, A, B, 64, A, 8, B, None) == 3


def test_model_create_host_validation(clib):
    from int4_weight_only_w4a16_gb300 import binding
    cfg = binding.ModelConfig(512, 1280, 1, 4, 2, 128, 1000, 1e-6, 1e6)
    layer = (binding.LayerWeights * 1)()
    q = binding.QMatrix(0x10000, 0x20000)
    h = ctypes.c_void_p()
    # null layer pointers
    assert clib.w4_model_create(ctypes.byref(cfg), layer, A, A, q, ctypes.byref(h)) == 1
    bad = binding.ModelConfig(512, 1280, 1, 4, 2, 64, 1000, 1e-6, 1e6)  # head_dim 64
    assert clib.w4_model_create(ctypes.byref(bad), layer, A, A, q, ctypes.byref(h)) == 2
    assert clib.w4_model_create(ctypes.byref(cfg), layer, A, A, q, None) == 1


def test_kv_host_validation(clib):
    # the cache handle is refused before it touches a device: null pointers, and
    # sizes checked against each other (max_context <= 16 * max_pages)
    from int4_weight_only_w4a16_gb300 import binding
    h = ctypes.c_void_p()
    kc = binding.KVConfig(64, 8, 4)
    layers = (binding.KVLayer * 1)(binding.KVLayer(0x10000, 0x20000))
    assert clib.w4_kv_create(None, ctypes.byref(kc), layers, A, B, A, 1 << 20, None, ctypes.byref(h)) == 1
    assert clib.w4_kv_workspace_size(None, ctypes.byref(kc)) == 0
    assert clib.w4_decode_step(None, None, A, A, None, None) == 1
    assert clib.w4_decode_graph_create(None, None, A, A, None, A, ctypes.byref(h)) == 1
    assert clib.w4_decode_launch_kernel(None, None, 1, 0, A, A, None, None) == 1
    assert clib.w4_decode_launches_per_step(None) == 0


def test_gemm_host_validation(clib):
    # W4A16 GEMM of the prompt pass: rejected before any launch
    assert clib.w4_gemm_w4a16(None, 4, 128, 128, A, B, A, B, 1 << 20, None) == 1              # NULL x
    assert clib.w4_gemm_w4a16(A, 4, 200, 128, B, A, B, A, 1 << 20, None) == 2                 # N % 128
    assert clib.w4_gemm_w4a16(A, 0, 128, 128, B, A, B, A, 1 << 20, None) == 2                 # n = 0
    assert clib.w4_gemm_w4a16(ODD, 4, 128, 128, B, A, B, A, 1 << 20, None) == 3               # misaligned x
    assert clib.w4_gemm_workspace_size(0, 128, 128) == 0


def test_prefill_host_validation(clib):
    # null model / workspaces / tokens are refused before anything touches a device
    assert clib.w4_prefill(None, None, B, 1 << 20, A, 4, 0, B, None, None) == 1
    assert clib.w4_prefill_workspace_size(None, None, 16) == 0
