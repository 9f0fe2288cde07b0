"""The model container (own on-disk format): CPU round trip and validation.

The writer and the mapped reader are host code, so these run without a GPU:
bit-exact round trip of every dtype, the stored config, page alignment of
the blobs, and rejection of a wrong magic, a truncated file, a flipped
header byte and (with verify) a flipped blob byte.
"""

import os
import zlib

import numpy as np
import pytest

import synth
from int4_weight_only_w4a16_gb300 import binding as bd

CFG = dict(synth.TINY)


def _tensors(seed):
    rng = np.random.default_rng(seed)
    return [
        ("layers.0.wqkv.packed", rng.integers(0, 2 ** 32, size=(64, 16), dtype=np.uint32)),
        ("layers.0.wqkv.scales", rng.normal(size=(64, 1)).astype(np.float16)),
        ("embed", rng.normal(size=(1000, 512)).astype(np.float16)),
        ("final_norm", rng.normal(size=(512,)).astype(np.float16)),
        ("counts", rng.integers(-5, 5, size=(3,), dtype=np.int32)),
        ("stats", rng.normal(size=(7, 5)).astype(np.float32)),
    ]


@pytest.fixture()
def written(host_lib, tmp_path):
    path = str(tmp_path / "model.w4c")
    ts = _tensors(1)
    bd.container_write(path, CFG, ts)
    return path, ts


def test_round_trip_is_bit_exact(written):
    path, ts = written
    c = bd.Container(path, verify=True)
    try:
        assert c.names == [n for n, _ in ts]
        for n, a in ts:
            b = c.array(n)
            assert b.dtype == a.dtype and b.shape == a.shape
            assert np.array_equal(b.view(np.uint8), a.view(np.uint8)), n
        for k in ("hidden", "ffn", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "vocab"):
            assert c.config[k] == CFG[k]
        assert c.config["rms_eps"] == np.float32(CFG["rms_eps"])
        assert c.config["rope_theta"] == np.float32(CFG["rope_theta"])
    finally:
        c.close()


def test_blobs_are_page_aligned_and_file_size_matches(written):
    path, ts = written
    raw = open(path, "rb").read()
    assert raw[:8] == b"W4A16MC\0"
    assert len(raw) % 4096 == 0
    n = int.from_bytes(raw[12:16], "little")
    assert n == len(ts)
    assert int.from_bytes(raw[16:24], "little") == len(raw)
    for i in range(n):
        e = raw[4096 + 112 * i: 4096 + 112 * (i + 1)]
        off = int.from_bytes(e[88:96], "little")
        size = int.from_bytes(e[96:104], "little")
        assert off % 4096 == 0 and off + size <= len(raw)
        assert raw[off:off + size] == np.ascontiguousarray(ts[i][1]).tobytes()


def _corrupt(path, offset, new=None, truncate=None):
    raw = bytearray(open(path, "rb").read())
    if truncate is not None:
        raw = raw[:truncate]
    else:
        raw[offset] = new if new is not None else raw[offset] ^ 0xFF
    with open(path, "wb") as f:
        f.write(raw)


@pytest.mark.parametrize("what", ["magic", "header_crc", "truncated", "blob_crc"])
def test_rejects_damaged_files(written, what):
    path, ts = written
    if what == "magic":
        _corrupt(path, 0, ord("X"))
    elif what == "header_crc":
        _corrupt(path, 30)              # a config byte: the header CRC no longer matches
    elif what == "truncated":
        _corrupt(path, 0, truncate=os.path.getsize(path) - 4096)
    else:
        raw = open(path, "rb").read()
        off = int.from_bytes(raw[4096 + 88: 4096 + 96], "little")
        _corrupt(path, off + 5)         # first tensor's payload
        bd.Container(path, verify=False).close()   # structure still valid without verify
    with pytest.raises(bd.W4Error) as e:
        bd.Container(path, verify=True)
    assert e.value.status == 10        # W4_ERR_IO


def test_writer_rejects_bad_descriptors(host_lib, tmp_path):
    path = str(tmp_path / "bad.w4c")
    a = np.zeros((4, 4), np.float16)
    with pytest.raises(bd.W4Error):
        bd.container_write(path, CFG, [("dup", a), ("dup", a)])
    with pytest.raises(bd.W4Error):
        bd.container_write(path, CFG, [("x" * 64, a)])
    with pytest.raises(bd.W4Error):
        bd.container_write(path, CFG, [("f64", np.zeros(3, np.float64))])
    with pytest.raises(bd.W4Error):
        bd.Container(str(tmp_path / "missing.w4c"))


def test_crcs_match_an_independent_crc32(written):
    # header and blob CRCs are the IEEE 802.3 CRC-32 that zlib also implements
    path, ts = written
    raw = open(path, "rb").read()
    assert int.from_bytes(raw[60:64], "little") == zlib.crc32(raw[:60])
    for i, (_, a) in enumerate(ts):
        e = raw[4096 + 112 * i: 4096 + 112 * (i + 1)]
        assert int.from_bytes(e[104:108], "little") == zlib.crc32(np.ascontiguousarray(a).tobytes())
