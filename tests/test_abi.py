"""The C-ABI library loads on a CPU-only machine, exports every function
include/kvarn.h declares, and rejects bad arguments on the host before any
launch. No compute call is made here."""
import ctypes
import os
import re

import pytest

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import build as kvbuild

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kvarn.h")


@pytest.fixture(scope="module")
def L():
    kvbuild.build()
    return kv.lib()


def declared():
    text = open(HDR).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(kvarn_\w+)\s*\(", text, re.M)))


def test_header_declares_the_calls():
    names = declared()
    for must in ("kvarn_encode_tiles", "kvarn_decode", "kvarn_decode_fp16", "kvarn_encode_latent",
                 "kvarn_decode_mla", "kvarn_page_bytes", "kvarn_decode_workspace_bytes"):
        assert must in names


def test_every_declared_symbol_is_exported(L):
    for name in declared():
        assert hasattr(L, name), name
    assert set(declared()) == set(kv.EXPORTED)


def test_page_bytes(L):
    assert kv.page_bytes(kv.dense_layout(128, 128, 8, 10)) == 1920
    assert kv.page_bytes(kv.dense_layout(128, 64, 8, 10)) == 2048
    assert kv.page_bytes(kv.dense_layout(256, 128, 4, 10)) == 3584
    assert kv.page_bytes(kv.latent_layout(10)) == 6528
    assert kv.fp16_page_bytes(kv.dense_layout(128, 128, 8, 10)) == 8192


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 64, -2), ("head_dim", 96, -2), ("tile_tokens", 32, -2), ("k_bits", 7, -2),
    ("v_bits", 1, -2), ("norm_iters", 0, -2), ("norm_iters", 9, -2), ("page_tokens", 32, -2),
    ("kv_dtype", 2, -2), ("num_kv_heads", 0, -1)])
def test_layout_rejections(L, field, value, code):
    lay = kv.dense_layout(128, 128, 8, 10)
    setattr(lay, field, value)
    assert L.kvarn_layout_check(ctypes.byref(lay)) == code
    assert L.kvarn_page_bytes(ctypes.byref(lay)) == -1


@pytest.mark.parametrize("kb", [2, 3, 4, 5, 6, 8])
@pytest.mark.parametrize("vb", [2, 3, 4, 5, 6, 8])
def test_width_pairs_with_fp16_scales(L, kb, vb):
    """Keys and values take their widths separately (gmlx page, "The two
    schemes"): every pair is accepted at head_dim 128 with fp16 or fp32
    scales and at head_dim 256 with fp16 scales (fp32 there only for k4v2),
    and the page is the K part then the V part at their own widths."""
    from oracle import layout
    for sb in (2, 4):
        lay = kv.dense_layout(128, 128, 8, 10, k_bits=kb, v_bits=vb, fp16_scales=sb == 2)
        assert L.kvarn_layout_check(ctypes.byref(lay)) == 0
        assert kv.page_bytes(lay) == layout.DenseLayout(128, 128, kb, vb, sb).page_bytes
    wide = kv.dense_layout(256, 128, 4, 10, k_bits=kb, v_bits=vb, fp16_scales=True)
    assert L.kvarn_layout_check(ctypes.byref(wide)) == 0
    assert kv.page_bytes(wide) == layout.DenseLayout(256, 128, kb, vb, 2).page_bytes
    wide32 = kv.dense_layout(256, 128, 4, 10, k_bits=kb, v_bits=vb, fp16_scales=False)
    assert L.kvarn_layout_check(ctypes.byref(wide32)) == (0 if (kb, vb) == (4, 2) else -2)


@pytest.mark.parametrize("kb,vb", [(7, 4), (4, 7), (1, 2), (6, 0)])
def test_width_pairs_rejected(L, kb, vb):
    lay = kv.dense_layout(128, 128, 8, 10, k_bits=kb, v_bits=vb, fp16_scales=True)
    assert L.kvarn_layout_check(ctypes.byref(lay)) == -2


def test_host_validation_before_launch(L):
    lay = kv.dense_layout(128, 128, 8, 10)
    P = ctypes.c_void_p
    a16 = P(1 << 20)          # aligned fake device address, never dereferenced
    bad = P((1 << 20) + 4)    # misaligned
    # encode: chunk not a multiple of the tile
    assert L.kvarn_encode_tiles(a16, a16, 0, 0, 1, 100, a16, a16, 8, ctypes.byref(lay), a16, a16, None) == -1
    # encode: null pointer
    assert L.kvarn_encode_tiles(None, a16, 0, 0, 1, 128, a16, a16, 8, ctypes.byref(lay), a16, a16, None) == -1
    # encode: misaligned k
    assert L.kvarn_encode_tiles(bad, a16, 0, 0, 1, 128, a16, a16, 8, ctypes.byref(lay), a16, a16, None) == -3
    # encode: nothing to do is ok and launches nothing
    assert L.kvarn_encode_tiles(None, None, 0, 0, 0, 0, None, None, 0, ctypes.byref(lay), None, None, None) == 0
    # decode: GQA group above 8
    ws = 1 << 30
    assert L.kvarn_decode(a16, 72, 0.1, a16, ctypes.byref(lay), a16, 1024, a16, 16384, None, None, 1, a16,
                          None, a16, ws, a16, None) == -2
    # decode: heads not a multiple of the KV heads
    assert L.kvarn_decode(a16, 12, 0.1, a16, ctypes.byref(lay), a16, 1024, a16, 16384, None, None, 1, a16,
                          None, a16, ws, a16, None) == -1
    # decode: block table narrower than the committed pages
    assert L.kvarn_decode(a16, 64, 0.1, a16, ctypes.byref(lay), a16, 10, a16, 16384, None, None, 1, a16,
                          None, a16, ws, a16, None) == -1
    # decode: workspace too small
    assert L.kvarn_decode(a16, 64, 0.1, a16, ctypes.byref(lay), a16, 1024, a16, 16384, None, None, 1, a16,
                          None, a16, 16, a16, None) == -5
    # decode: misaligned q
    assert L.kvarn_decode(bad, 64, 0.1, a16, ctypes.byref(lay), a16, 1024, a16, 16384, None, None, 1, a16,
                          None, a16, ws, a16, None) == -3
    # mla: head count not a multiple of 16
    lat = kv.latent_layout(10)
    assert L.kvarn_decode_mla(a16, a16, 24, 0.1, a16, ctypes.byref(lat), a16, 512, a16, 8192, None, None,
                              1, a16, None, a16, ws, a16, None) == -2


def test_workspace_bytes(L):
    lay = kv.dense_layout(128, 128, 8, 32768)
    n = kv.decode_workspace_bytes(lay, 32, 64, 16384)
    assert n > 0 and n % 16 == 0
    assert kv.decode_workspace_bytes(lay, 32, 64, 0) > 0


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5):
        assert L.kvarn_status_string(code)


def test_copy_wait_test_rejects_bad_arguments(L):
    assert L.kvarn_set_copy_wait_test(-5, 0) == -1
    assert L.kvarn_set_copy_wait_test(0, 2) == -1
    assert L.kvarn_set_copy_wait_test(0, 0) == 0
