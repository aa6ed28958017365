"""GB300 (sm_103a) KVarN KV-cache codec and compressed-cache decode attention.

A thin ctypes binding over libkvarn.so (C ABI in include/kvarn.h): argument
marshalling only, every step of the codec and the attention runs in the
library's CUDA kernels. PyTorch provides device memory and streams. The
library is built in-tree by ``quantized_kv_cache_kvarn_gb300.build`` and
loading fails loudly when it is missing; there is no CPU path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libkvarn.so")

FP16, BF16 = 0, 1
DEVERR_PAGE_RANGE, DEVERR_NO_TAIL, DEVERR_TIMEOUT, DEVERR_SEQ_LEN = 0x1, 0x2, 0x4, 0x8


class KvarnError(RuntimeError):
    pass


class Layout(ctypes.Structure):
    """Mirror of kvarn_layout."""
    _fields_ = [("head_dim", ctypes.c_int32), ("tile_tokens", ctypes.c_int32),
                ("page_tokens", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("k_bits", ctypes.c_int32), ("v_bits", ctypes.c_int32),
                ("norm_iters", ctypes.c_int32), ("rope_dim", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("scale_dtype", ctypes.c_int32),
                ("num_pages", ctypes.c_int64)]


def dense_layout(head_dim, tile_tokens, num_kv_heads, num_pages, kv_dtype=FP16, norm_iters=2,
                 k_bits=4, v_bits=2, fp16_scales=False) -> Layout:
    return Layout(head_dim, tile_tokens, 16, num_kv_heads, k_bits, v_bits, norm_iters, 0,
                  kv_dtype, 1 if fp16_scales else 0, num_pages)


def latent_layout(num_pages, kv_dtype=BF16, norm_iters=2) -> Layout:
    return Layout(512, 128, 16, 1, 4, 0, norm_iters, 64, kv_dtype, 0, num_pages)


_lib = None
_P = ctypes.c_void_p
_I32, _I64, _F32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
_LP = ctypes.POINTER(Layout)

_SIGS = {
    "kvarn_version": ([], _I32),
    "kvarn_status_string": ([_I32], ctypes.c_char_p),
    "kvarn_layout_check": ([_LP], _I32),
    "kvarn_page_bytes": ([_LP], _I64),
    "kvarn_encode_tiles": ([_P, _P, _I64, _I64, _I32, _I32, _P, _P, _I32, _LP, _P, _P, _P], _I32),
    "kvarn_encode_stage_floats": ([_LP, _I32, _I32], _I64),
    "kvarn_encode_tiles_staged": ([_P, _P, _I64, _I64, _I32, _I32, _P, _P, _I32, _LP, _P, _P, _P, _P], _I32),
    "kvarn_append": ([_P, _P, _P, _I32, _P, _P, _I32, _P, _I32, _LP, _P, _P, _P], _I32),
    "kvarn_decode_workspace_bytes": ([_LP, _I32, _I32, _I32], _I64),
    "kvarn_decode": ([_P, _I32, _F32, _P, _LP, _P, _I32, _P, _I32, _P, _P, _I32, _P, _P, _P, _I64,
                      _P, _P], _I32),
    "kvarn_decode_verify_workspace_bytes": ([_LP, _I32, _I32, _I32, _I32], _I64),
    "kvarn_decode_verify": ([_P, _I32, _I32, _F32, _P, _LP, _P, _I32, _P, _I32, _P, _P, _I32, _I32, _P, _P,
                             _P, _I64, _P, _P], _I32),
    "kvarn_decode_window_workspace_bytes": ([_LP, _I32, _I32, _I32, _I32, _I32, _I32], _I64),
    "kvarn_decode_window": ([_P, _I32, _I32, _F32, _P, _LP, _P, _I32, _P, _I32, _I32, _P, _P, _I32, _P, _P,
                             _I32, _I32, _P, _P, _P, _I64, _P, _P], _I32),
    "kvarn_fp16_page_bytes": ([_LP], _I64),
    "kvarn_store_fp16": ([_P, _P, _I64, _I64, _I32, _I32, _I32, _P, _I32, _LP, _P, _P, _P], _I32),
    "kvarn_decode_fp16": ([_P, _I32, _F32, _P, _LP, _P, _I32, _P, _I32, _I32, _P, _P, _P, _I64, _P,
                           _P], _I32),
    "kvarn_encode_latent": ([_P, _I64, _P, _I64, _I32, _I32, _P, _P, _I32, _LP, _P, _P, _P], _I32),
    "kvarn_decode_mla": ([_P, _P, _I32, _F32, _P, _LP, _P, _I32, _P, _I32, _P, _P, _I32, _P, _P, _P,
                          _I64, _P, _P], _I32),
    "kvarn_read_error_flags": ([_P, _P, _P], _I32),
    "kvarn_set_copy_wait_test": ([_I64, _I32], _I32),
    "kvarn_affine_page_bytes": ([_LP], _I64),
    "kvarn_affine_encode_tiles": ([_P, _P, _I64, _I64, _I32, _I32, _P, _P, _I32, _LP, _P, _P, _P], _I32),
    "kvarn_affine_decode_workspace_bytes": ([_LP, _I32, _I32, _I32], _I64),
    "kvarn_affine_decode": ([_P, _I32, _F32, _P, _LP, _P, _I32, _P, _I32, _P, _P, _I32, _P, _P, _P, _I64,
                             _P, _P], _I32),
    "kvarn_decode_noalloc": ([_P, _I32, _F32, _P, _LP, _P, _I32, _P, _I32, _P, _P, _I32, _P, _P, _P, _P],
                             _I32),
}

NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024

EXPORTED = tuple(_SIGS)


def lib() -> ctypes.CDLL:
    """Load libkvarn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise KvarnError(f"libkvarn.so is not built ({LIB_PATH}); run "
                             "python -m quantized_kv_cache_kvarn_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != 0:
        raise KvarnError(f"{what}: {lib().kvarn_status_string(status).decode()} ({status})")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise KvarnError("tensor must live on the GPU")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def page_bytes(layout: Layout) -> int:
    n = lib().kvarn_page_bytes(ctypes.byref(layout))
    if n < 0:
        raise KvarnError("invalid layout")
    return n


def fp16_page_bytes(layout: Layout) -> int:
    n = lib().kvarn_fp16_page_bytes(ctypes.byref(layout))
    if n < 0:
        raise KvarnError("invalid layout")
    return n


def decode_workspace_bytes(layout: Layout, num_seqs: int, num_q_heads: int, max_seq_len: int) -> int:
    n = lib().kvarn_decode_workspace_bytes(ctypes.byref(layout), num_seqs, num_q_heads, max_seq_len)
    if n < 0:
        raise KvarnError("invalid decode arguments")
    return n


def new_error_word(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def read_error_flags(err: torch.Tensor, stream=None) -> int:
    out = ctypes.c_uint32(0)
    _check(lib().kvarn_read_error_flags(_ptr(err), ctypes.byref(out), _stream(stream)), "read_error_flags")
    return out.value


def alloc_cache(layout: Layout, device=None) -> torch.Tensor:
    """Zeroed cache bytes: [num_pages, Hkv, page_bytes] (dense) or
    [num_pages, page_bytes] (latent)."""
    pb = page_bytes(layout)
    if layout.rope_dim:
        return torch.zeros((layout.num_pages, pb), dtype=torch.uint8, device=device or "cuda")
    return torch.zeros((layout.num_pages, layout.num_kv_heads, pb), dtype=torch.uint8,
                       device=device or "cuda")


def encode_tiles(k, v, layout: Layout, tile_start, block_table, cache, err, chunk_tokens=None,
                 stream=None):
    """k, v: [B, Hkv, C, D] (any seq/head strides, contiguous rows)."""
    B = k.shape[0]
    C = k.shape[2] if chunk_tokens is None else chunk_tokens
    assert k.stride() == v.stride() and k.stride(3) == 1 and k.stride(2) == k.shape[3]
    _check(lib().kvarn_encode_tiles(_ptr(k), _ptr(v), k.stride(0), k.stride(1), B, C, _ptr(tile_start),
                                    _ptr(block_table), block_table.stride(0), ctypes.byref(layout),
                                    _ptr(cache), _ptr(err), _stream(stream)), "encode_tiles")


def encode_stage_floats(layout: Layout, num_seqs: int, chunk_tokens: int) -> int:
    n = lib().kvarn_encode_stage_floats(ctypes.byref(layout), num_seqs, chunk_tokens)
    if n < 0:
        raise KvarnError("invalid arguments for kvarn_encode_stage_floats")
    return n


def encode_tiles_staged(k, v, layout: Layout, tile_start, block_table, cache, stages, err, chunk_tokens=None,
                        stream=None):
    """encode_tiles that also fills `stages` (fp32, encode_stage_floats(...)
    floats) with the fp32 intermediates of every encoded tile."""
    B = k.shape[0]
    C = k.shape[2] if chunk_tokens is None else chunk_tokens
    assert k.stride() == v.stride() and k.stride(3) == 1 and k.stride(2) == k.shape[3]
    assert stages.dtype == torch.float32 and stages.numel() >= encode_stage_floats(layout, B, C)
    _check(lib().kvarn_encode_tiles_staged(_ptr(k), _ptr(v), k.stride(0), k.stride(1), B, C, _ptr(tile_start),
                                           _ptr(block_table), block_table.stride(0), ctypes.byref(layout),
                                           _ptr(cache), _ptr(stages), _ptr(err), _stream(stream)),
           "encode_tiles_staged")


def append(k, v, seq_lens, max_seq_len, tail_k, tail_v, block_table, layout: Layout, cache, err, stream=None):
    """k, v: [B, Hkv, D] newest tokens; tail_k/v: [B, Hkv, N, D]."""
    assert k.is_contiguous() and v.is_contiguous() and tail_k.is_contiguous() and tail_v.is_contiguous()
    _check(lib().kvarn_append(_ptr(k), _ptr(v), _ptr(seq_lens), max_seq_len, _ptr(tail_k), _ptr(tail_v),
                              k.shape[0], _ptr(block_table), block_table.stride(0), ctypes.byref(layout),
                              _ptr(cache), _ptr(err), _stream(stream)), "append")


def decode(q, layout: Layout, cache, block_table, seq_lens, max_seq_len, out, workspace, err,
           sm_scale, tail_k=None, tail_v=None, lse=None, stream=None):
    B, Hq, _ = q.shape
    _check(lib().kvarn_decode(_ptr(q), Hq, sm_scale, _ptr(cache), ctypes.byref(layout),
                              _ptr(block_table), block_table.stride(0), _ptr(seq_lens), max_seq_len,
                              _ptr(tail_k), _ptr(tail_v), B, _ptr(out), _ptr(lse), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _ptr(err),
                              _stream(stream)), "decode")


def decode_verify_workspace_bytes(layout: Layout, num_seqs: int, num_q_heads: int, num_queries: int,
                                  max_seq_len: int) -> int:
    n = lib().kvarn_decode_verify_workspace_bytes(ctypes.byref(layout), num_seqs, num_q_heads, num_queries,
                                                  max_seq_len)
    if n < 0:
        raise ValueError("invalid arguments for kvarn_decode_verify_workspace_bytes")
    return n


def decode_verify(q, layout: Layout, cache, block_table, seq_lens, max_seq_len, out, workspace, err,
                  sm_scale, tail_k=None, tail_v=None, lse=None, stream=None):
    """q: [B, Q, Hq, D]; tail_k/v: [B, Hkv, capacity, D]; out: [B, Q, Hq, D]."""
    B, Q, Hq, _ = q.shape
    cap = tail_k.shape[2] if tail_k is not None else layout.tile_tokens + Q - 2
    _check(lib().kvarn_decode_verify(_ptr(q), Hq, Q, sm_scale, _ptr(cache), ctypes.byref(layout),
                                     _ptr(block_table), block_table.stride(0), _ptr(seq_lens), max_seq_len,
                                     _ptr(tail_k), _ptr(tail_v), max(cap, 1), B, _ptr(out), _ptr(lse),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(err),
                                     _stream(stream)), "decode_verify")


def decode_window_workspace_bytes(layout: Layout, num_seqs: int, num_q_heads: int, num_queries: int,
                                  max_seq_len: int, sink_tokens: int, recent_tokens: int) -> int:
    n = lib().kvarn_decode_window_workspace_bytes(ctypes.byref(layout), num_seqs, num_q_heads, num_queries,
                                                  max_seq_len, sink_tokens, recent_tokens)
    if n < 0:
        raise ValueError("invalid arguments for kvarn_decode_window_workspace_bytes")
    return n


def decode_window(q, layout: Layout, cache, block_table, seq_lens, max_seq_len, out, workspace, err,
                  sm_scale, sink_k=None, sink_v=None, recent_tokens=0, tail_k=None, tail_v=None, lse=None,
                  stream=None):
    """q: [B, Q, Hq, D]; sink_k/v: [B, Hkv, S, D] (S a multiple of N) or None;
    tail_k/v: [B, Hkv, capacity, D]; out: [B, Q, Hq, D]."""
    B, Q, Hq, _ = q.shape
    S = sink_k.shape[2] if sink_k is not None else 0
    cap = tail_k.shape[2] if tail_k is not None else recent_tokens + layout.tile_tokens + Q - 2
    _check(lib().kvarn_decode_window(_ptr(q), Hq, Q, sm_scale, _ptr(cache), ctypes.byref(layout),
                                     _ptr(block_table), block_table.stride(0), _ptr(seq_lens), max_seq_len, S,
                                     _ptr(sink_k), _ptr(sink_v), recent_tokens, _ptr(tail_k), _ptr(tail_v),
                                     max(cap, 1), B, _ptr(out), _ptr(lse), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _ptr(err), _stream(stream)),
           "decode_window")


def alloc_fp16_cache(layout: Layout, device=None) -> torch.Tensor:
    return torch.zeros((layout.num_pages, layout.num_kv_heads, fp16_page_bytes(layout)),
                       dtype=torch.uint8, device=device or "cuda")


def store_fp16(k, v, layout: Layout, token0, count, block_table, cache, err, stream=None):
    B = k.shape[0]
    _check(lib().kvarn_store_fp16(_ptr(k), _ptr(v), k.stride(0), k.stride(1), B, token0, count,
                                  _ptr(block_table), block_table.stride(0), ctypes.byref(layout),
                                  _ptr(cache), _ptr(err), _stream(stream)), "store_fp16")


def decode_fp16(q, layout: Layout, cache, block_table, seq_lens, max_seq_len, out, workspace, err,
                sm_scale, lse=None, stream=None):
    B, Hq, _ = q.shape
    _check(lib().kvarn_decode_fp16(_ptr(q), Hq, sm_scale, _ptr(cache), ctypes.byref(layout),
                                   _ptr(block_table), block_table.stride(0), _ptr(seq_lens),
                                   max_seq_len, B, _ptr(out), _ptr(lse), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _ptr(err),
                                   _stream(stream)), "decode_fp16")


def encode_latent(latent, rope, layout: Layout, tile_start, block_table, cache, err,
                  chunk_tokens=None, stream=None):
    """latent [B, C, 512], rope [B, C, 64] fp16 (contiguous rows)."""
    B = latent.shape[0]
    C = latent.shape[1] if chunk_tokens is None else chunk_tokens
    _check(lib().kvarn_encode_latent(_ptr(latent), latent.stride(0), _ptr(rope), rope.stride(0), B, C,
                                     _ptr(tile_start), _ptr(block_table), block_table.stride(0),
                                     ctypes.byref(layout), _ptr(cache), _ptr(err), _stream(stream)),
           "encode_latent")


def decode_mla(q_latent, q_rope, layout: Layout, cache, block_table, seq_lens, max_seq_len, out,
               workspace, err, sm_scale, tail_latent=None, tail_rope=None, lse=None, stream=None):
    B, H, _ = q_latent.shape
    _check(lib().kvarn_decode_mla(_ptr(q_latent), _ptr(q_rope), H, sm_scale, _ptr(cache),
                                  ctypes.byref(layout), _ptr(block_table), block_table.stride(0),
                                  _ptr(seq_lens), max_seq_len, _ptr(tail_latent), _ptr(tail_rope), B,
                                  _ptr(out), _ptr(lse), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _ptr(err),
                                  _stream(stream)), "decode_mla")


def decode_noalloc(q, layout: Layout, cache, block_table, seq_lens, max_seq_len, out, err, sm_scale,
                   tail_k=None, tail_v=None, lse=None, stream=None):
    """kvarn_decode with the split-K scratch in the library's own static
    device array (NOALLOC_SCRATCH_BYTES per device) instead of a caller
    workspace; for callers that can not allocate device memory. Calls that
    overlap on the GPU share that array and race."""
    B, Hq, _ = q.shape
    _check(lib().kvarn_decode_noalloc(_ptr(q), Hq, sm_scale, _ptr(cache), ctypes.byref(layout),
                                      _ptr(block_table), block_table.stride(0), _ptr(seq_lens),
                                      max_seq_len, _ptr(tail_k), _ptr(tail_v), B, _ptr(out), _ptr(lse),
                                      _ptr(err), _stream(stream)), "decode_noalloc")


# ------------------------------------------------------------------ affine
# The affine comparison codec (per-token groups of 64 channels with an fp16
# scale and offset each, no rotation) on the same paged decode skeleton.

def affine_layout(num_kv_heads, num_pages, bits, kv_dtype=FP16) -> Layout:
    """head_dim 128, 128-token tiles, keys and values at `bits` (2, 3, 4, 6, 8)."""
    return Layout(128, 128, 16, num_kv_heads, bits, bits, 1, 0, kv_dtype, 1, num_pages)


def affine_page_bytes(layout: Layout) -> int:
    n = lib().kvarn_affine_page_bytes(ctypes.byref(layout))
    if n < 0:
        raise KvarnError("invalid affine layout")
    return n


def alloc_affine_cache(layout: Layout, device=None) -> torch.Tensor:
    return torch.zeros((layout.num_pages, layout.num_kv_heads, affine_page_bytes(layout)), dtype=torch.uint8,
                       device=device or "cuda")


def affine_encode_tiles(k, v, layout: Layout, tile_start, block_table, cache, err, chunk_tokens=None,
                        stream=None):
    """k, v: [B, Hkv, C, D] (any seq/head strides, contiguous rows)."""
    B = k.shape[0]
    C = k.shape[2] if chunk_tokens is None else chunk_tokens
    assert k.stride() == v.stride() and k.stride(3) == 1 and k.stride(2) == k.shape[3]
    _check(lib().kvarn_affine_encode_tiles(_ptr(k), _ptr(v), k.stride(0), k.stride(1), B, C, _ptr(tile_start),
                                           _ptr(block_table), block_table.stride(0), ctypes.byref(layout),
                                           _ptr(cache), _ptr(err), _stream(stream)), "affine_encode_tiles")


def affine_decode_workspace_bytes(layout: Layout, num_seqs: int, num_q_heads: int, max_seq_len: int) -> int:
    n = lib().kvarn_affine_decode_workspace_bytes(ctypes.byref(layout), num_seqs, num_q_heads, max_seq_len)
    if n < 0:
        raise KvarnError("invalid affine decode arguments")
    return n


def affine_decode(q, layout: Layout, cache, block_table, seq_lens, max_seq_len, out, workspace, err,
                  sm_scale, tail_k=None, tail_v=None, lse=None, stream=None):
    B, Hq, _ = q.shape
    _check(lib().kvarn_affine_decode(_ptr(q), Hq, sm_scale, _ptr(cache), ctypes.byref(layout),
                                     _ptr(block_table), block_table.stride(0), _ptr(seq_lens), max_seq_len,
                                     _ptr(tail_k), _ptr(tail_v), B, _ptr(out), _ptr(lse), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _ptr(err),
                                     _stream(stream)), "affine_decode")


def set_copy_wait_test(cycles: int, withhold: bool = False) -> None:
    """Diagnostic: clock cycles the dense decode kernels wait for a page copy
    before they flag DEVERR_TIMEOUT and return (0: the default), and whether
    every copy is announced larger than it is so that every wait runs out."""
    _check(lib().kvarn_set_copy_wait_test(cycles, 1 if withhold else 0), "set_copy_wait_test")
