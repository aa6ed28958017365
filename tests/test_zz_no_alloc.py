"""kvarn_decode_noalloc, the decode entry point for callers that can not
allocate device memory (its split-K scratch is a static device array inside
the library), gives the same output as kvarn_decode with a caller workspace,
on two calls in a row with different queries, and both agree with the
oracle's decode of the same pages. Called through the C ABI.

This file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import workloads as W
from oracle import attention, layout
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def built():
    from quantized_kv_cache_kvarn_gb300 import build
    build.build()
    return kv.lib()


def test_noalloc_matches_workspace_decode_twice(built):
    dev = "cuda"
    wl = W.WORKLOADS["dense32b"].with_(num_seqs=3, num_q_heads=16, num_kv_heads=2, context=1300)
    case = W.make_dense(wl, device="cpu")
    lens = torch.tensor([1300, 640, 77], dtype=torch.int32)
    lay = kv.dense_layout(128, 128, 2, case.num_pages)
    cache = kv.alloc_cache(lay, dev)
    err = kv.new_error_word(dev)
    bt = case.block_table.to(dev)
    for b in range(3):
        tiles = int(lens[b]) // 128
        if tiles:
            kv.encode_tiles(case.k[b:b + 1].to(dev), case.v[b:b + 1].to(dev), lay,
                            torch.zeros(1, dtype=torch.int32, device=dev), bt[b:b + 1], cache, err,
                            chunk_tokens=tiles * 128)
    tk = torch.from_numpy(parity.tails(case.k.float().numpy(), lens.numpy(), 128)).half().to(dev)
    tv = torch.from_numpy(parity.tails(case.v.float().numpy(), lens.numpy(), 128)).half().to(dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, 3, 16, 1300), dtype=torch.uint8, device=dev)
    P = ctypes.c_void_p
    for call in range(2):
        q = (case.q if call == 0 else -0.5 * case.q).contiguous().to(dev)
        ref = torch.empty((3, 16, 128), dtype=torch.float32, device=dev)
        ref_lse = torch.empty((3, 16), dtype=torch.float32, device=dev)
        kv.decode(q, lay, cache, bt, lens.to(dev), 1300, ref, ws, err, 0.088, tk, tv, lse=ref_lse)
        out = torch.full((3, 16, 128), float("nan"), dtype=torch.float32, device=dev)
        lse = torch.full((3, 16), float("nan"), dtype=torch.float32, device=dev)
        st = built.kvarn_decode_noalloc(P(q.data_ptr()), 16, ctypes.c_float(0.088), P(cache.data_ptr()),
                                        ctypes.byref(lay), P(bt.data_ptr()), bt.stride(0),
                                        P(lens.to(dev).data_ptr()), 1300, P(tk.data_ptr()), P(tv.data_ptr()),
                                        3, P(out.data_ptr()), P(lse.data_ptr()), P(err.data_ptr()),
                                        P(torch.cuda.current_stream().cuda_stream))
        torch.cuda.synchronize()
        assert st == 0
        assert kv.read_error_flags(err) == 0
        assert np.abs(parity.f64(out) - parity.f64(ref)).max() <= parity.OUT_ATOL
        assert np.abs(parity.f64(lse) - parity.f64(ref_lse)).max() <= 1e-4
        # the oracle's decode of the same (GPU-written) pages and tails
        oref, olse = attention.decode(parity.f64(q), cache.cpu().numpy(), layout.DenseLayout(128, 128),
                                      case.block_table.numpy(), lens.numpy(), 0.088, parity.f64(tk), parity.f64(tv))
        assert np.abs(parity.f64(out) - oref).max() <= parity.OUT_ATOL
        assert np.abs(parity.f64(lse) - olse).max() <= 1e-4


def test_noalloc_rejects_beyond_its_scratch(built):
    """A batch whose partials exceed the static array is refused on the host
    with KVARN_EWORKSPACE, before any launch."""
    lay = kv.dense_layout(128, 128, 8, 1 << 20)
    need = kv.decode_workspace_bytes(lay, 4096, 64, 16384)
    assert need > kv.NOALLOC_SCRATCH_BYTES
    P = ctypes.c_void_p
    a = P(1 << 20)
    st = built.kvarn_decode_noalloc(a, 64, ctypes.c_float(0.1), a, ctypes.byref(lay), a, 1024, a, 16384,
                                    None, None, 4096, a, None, a, None)
    assert st == -5
