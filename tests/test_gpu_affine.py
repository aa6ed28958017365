"""GPU parity of the affine comparison codec (gmlx page, "The two schemes":
per-token groups of 64 values, N-bit codes with an fp16 scale and offset per
group) on the library's paged skeleton, through the C ABI: the pages the GPU
encoder writes against the oracle's quantisation of the same inputs (codes,
scales and offsets bit for bit), and the GPU decode against the oracle's
decode of the same pages."""
import numpy as np
import pytest
import torch

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import workloads as W
from oracle import affine
from tests import parity

pytestmark = pytest.mark.gpu

BITS = [2, 3, 4, 6, 8]


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_kv_cache_kvarn_gb300 import build
    build.build()
    kv.lib()


def _case(dtype="fp16", B=3, Hkv=2, Hq=16, L=700, min_L=None):
    wname = "dense32b" if dtype == "fp16" else "hybrid"
    over = dict(num_seqs=B, num_q_heads=Hq, num_kv_heads=Hkv, context=L, head_dim=128, tile_tokens=128)
    if min_L is not None:
        wname = "g64"
        over.update(min_context=min_L)
    wl = W.WORKLOADS[wname].with_(**over)
    return wl, W.make_dense(wl, device="cpu")


def _gpu_encode(wl, case, bits, dev="cuda"):
    lay = kv.affine_layout(wl.num_kv_heads, case.num_pages, bits, kv.BF16 if wl.dtype == "bf16" else kv.FP16)
    cache = kv.alloc_affine_cache(lay, dev)
    err = kv.new_error_word(dev)
    bt = case.block_table.to(dev)
    for b in range(wl.num_seqs):
        tiles = int(case.seq_lens[b]) // 128
        if tiles:
            kv.affine_encode_tiles(case.k[b:b + 1].to(dev), case.v[b:b + 1].to(dev), lay,
                                   torch.zeros(1, dtype=torch.int32, device=dev), bt[b:b + 1], cache, err,
                                   chunk_tokens=tiles * 128)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    return lay, cache


@pytest.mark.parametrize("bits", BITS)
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_affine_encode_matches_oracle(bits, dtype):
    wl, case = _case(dtype, L=520)
    lay, cache = _gpu_encode(wl, case, bits)
    olay = affine.AffineLayout(128, bits, bits)
    assert kv.affine_page_bytes(lay) == olay.page_bytes
    g = cache.cpu().numpy()
    k, v = parity.f64(case.k), parity.f64(case.v)
    n = 0
    for b in range(wl.num_seqs):
        for h in range(wl.num_kv_heads):
            for t in range(int(case.seq_lens[b]) // 128):
                pages = [int(x) for x in case.block_table[b, 8 * t:8 * t + 8]]
                gk, gv = affine.read_tokens(g, olay, pages, h)
                for got, x in ((gk, k[b, h, 128 * t:128 * t + 128]), (gv, v[b, h, 128 * t:128 * t + 128])):
                    ref = affine.quantize(x, bits)
                    for a, r in zip(got, ref):
                        np.testing.assert_array_equal(a, r)
                    n += 1
    assert n > 0


@pytest.mark.parametrize("bits", BITS)
def test_affine_decode_on_oracle_pages_matches_oracle(bits):
    wl, case = _case(min_L=1)
    k, v = parity.f64(case.k), parity.f64(case.v)
    bt, lens = case.block_table.numpy(), case.seq_lens.numpy()
    olay = affine.AffineLayout(128, bits, bits)
    ocache = np.zeros((case.num_pages, wl.num_kv_heads, olay.page_bytes), np.uint8)
    for b in range(wl.num_seqs):
        C = (int(lens[b]) // 128) * 128
        if C:
            affine.encode_into_cache(ocache, olay, k[b:b + 1, :, :C], v[b:b + 1, :, :C], bt[b:b + 1], 128)
    tk, tv = parity.tails(k, lens, 128), parity.tails(v, lens, 128)
    sm = W.default_sm_scale(wl)
    ref, ref_lse = affine.decode(parity.f64(case.q), ocache, olay, bt, lens, sm, 128, tk, tv)
    dev = "cuda"
    lay = kv.affine_layout(wl.num_kv_heads, case.num_pages, bits)
    Lmax = int(lens.max())
    out = torch.empty((wl.num_seqs, wl.num_q_heads, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((wl.num_seqs, wl.num_q_heads), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.affine_decode_workspace_bytes(lay, wl.num_seqs, wl.num_q_heads, Lmax), dtype=torch.uint8,
                     device=dev)
    err = kv.new_error_word(dev)
    kv.affine_decode(case.q.to(dev), lay, torch.from_numpy(ocache).to(dev), case.block_table.to(dev),
                     case.seq_lens.to(dev), Lmax, out, ws, err, sm, torch.from_numpy(tk).half().to(dev),
                     torch.from_numpy(tv).half().to(dev), lse=lse)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    diff = np.abs(parity.f64(out) - ref).max()
    parity.report(f"affine {bits}-bit decode on oracle pages: lens {lens.tolist()}, max |out - oracle| = {diff:.3e}")
    assert diff <= parity.OUT_ATOL
    np.testing.assert_allclose(parity.f64(lse), ref_lse, atol=1e-4, rtol=0)


@pytest.mark.parametrize("bits,dtype", [(4, "fp16"), (8, "fp16"), (4, "bf16")])
def test_affine_end_to_end(bits, dtype):
    """GPU encode then GPU decode against the oracle's encode and decode."""
    wl, case = _case(dtype, B=2, L=900)
    lay, cache = _gpu_encode(wl, case, bits)
    k, v = parity.f64(case.k), parity.f64(case.v)
    bt, lens = case.block_table.numpy(), case.seq_lens.numpy()
    olay = affine.AffineLayout(128, bits, bits)
    ocache = np.zeros((case.num_pages, wl.num_kv_heads, olay.page_bytes), np.uint8)
    for b in range(wl.num_seqs):
        C = (int(lens[b]) // 128) * 128
        affine.encode_into_cache(ocache, olay, k[b:b + 1, :, :C], v[b:b + 1, :, :C], bt[b:b + 1], 128)
    dt = W.TORCH_DTYPE[wl.dtype]
    tk, tv = parity.tails(k, lens, 128), parity.tails(v, lens, 128)
    sm = W.default_sm_scale(wl)
    ref, _ = affine.decode(parity.f64(case.q), ocache, olay, bt, lens, sm, 128, tk, tv)
    dev = "cuda"
    out = torch.empty((wl.num_seqs, wl.num_q_heads, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.affine_decode_workspace_bytes(lay, wl.num_seqs, wl.num_q_heads, int(lens.max())),
                     dtype=torch.uint8, device=dev)
    err = kv.new_error_word(dev)
    kv.affine_decode(case.q.to(dev), lay, cache, case.block_table.to(dev), case.seq_lens.to(dev), int(lens.max()),
                     out, ws, err, sm, torch.from_numpy(tk).to(dt).to(dev), torch.from_numpy(tv).to(dt).to(dev))
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    diff = np.abs(parity.f64(out) - ref).max()
    parity.report(f"affine {bits}-bit {dtype} end to end: max |out - oracle| = {diff:.3e}")
    assert diff <= parity.OUT_ATOL
