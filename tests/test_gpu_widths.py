"""GPU parity of the other code widths (gmlx page, "The two schemes": kvarn
widths 2, 3, 4, 5, 6 and 8, set separately for keys and values), with fp16
and fp32 scales at head_dim 128 and fp16 scales at 256, through the C ABI: the
pages the GPU encoder writes against the oracle's encoding, and the GPU
decode of pages the oracle wrote against the oracle's decode."""
import numpy as np
import pytest
import torch

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import workloads as W
from oracle import attention, layout
from tests import parity

pytestmark = pytest.mark.gpu

BITS = (2, 3, 4, 5, 6, 8)
# every compiled (key width, value width) pair (the gmlx page sets the two
# widths separately, GMLX_KVARN_BITS), the tile size alternating so that each
# size meets every key and every value width: head_dim 128 with fp16 scales
# and with fp32 scales, head_dim 256 with fp16 scales; (k, v, N, D, scale bytes)
WIDTHS = [(kb, vb, 128 if (i + j) % 2 == 0 else 64, 128, 2) for i, kb in enumerate(BITS) for j, vb in enumerate(BITS)]
WIDTHS += [(b, b, 64 if (i % 2 == 0) else 128, 128, 2) for i, b in enumerate(BITS)] + [(4, 2, 64, 128, 2)]
WIDTHS += [(kb, vb, 64 if (i + j) % 2 == 0 else 128, 128, 4) for i, kb in enumerate(BITS) for j, vb in enumerate(BITS)]
WIDTHS += [(kb, vb, 128 if (i + j) % 2 == 0 else 64, 256, 2) for i, kb in enumerate(BITS) for j, vb in enumerate(BITS)]
WIDTHS += [(b, b, 64 if (i % 2 == 0) else 128, 256, 2) for i, b in enumerate(BITS)]
WIDTHS = list(dict.fromkeys(WIDTHS))


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_kv_cache_kvarn_gb300 import build
    build.build()
    kv.lib()


def _case(N, D=128):
    wl = W.WORKLOADS["dense32b"].with_(num_seqs=2, num_q_heads=8, num_kv_heads=2, context=2 * N + 37,
                                       tile_tokens=N, head_dim=D)
    return wl, W.make_dense(wl, device="cpu")


@pytest.mark.parametrize("kb,vb,N,D,sb", WIDTHS)
def test_encode_matches_oracle(kb, vb, N, D, sb):
    wl, case = _case(N, D)
    dev = "cuda"
    lay = kv.dense_layout(D, N, wl.num_kv_heads, case.num_pages, k_bits=kb, v_bits=vb, fp16_scales=sb == 2)
    assert kv.page_bytes(lay) == layout.DenseLayout(D, N, kb, vb, sb).page_bytes
    cache = kv.alloc_cache(lay, dev)
    err = kv.new_error_word(dev)
    T = int(case.seq_lens[0]) // N
    kv.encode_tiles(case.k.to(dev), case.v.to(dev), lay, torch.zeros(wl.num_seqs, dtype=torch.int32, device=dev),
                    case.block_table.to(dev), cache, err, chunk_tokens=T * N)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    st_k, st_v = parity.check_dense_pages(cache.cpu().numpy(), parity.f64(case.k), parity.f64(case.v),
                                          case.block_table.numpy(), case.seq_lens.numpy(), N, D,
                                          kb=kb, vb=vb, sb=sb)
    print(f"\nK{kb}V{vb} N{N} D{D} S{8 * sb}: K codes {st_k['mismatch']}/{st_k['codes']} differ, V {st_v['mismatch']}/"
          f"{st_v['codes']}")


@pytest.mark.parametrize("kb,vb,N,D,sb", WIDTHS)
def test_decode_on_oracle_pages_matches_oracle(kb, vb, N, D, sb):
    wl, case = _case(N, D)
    k, v = parity.f64(case.k), parity.f64(case.v)
    bt, lens = case.block_table.numpy(), case.seq_lens.numpy()
    ocache = parity.oracle_dense_cache(k, v, bt, lens, N, D, case.num_pages, kb=kb, vb=vb, sb=sb)
    tk, tv = parity.tails(k, lens, N), parity.tails(v, lens, N)
    sm = W.default_sm_scale(wl)
    ref, ref_lse = attention.decode(parity.f64(case.q), ocache, layout.DenseLayout(D, N, kb, vb, sb), bt, lens,
                                    sm, tk, tv)
    dev = "cuda"
    lay = kv.dense_layout(D, N, wl.num_kv_heads, case.num_pages, k_bits=kb, v_bits=vb, fp16_scales=sb == 2)
    Lmax = int(lens.max())
    out = torch.empty((wl.num_seqs, wl.num_q_heads, D), dtype=torch.float32, device=dev)
    lse = torch.empty((wl.num_seqs, wl.num_q_heads), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, wl.num_seqs, wl.num_q_heads, Lmax), dtype=torch.uint8,
                     device=dev)
    err = kv.new_error_word(dev)
    kv.decode(case.q.to(dev), lay, torch.from_numpy(ocache).to(dev), case.block_table.to(dev),
              case.seq_lens.to(dev), Lmax, out, ws, err, sm, torch.from_numpy(tk).half().to(dev),
              torch.from_numpy(tv).half().to(dev), lse=lse)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    diff = np.abs(parity.f64(out) - ref).max()
    print(f"\nK{kb}V{vb} N{N} D{D} S{8 * sb}: max |out - oracle| = {diff:.3e}")
    assert diff <= parity.OUT_ATOL
    np.testing.assert_allclose(parity.f64(lse), ref_lse, atol=1e-4, rtol=0)
