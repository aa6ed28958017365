"""GPU parity of the MLA latent codec and decode against the oracle, through
the C ABI, on seeded inputs shaped like the MLA workload (512-wide bf16
latent with 2% outlier channels, 64-wide fp16 rope, 128 query heads in groups
of 16) but small enough for the oracle."""
import numpy as np
import pytest
import torch

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import workloads as W
from oracle import codec, layout, mla
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_kv_cache_kvarn_gb300 import build
    build.build()
    kv.lib()


def _case(num_seqs=2, heads=32, context=424, lens=None):
    wl = W.WORKLOADS["mla"].with_(num_seqs=num_seqs, num_q_heads=heads, context=context)
    case = W.make_latent(wl, device="cpu")
    if lens is not None:
        case.seq_lens = torch.tensor(lens, dtype=torch.int32)
    return wl, case


def _gpu_encode(wl, case, dev="cuda"):
    lay = kv.latent_layout(case.num_pages, kv.BF16, wl.norm_iters)
    cache = kv.alloc_cache(lay, dev)
    err = kv.new_error_word(dev)
    bt = case.block_table.to(dev)
    for b in range(wl.num_seqs):
        tiles = int(case.seq_lens[b]) // 128
        if tiles:
            kv.encode_latent(case.latent[b:b + 1].to(dev), case.rope[b:b + 1].to(dev), lay,
                             torch.zeros(1, dtype=torch.int32, device=dev), bt[b:b + 1], cache, err,
                             chunk_tokens=tiles * 128)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    return lay, cache


def test_encode_latent_matches_oracle():
    wl, case = _case()
    lay, cache = _gpu_encode(wl, case)
    g = cache.cpu().numpy()
    olay = layout.LatentLayout(512, 64, 128)
    lat = parity.f64(case.latent)
    stats = parity.new_stats()
    for b in range(wl.num_seqs):
        for t in range(int(case.seq_lens[b]) // 128):
            pages = [int(case.block_table[b, t * 8 + p]) for p in range(8)]
            enc, rope = mla.read_tile(g, olay, pages)
            ref = codec.encode_tile(lat[b, t * 128:(t + 1) * 128], 4, 2)
            parity.compare_tile(enc, ref, 4, stats)
            np.testing.assert_array_equal(rope, parity.f64(case.rope[b, t * 128:(t + 1) * 128]))
    print(f"\nmla encode: codes {stats['mismatch']}/{stats['codes']} differ (max dist {stats['max_dist']:.2e}); "
          f"scale rel {stats['scale_rel']:.2e}")
    assert stats["scale_rel"] <= parity.SCALE_RTOL
    assert stats["mismatch"] <= max(4, 1e-3 * stats["codes"])


@pytest.mark.parametrize("lens", [None, [128, 300]])
def test_decode_mla_on_oracle_pages(lens):
    wl, case = _case(lens=lens)
    olay = layout.LatentLayout(512, 64, 128)
    lat, rope = parity.f64(case.latent), parity.f64(case.rope)
    bt, sl = case.block_table.numpy(), case.seq_lens.numpy()
    ocache = np.zeros((case.num_pages, olay.page_bytes), np.uint8)
    for b in range(wl.num_seqs):
        tiles = int(sl[b]) // 128
        if tiles:
            mla.encode_into_cache(ocache, olay, lat[b:b + 1, :tiles * 128], rope[b:b + 1, :tiles * 128],
                                  bt[b:b + 1], [0])
    B = wl.num_seqs
    tl = np.zeros((B, 128, 512))
    tr = np.zeros((B, 128, 64))
    for b in range(B):
        c = (int(sl[b]) // 128) * 128
        tl[b, :int(sl[b]) - c] = lat[b, c:int(sl[b])]
        tr[b, :int(sl[b]) - c] = rope[b, c:int(sl[b])]
    sm = W.default_sm_scale(wl)
    ref, ref_lse = mla.decode(parity.f64(case.q_latent), parity.f64(case.q_rope), ocache, olay, bt, sl, sm, tl, tr)

    dev = "cuda"
    lay = kv.latent_layout(case.num_pages, kv.BF16)
    H = wl.num_q_heads
    Lmax = int(sl.max())
    out = torch.empty((B, H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, B, H, Lmax), dtype=torch.uint8, device=dev)
    err = kv.new_error_word(dev)
    kv.decode_mla(case.q_latent.to(dev), case.q_rope.to(dev), lay, torch.from_numpy(ocache).to(dev),
                  case.block_table.to(dev), torch.from_numpy(sl).to(dev), Lmax, out, ws, err, sm,
                  torch.from_numpy(tl).to(torch.bfloat16).to(dev), torch.from_numpy(tr).half().to(dev), lse=lse)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    diff = np.abs(parity.f64(out) - ref).max()
    print(f"\nmla decode lens={list(sl)}: max |out - oracle| = {diff:.3e}, "
          f"max |lse - oracle| = {np.abs(parity.f64(lse) - ref_lse).max():.3e}")
    assert diff <= parity.OUT_ATOL
    np.testing.assert_allclose(parity.f64(lse), ref_lse, atol=1e-4, rtol=0)


def test_decode_mla_fp16_queries_many_splits():
    """fp16 queries and tails, all 128 heads, one 4096 + 60-token sequence: the
    split plan cuts the 32 tiles over several CTA pairs (a short last split),
    whose partials the merge combines with the tail's."""
    wl, case = _case(num_seqs=1, heads=128, context=4156)
    olay = layout.LatentLayout(512, 64, 128)
    lat, rope = parity.f64(case.latent), parity.f64(case.rope)
    bt, sl = case.block_table.numpy(), case.seq_lens.numpy()
    ocache = np.zeros((case.num_pages, olay.page_bytes), np.uint8)
    mla.encode_into_cache(ocache, olay, lat[:, :4096], rope[:, :4096], bt, [0])
    tl = np.zeros((1, 128, 512))
    tr = np.zeros((1, 128, 64))
    tl[0, :60], tr[0, :60] = lat[0, 4096:4156], rope[0, 4096:4156]
    ql = case.q_latent.to(torch.float16)
    qr = case.q_rope.to(torch.float16)
    sm = W.default_sm_scale(wl)
    ref, ref_lse = mla.decode(parity.f64(ql), parity.f64(qr), ocache, olay, bt, sl, sm, tl, tr)

    dev = "cuda"
    lay = kv.latent_layout(case.num_pages, kv.FP16)
    out = torch.empty((1, 128, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((1, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, 1, 128, 4156), dtype=torch.uint8, device=dev)
    err = kv.new_error_word(dev)
    kv.decode_mla(ql.to(dev), qr.to(dev), lay, torch.from_numpy(ocache).to(dev), case.block_table.to(dev),
                  torch.from_numpy(sl).to(dev), 4156, out, ws, err, sm,
                  torch.from_numpy(tl).half().to(dev), torch.from_numpy(tr).half().to(dev), lse=lse)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    diff = np.abs(parity.f64(out) - ref).max()
    print(f"\nmla decode fp16, 32 tiles + 60: max |out - oracle| = {diff:.3e}")
    assert diff <= parity.OUT_ATOL
    np.testing.assert_allclose(parity.f64(lse), ref_lse, atol=1e-4, rtol=0)


@pytest.mark.parametrize("heads", [16, 48])
def test_decode_mla_head_counts_inside_a_warp(heads):
    """Head counts whose last row falls inside a warp of the tensor-memory
    lanes (16, 48): the padded rows take part in the tensor-memory loads and
    write nothing."""
    wl, case = _case(num_seqs=1, heads=heads, context=300)
    olay = layout.LatentLayout(512, 64, 128)
    lat, rope = parity.f64(case.latent), parity.f64(case.rope)
    bt, sl = case.block_table.numpy(), case.seq_lens.numpy()
    ocache = np.zeros((case.num_pages, olay.page_bytes), np.uint8)
    mla.encode_into_cache(ocache, olay, lat[:, :256], rope[:, :256], bt, [0])
    tl = np.zeros((1, 128, 512))
    tr = np.zeros((1, 128, 64))
    tl[0, :44], tr[0, :44] = lat[0, 256:300], rope[0, 256:300]
    sm = W.default_sm_scale(wl)
    ref, _ = mla.decode(parity.f64(case.q_latent), parity.f64(case.q_rope), ocache, olay, bt, sl, sm, tl, tr)
    dev = "cuda"
    lay = kv.latent_layout(case.num_pages, kv.BF16)
    out = torch.empty((1, heads, 512), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, 1, heads, 300), dtype=torch.uint8, device=dev)
    err = kv.new_error_word(dev)
    kv.decode_mla(case.q_latent.to(dev), case.q_rope.to(dev), lay, torch.from_numpy(ocache).to(dev),
                  case.block_table.to(dev), torch.from_numpy(sl).to(dev), 300, out, ws, err, sm,
                  torch.from_numpy(tl).to(torch.bfloat16).to(dev), torch.from_numpy(tr).half().to(dev))
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    diff = np.abs(parity.f64(out) - ref).max()
    print(f"\nmla decode {heads} heads: max |out - oracle| = {diff:.3e}")
    assert diff <= parity.OUT_ATOL
