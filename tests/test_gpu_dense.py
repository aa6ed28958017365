"""GPU parity of the dense codec and decode attention against the oracle,
through the C ABI, on seeded inputs shaped like the named workloads but small
enough for the oracle (several tiles, ragged splits, variable lengths, fp16
tails, bf16 and head_dim 256)."""
import numpy as np
import pytest
import torch

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import workloads as W
from oracle import attention, layout
from tests import parity

pytestmark = pytest.mark.gpu

CASES = {
    # name: (workload, overrides)
    "toy": ("toy", {}),
    "dense_small": ("dense32b", dict(num_seqs=2, num_q_heads=16, num_kv_heads=2, context=1152)),
    "g64_small": ("g64", dict(num_seqs=3, num_q_heads=16, num_kv_heads=2, context=1000, min_context=1)),
    "hybrid_small": ("hybrid", dict(num_seqs=2, num_q_heads=12, num_kv_heads=2, context=768)),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_kv_cache_kvarn_gb300 import build
    build.build()
    kv.lib()


def _case(name):
    wname, over = CASES[name]
    wl = W.WORKLOADS[wname].with_(**over)
    return wl, W.make_dense(wl, device="cpu")


def _gpu_encode(wl, case, dev="cuda"):
    lay = kv.dense_layout(wl.head_dim, wl.tile_tokens, wl.num_kv_heads, case.num_pages,
                          kv.BF16 if wl.dtype == "bf16" else kv.FP16, wl.norm_iters)
    cache = kv.alloc_cache(lay, dev)
    err = kv.new_error_word(dev)
    # encode every committed tile, one sequence at a time (lengths differ)
    bt = case.block_table.to(dev)
    for b in range(wl.num_seqs):
        tiles = int(case.seq_lens[b]) // wl.tile_tokens
        if tiles:
            kv.encode_tiles(case.k[b:b + 1].to(dev), case.v[b:b + 1].to(dev), lay,
                            torch.zeros(1, dtype=torch.int32, device=dev), bt[b:b + 1], cache, err,
                            chunk_tokens=tiles * wl.tile_tokens)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    return lay, cache


@pytest.mark.parametrize("name", list(CASES))
def test_encode_matches_oracle(name):
    wl, case = _case(name)
    lay, cache = _gpu_encode(wl, case)
    st_k, st_v = parity.check_dense_pages(cache.cpu().numpy(), parity.f64(case.k), parity.f64(case.v),
                                          case.block_table.numpy(), case.seq_lens.numpy(),
                                          wl.tile_tokens, wl.head_dim)
    print(f"\n{name}: K codes {st_k['mismatch']}/{st_k['codes']} differ (max dist {st_k['max_dist']:.2e}, "
          f"{st_k['within_1ulp']} within 1 ulp); V {st_v['mismatch']}/{st_v['codes']}; "
          f"scale rel {max(st_k['scale_rel'], st_v['scale_rel']):.2e}")


def test_encode_is_idempotent_and_touches_only_its_pages():
    wl, case = _case("dense_small")
    lay, cache1 = _gpu_encode(wl, case)
    lay, cache2 = _gpu_encode(wl, case)
    assert torch.equal(cache1, cache2)
    # pages never named by the block table stay zero
    used = set(case.block_table[case.block_table >= 0].tolist())
    unused = [p for p in range(case.num_pages) if p not in used]
    if unused:
        assert int(cache1[unused].abs().sum()) == 0


def test_negative_tile_start_skips_the_sequence():
    """One commit call for a batch in which only some sequences filled a
    tile: a negative tile_start leaves that sequence's pages untouched and
    the others get exactly the bytes of a call without it."""
    wl, case = _case("dense_small")
    dev = "cuda"
    lay = kv.dense_layout(wl.head_dim, wl.tile_tokens, wl.num_kv_heads, case.num_pages)
    N = wl.tile_tokens
    bt = case.block_table.to(dev)
    k, v = case.k[:, :, N:2 * N].contiguous().to(dev), case.v[:, :, N:2 * N].contiguous().to(dev)
    both = kv.alloc_cache(lay, dev)
    err = kv.new_error_word(dev)
    kv.encode_tiles(k, v, lay, torch.tensor([1, 1], dtype=torch.int32, device=dev), bt, both, err, chunk_tokens=N)
    only1 = kv.alloc_cache(lay, dev)
    kv.encode_tiles(k, v, lay, torch.tensor([-1, 1], dtype=torch.int32, device=dev), bt, only1, err, chunk_tokens=N)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    ppt = N // 16
    pages0 = case.block_table[0, ppt:2 * ppt].tolist()
    pages1 = case.block_table[1, ppt:2 * ppt].tolist()
    assert int(only1[pages0].abs().sum()) == 0
    assert torch.equal(only1[pages1], both[pages1])
    assert int(both[pages0].abs().sum()) > 0


@pytest.mark.parametrize("name", list(CASES))
def test_decode_on_oracle_pages_matches_oracle(name):
    wl, case = _case(name)
    k, v = parity.f64(case.k), parity.f64(case.v)
    bt, lens = case.block_table.numpy(), case.seq_lens.numpy()
    N, D = wl.tile_tokens, wl.head_dim
    ocache = parity.oracle_dense_cache(k, v, bt, lens, N, D, case.num_pages)
    tk, tv = parity.tails(k, lens, N), parity.tails(v, lens, N)
    sm = W.default_sm_scale(wl)
    ref, ref_lse = attention.decode(parity.f64(case.q), ocache, layout.DenseLayout(D, N), bt, lens, sm, tk, tv)

    dev = "cuda"
    dt = W.TORCH_DTYPE[wl.dtype]
    lay = kv.dense_layout(D, N, wl.num_kv_heads, case.num_pages, kv.BF16 if wl.dtype == "bf16" else kv.FP16)
    Lmax = int(lens.max())
    out = torch.empty((wl.num_seqs, wl.num_q_heads, D), dtype=torch.float32, device=dev)
    lse = torch.empty((wl.num_seqs, wl.num_q_heads), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, wl.num_seqs, wl.num_q_heads, Lmax), dtype=torch.uint8,
                     device=dev)
    err = kv.new_error_word(dev)
    tail_k = torch.from_numpy(tk).to(dt).to(dev)
    tail_v = torch.from_numpy(tv).to(dt).to(dev)
    kv.decode(case.q.to(dev), lay, torch.from_numpy(ocache).to(dev), case.block_table.to(dev),
              case.seq_lens.to(dev), Lmax, out, ws, err, sm, tail_k, tail_v, lse=lse)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    diff = np.abs(parity.f64(out) - ref).max()
    print(f"\n{name}: max |out - oracle| = {diff:.3e}, max |lse - oracle| = "
          f"{np.abs(parity.f64(lse) - ref_lse).max():.3e}")
    assert diff <= parity.OUT_ATOL
    np.testing.assert_allclose(parity.f64(lse), ref_lse, atol=1e-4, rtol=0)


@pytest.mark.parametrize("name", ["toy", "g64_small"])
def test_end_to_end_close_to_oracle(name):
    """GPU encode then GPU decode against oracle encode then oracle decode. The
    only difference between the two caches is the few near-boundary code
    flips, so the bound is the output tolerance itself."""
    wl, case = _case(name)
    lay, cache = _gpu_encode(wl, case)
    k, v = parity.f64(case.k), parity.f64(case.v)
    bt, lens = case.block_table.numpy(), case.seq_lens.numpy()
    N, D = wl.tile_tokens, wl.head_dim
    ocache = parity.oracle_dense_cache(k, v, bt, lens, N, D, case.num_pages)
    tk, tv = parity.tails(k, lens, N), parity.tails(v, lens, N)
    sm = W.default_sm_scale(wl)
    ref, _ = attention.decode(parity.f64(case.q), ocache, layout.DenseLayout(D, N), bt, lens, sm, tk, tv)
    dev = "cuda"
    dt = W.TORCH_DTYPE[wl.dtype]
    Lmax = int(lens.max())
    out = torch.empty((wl.num_seqs, wl.num_q_heads, D), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, wl.num_seqs, wl.num_q_heads, Lmax), dtype=torch.uint8,
                     device=dev)
    err = kv.new_error_word(dev)
    kv.decode(case.q.to(dev), lay, cache, case.block_table.to(dev), case.seq_lens.to(dev), Lmax, out, ws,
              err, sm, torch.from_numpy(tk).to(dt).to(dev), torch.from_numpy(tv).to(dt).to(dev))
    torch.cuda.synchronize()
    diff = np.abs(parity.f64(out) - ref).max()
    print(f"\n{name}: end-to-end max |out - oracle| = {diff:.3e}")
    assert diff <= parity.OUT_ATOL


def test_decode_edge_lengths():
    """Empty sequence, tail only, exactly one tile, one tile plus one token."""
    wl = W.WORKLOADS["dense32b"].with_(num_seqs=4, num_q_heads=8, num_kv_heads=1, context=256)
    case = W.make_dense(wl, device="cpu")
    lens = np.array([0, 77, 128, 129], dtype=np.int32)
    k, v = parity.f64(case.k), parity.f64(case.v)
    bt = case.block_table.numpy()
    ocache = parity.oracle_dense_cache(k, v, bt, lens, 128, 128, case.num_pages)
    tk, tv = parity.tails(k, lens, 128), parity.tails(v, lens, 128)
    ref, ref_lse = attention.decode(parity.f64(case.q), ocache, layout.DenseLayout(128, 128), bt, lens, 0.1,
                                    tk, tv)
    dev = "cuda"
    lay = kv.dense_layout(128, 128, 1, case.num_pages)
    out = torch.empty((4, 8, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((4, 8), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, 4, 8, 256), dtype=torch.uint8, device=dev)
    err = kv.new_error_word(dev)
    kv.decode(case.q.to(dev), lay, torch.from_numpy(ocache).to(dev), case.block_table.to(dev),
              torch.from_numpy(lens).to(dev), 256, out, ws, err, 0.1,
              torch.from_numpy(tk).half().to(dev), torch.from_numpy(tv).half().to(dev), lse=lse)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    o = parity.f64(out)
    assert (o[0] == 0).all() and np.isneginf(parity.f64(lse)[0]).all()
    assert np.abs(o[1:] - ref[1:]).max() <= parity.OUT_ATOL


def test_decode_many_ragged_sequences():
    """More sequences than a warp scans at once (the CTAs locate their tiles
    with warp-wide scans over 32 sequences at a time), lengths from empty to
    five tiles with and without tails: every CTA range of the flattened tile
    list crosses unit boundaries, so units get one to several partials."""
    B, Hq, Hkv, N, Lmax = 70, 8, 2, 128, 640
    wl = W.WORKLOADS["dense32b"].with_(num_seqs=B, num_q_heads=Hq, num_kv_heads=Hkv, context=Lmax)
    case = W.make_dense(wl, device="cpu")
    rng = np.random.default_rng(7)
    lens = rng.integers(0, Lmax + 1, size=B).astype(np.int32)
    lens[:6] = [0, N, 2 * N, 5 * N, 1, N - 1]
    lens[40:44] = 0
    k, v = parity.f64(case.k), parity.f64(case.v)
    bt = case.block_table.numpy()
    ocache = parity.oracle_dense_cache(k, v, bt, lens, N, 128, case.num_pages)
    tk, tv = parity.tails(k, lens, N), parity.tails(v, lens, N)
    ref, ref_lse = attention.decode(parity.f64(case.q), ocache, layout.DenseLayout(128, N), bt, lens, 0.1, tk, tv)
    dev = "cuda"
    lay = kv.dense_layout(128, N, Hkv, case.num_pages)
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, B, Hq, Lmax), dtype=torch.uint8, device=dev)
    err = kv.new_error_word(dev)
    for _ in range(2):  # the second call reuses a workspace full of the first call's partials
        kv.decode(case.q.to(dev), lay, torch.from_numpy(ocache).to(dev), case.block_table.to(dev),
                  torch.from_numpy(lens).to(dev), Lmax, out, ws, err, 0.1,
                  torch.from_numpy(tk).half().to(dev), torch.from_numpy(tv).half().to(dev), lse=lse)
        torch.cuda.synchronize()
        assert kv.read_error_flags(err) == 0
        o, l = parity.f64(out), parity.f64(lse)
        empty = lens == 0
        assert (o[empty] == 0).all() and np.isneginf(l[empty]).all()
        diff = np.abs(o[~empty] - ref[~empty]).max()
        print(f"\nmany_ragged: max |out - oracle| = {diff:.3e}, "
              f"max |lse - oracle| = {np.abs(l[~empty] - ref_lse[~empty]).max():.3e}")
        assert diff <= parity.OUT_ATOL
        assert np.abs(l[~empty] - ref_lse[~empty]).max() <= 1e-4


def test_device_errors_are_flagged_not_faulted():
    """A block-table entry outside the cache and a missing tail set bits of the
    error word; the kernel reads a valid page instead and finishes."""
    wl = W.WORKLOADS["toy"].with_(context=300)
    case = W.make_dense(wl, device="cpu")
    dev = "cuda"
    lay = kv.dense_layout(128, 128, 1, case.num_pages)
    cache = kv.alloc_cache(lay, dev)
    err = kv.new_error_word(dev)
    bt = case.block_table.clone()
    bt[0, 3] = case.num_pages + 5
    kv.encode_tiles(case.k.to(dev), case.v.to(dev), lay, torch.zeros(1, dtype=torch.int32, device=dev),
                    bt.to(dev), cache, err, chunk_tokens=256)
    assert kv.read_error_flags(err) & kv.DEVERR_PAGE_RANGE
    err.zero_()
    out = torch.empty((1, 4, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, 1, 4, 300), dtype=torch.uint8, device=dev)
    kv.decode(case.q.to(dev), lay, cache, bt.to(dev), case.seq_lens.to(dev), 300, out, ws, err, 0.1)
    flags = kv.read_error_flags(err)
    assert flags & kv.DEVERR_PAGE_RANGE and flags & kv.DEVERR_NO_TAIL


@pytest.mark.parametrize("D", [128, 256])
def test_fp16_bypass_matches_plain_attention(D):
    """The uncompressed path on the same skeleton (the decode kernel with no
    codec, 32-token tiles) equals plain attention over the raw tokens: ragged
    last pages and tiles, a one-page sequence, an empty one; the rows past a
    length in its last page hold NaN and must take no weight."""
    B = 4
    wl = W.WORKLOADS["dense32b"].with_(num_seqs=B, num_q_heads=16, num_kv_heads=2, context=700, head_dim=D)
    case = W.make_dense(wl, device="cpu")
    lens = np.array([700, 333, 16, 0], dtype=np.int32)
    dev = "cuda"
    num_pages = B * ((700 + 15) // 16)
    bt = torch.arange(num_pages, dtype=torch.int32).flip(0).reshape(B, -1).contiguous()
    lay = kv.dense_layout(D, 128, 2, num_pages)
    cache = kv.alloc_fp16_cache(lay, dev)
    err = kv.new_error_word(dev)
    kpad = torch.full((B, 2, 704, D), float("nan"), dtype=torch.float16)
    vpad = torch.full_like(kpad, float("nan"))
    for b in range(B):
        kpad[b, :, :lens[b]] = case.k[b, :, :lens[b]]
        vpad[b, :, :lens[b]] = case.v[b, :, :lens[b]]
    kv.store_fp16(kpad.to(dev), vpad.to(dev), lay, 0, 704, bt.to(dev), cache, err)
    out = torch.empty((B, 16, D), dtype=torch.float32, device=dev)
    lse = torch.empty((B, 16), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, B, 16, 700), dtype=torch.uint8, device=dev)
    sm = 1 / np.sqrt(D)
    kv.decode_fp16(case.q.to(dev), lay, cache, bt.to(dev), torch.from_numpy(lens).to(dev), 700, out, ws, err, sm,
                   lse=lse)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    o, l = parity.f64(out), parity.f64(lse)
    assert (o[3] == 0).all() and np.isneginf(l[3]).all()
    worst = 0.0
    for b in range(3):
        for h in range(16):
            ref, rl = attention.softmax_attention(parity.f64(case.q[b, h]), parity.f64(case.k[b, h // 8, :lens[b]]),
                                                  parity.f64(case.v[b, h // 8, :lens[b]]), sm)
            worst = max(worst, float(np.abs(o[b, h] - ref).max()))
            assert abs(l[b, h] - rl) <= 1e-4
    parity.report(f"fp16 pages D{D}: max |out - plain attention| = {worst:.3e}")
    assert worst <= parity.OUT_ATOL
