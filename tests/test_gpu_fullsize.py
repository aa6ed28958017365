"""Full-size parity on the five named workloads, in the launch configuration
the benchmark times (whole batch, full context, the library's own split
plan).

For each workload the CUDA path encodes the whole cache from inputs drawn
on the device. Sampled (sequence, KV head) pairs are then checked against
the oracle one by one: their pages against the oracle's encoding of the
same tokens, and their decode outputs against the oracle's decode over the
oracle's pages (which replace the GPU-written pages of those pairs before
the GPU decode runs, so that the decode comparison does not depend on the
few near-boundary code flips)."""
import numpy as np
import pytest
import torch

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import workloads as W
from oracle import attention, codec, layout, mla
from tests import parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_kv_cache_kvarn_gb300 import build
    build.build()
    kv.lib()


def _encode_dense(case, wl, lay, cache, err, chunk_from=None):
    """Encode every committed tile; for `chunk_from` = (start_token, chunk),
    the last `chunk` tokens of every sequence are encoded in a second call
    (the prefill-chunk path, tile_start > 0)."""
    N = wl.tile_tokens
    lens = case.seq_lens.cpu().tolist()
    if len(set(lens)) == 1 and chunk_from is None:
        kv.encode_tiles(case.k, case.v, lay, torch.zeros(wl.num_seqs, dtype=torch.int32, device=DEV),
                        case.block_table, cache, err, chunk_tokens=(lens[0] // N) * N)
        return
    if chunk_from is not None:
        start, chunk = chunk_from
        kv.encode_tiles(case.k, case.v, lay, torch.zeros(wl.num_seqs, dtype=torch.int32, device=DEV),
                        case.block_table, cache, err, chunk_tokens=start)
        ts = torch.full((wl.num_seqs,), start // N, dtype=torch.int32, device=DEV)
        kv.encode_tiles(case.k[:, :, start:], case.v[:, :, start:], lay, ts, case.block_table, cache, err,
                        chunk_tokens=chunk)
        return
    for b, L in enumerate(lens):
        if L // N:
            kv.encode_tiles(case.k[b:b + 1], case.v[b:b + 1], lay, torch.zeros(1, dtype=torch.int32, device=DEV),
                            case.block_table[b:b + 1], cache, err, chunk_tokens=(L // N) * N)


@pytest.mark.parametrize("name,pairs,chunk", [
    # pairs spread over the batch (first, middle and last sequences, several
    # KV heads), so that the sampled units sit in different CTA ranges of
    # the full-size split plan
    ("dense32b", [(0, 0), (3, 5), (17, 3), (30, 0), (31, 7)], None),
    ("g64", [(0, 0), (1, 2), (17, 7), (31, 4)], None),
    ("hybrid", [(0, 0), (5, 3), (7, 1)], (61440, 4096)),
])
def test_dense_fullsize(name, pairs, chunk):
    wl = W.WORKLOADS[name]
    case = W.make_dense(wl, device=DEV)
    N, D = wl.tile_tokens, wl.head_dim
    dt = kv.BF16 if wl.dtype == "bf16" else kv.FP16
    lay = kv.dense_layout(D, N, wl.num_kv_heads, case.num_pages, dt, wl.norm_iters)
    cache = kv.alloc_cache(lay, DEV)
    err = kv.new_error_word(DEV)
    _encode_dense(case, wl, lay, cache, err, chunk)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0

    lens = case.seq_lens.cpu().numpy()
    bt = case.block_table.cpu().numpy()
    olay = layout.DenseLayout(D, N)
    ppt = N // 16
    host = np.zeros((case.num_pages, wl.num_kv_heads, olay.page_bytes), np.uint8)
    st_k, st_v = parity.new_stats(), parity.new_stats()
    G = wl.group
    for b, h in pairs:
        L = int(lens[b])
        T = L // N
        pages = bt[b, :T * ppt]
        gpu_pages = cache[torch.from_numpy(pages).long().to(DEV), h].cpu().numpy()
        host[pages, h] = gpu_pages
        kbh = parity.f64(case.k[b, h, :L])
        vbh = parity.f64(case.v[b, h, :L])
        for t in range(T):
            pg = [int(x) for x in pages[t * ppt:(t + 1) * ppt]]
            gk, gv = layout.read_tile(host, olay, pg, h)
            ek = codec.encode_tile(kbh[t * N:(t + 1) * N], 4, wl.norm_iters)
            ev = codec.encode_tile(vbh[t * N:(t + 1) * N], 2, wl.norm_iters)
            parity.compare_tile(gk, ek, 4, st_k)
            parity.compare_tile(gv, ev, 2, st_v)
            layout.write_tile(host, olay, pg, h, ek, ev)      # oracle pages for the decode check
        cache[torch.from_numpy(pages).long().to(DEV), h] = torch.from_numpy(host[pages, h]).to(DEV)
    for st in (st_k, st_v):
        assert st["scale_rel"] <= parity.SCALE_RTOL, st
        assert st["mismatch"] <= max(4, 1e-3 * st["codes"]), st
    print(f"\n{name}: K codes {st_k['mismatch']}/{st_k['codes']} differ, V {st_v['mismatch']}/{st_v['codes']}, "
          f"scale rel {max(st_k['scale_rel'], st_v['scale_rel']):.2e}")

    # tails (raw tokens past the last full tile) and the decode of the whole batch
    tk = torch.zeros((wl.num_seqs, wl.num_kv_heads, N, D), dtype=case.k.dtype, device=DEV)
    tv = torch.zeros_like(tk)
    for b in range(wl.num_seqs):
        c, L = (int(lens[b]) // N) * N, int(lens[b])
        if L > c:
            tk[b, :, :L - c] = case.k[b, :, c:L]
            tv[b, :, :L - c] = case.v[b, :, c:L]
    Lmax = int(lens.max())
    out = torch.empty((wl.num_seqs, wl.num_q_heads, D), dtype=torch.float32, device=DEV)
    ws = torch.empty(kv.decode_workspace_bytes(lay, wl.num_seqs, wl.num_q_heads, Lmax), dtype=torch.uint8,
                     device=DEV)
    sm = W.default_sm_scale(wl)
    kv.decode(case.q, lay, cache, case.block_table, case.seq_lens, Lmax, out, ws, err, sm, tk, tv)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    heads = [(b, h * G + j) for b, h in pairs for j in range(G)]
    tk_h, tv_h = parity.f64(tk), parity.f64(tv)
    ref, _ = attention.decode(parity.f64(case.q), host, olay, bt, lens, sm, tk_h, tv_h, heads=heads)
    o = parity.f64(out)
    diff = max(np.abs(o[b, hq] - ref[b, hq]).max() for b, hq in heads)
    print(f"{name}: max |out - oracle| over {len(heads)} sampled heads = {diff:.3e}")
    assert diff <= parity.OUT_ATOL


def test_mla_fullsize():
    wl = W.WORKLOADS["mla"]
    case = W.make_latent(wl, device=DEV)
    lay = kv.latent_layout(case.num_pages, kv.BF16, wl.norm_iters)
    cache = kv.alloc_cache(lay, DEV)
    err = kv.new_error_word(DEV)
    L = wl.context
    kv.encode_latent(case.latent, case.rope, lay, torch.zeros(wl.num_seqs, dtype=torch.int32, device=DEV),
                     case.block_table, cache, err, chunk_tokens=L)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    bt = case.block_table.cpu().numpy()
    olay = layout.LatentLayout(512, 64, 128)
    host = np.zeros((case.num_pages, olay.page_bytes), np.uint8)
    stats = parity.new_stats()
    seqs = [7, 50]
    for b in seqs:
        pages = bt[b, :L // 16]
        host[pages] = cache[torch.from_numpy(pages).long().to(DEV)].cpu().numpy()
        lat = parity.f64(case.latent[b])
        rope = parity.f64(case.rope[b])
        for t in range(L // 128):
            pg = [int(x) for x in pages[t * 8:(t + 1) * 8]]
            enc, rp = mla.read_tile(host, olay, pg)
            ref = codec.encode_tile(lat[t * 128:(t + 1) * 128], 4, wl.norm_iters)
            parity.compare_tile(enc, ref, 4, stats)
            np.testing.assert_array_equal(rp, rope[t * 128:(t + 1) * 128])
            mla.write_tile(host, olay, pg, ref, rope[t * 128:(t + 1) * 128])
        cache[torch.from_numpy(pages).long().to(DEV)] = torch.from_numpy(host[pages]).to(DEV)
    assert stats["scale_rel"] <= parity.SCALE_RTOL, stats
    assert stats["mismatch"] <= max(4, 1e-3 * stats["codes"]), stats
    out = torch.empty((wl.num_seqs, 128, 512), dtype=torch.float32, device=DEV)
    ws = torch.empty(kv.decode_workspace_bytes(lay, wl.num_seqs, 128, L), dtype=torch.uint8, device=DEV)
    sm = W.default_sm_scale(wl)
    kv.decode_mla(case.q_latent, case.q_rope, lay, cache, case.block_table, case.seq_lens, L, out, ws, err, sm)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    heads = [(b, h) for b in seqs for h in (0, 37, 90, 127)]
    ref, _ = mla.decode(parity.f64(case.q_latent), parity.f64(case.q_rope), host, olay, bt,
                        case.seq_lens.cpu().numpy(), sm, heads=heads)
    o = parity.f64(out)
    diff = max(np.abs(o[b, h] - ref[b, h]).max() for b, h in heads)
    print(f"\nmla: codes {stats['mismatch']}/{stats['codes']} differ; max |out - oracle| = {diff:.3e}")
    assert diff <= parity.OUT_ATOL


def test_degenerate_tiles():
    """Constant tiles, zero tiles and a tile with one constant column: the
    std passes fall back to 1 and a zero-range row gets delta 0; the CUDA
    encoder must agree with the oracle on all of them."""
    wl = W.WORKLOADS["dense32b"].with_(num_seqs=1, num_q_heads=8, num_kv_heads=1, context=512)
    case = W.make_dense(wl, device="cpu")
    k, v = case.k.clone(), case.v.clone()
    k[0, 0, :128] = 3.0                  # constant tile
    v[0, 0, :128] = 0.0                  # zero tile
    k[0, 0, 128:256, 17] = -2.0          # one constant channel
    v[0, 0, 256:384] = v[0, 0, 256:257]  # all tokens equal (every column constant)
    lay = kv.dense_layout(128, 128, 1, case.num_pages)
    cache = kv.alloc_cache(lay, DEV)
    err = kv.new_error_word(DEV)
    kv.encode_tiles(k.to(DEV), v.to(DEV), lay, torch.zeros(1, dtype=torch.int32, device=DEV),
                    case.block_table.to(DEV), cache, err)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    g = cache.cpu().numpy()
    olay = layout.DenseLayout(128, 128)
    for t in range(4):
        pg = [int(x) for x in case.block_table[0, t * 8:(t + 1) * 8]]
        gk, gv = layout.read_tile(g, olay, pg, 0)
        for got, x, bits in ((gk, parity.f64(k[0, 0, t * 128:(t + 1) * 128]), 4),
                             (gv, parity.f64(v[0, 0, t * 128:(t + 1) * 128]), 2)):
            ref = codec.encode_tile(x, bits, 2)
            st = parity.new_stats()
            parity.compare_tile(got, ref, bits, st)   # near-boundary flips only
            assert st["mismatch"] <= 4 and st["scale_rel"] <= parity.SCALE_RTOL, (t, bits, st)
            rec = codec.dequantize(got["codes"], got["a"], got["b"], got["c"])
            assert np.isfinite(rec).all()


@pytest.mark.parametrize("Q,S,R,pairs", [(1, 128, 1024, [(0, 0), (13, 6), (31, 7)]),
                                         (4, 128, 256, [(2, 1), (29, 4)])])
def test_window_fullsize(Q, S, R, pairs):
    """The raw-record decode (sink S + recent R raw tokens, Q query tokens)
    on the full dense32b batch: every (sequence, KV head) unit has S + R or
    more raw tokens, so the raw records span several splits of the full-size
    plan. Sampled pairs get the oracle's pages; their rows are checked
    against the oracle's window decode."""
    wl = W.WORKLOADS["dense32b"]
    case = W.make_dense(wl, device=DEV)
    N, D, B, Hkv = wl.tile_tokens, wl.head_dim, wl.num_seqs, wl.num_kv_heads
    lay = kv.dense_layout(D, N, Hkv, case.num_pages, kv.FP16, wl.norm_iters)
    cache = kv.alloc_cache(lay, DEV)
    err = kv.new_error_word(DEV)
    _encode_dense(case, wl, lay, cache, err)
    torch.cuda.synchronize()
    lens = case.seq_lens.cpu().numpy()
    bt = case.block_table.cpu().numpy()
    olay = layout.DenseLayout(D, N)
    ppt = N // 16
    host = np.zeros((case.num_pages, Hkv, olay.page_bytes), np.uint8)
    for b, h in pairs:
        L = int(lens[b])
        C = attention.window_committed(L, Q, N, S, R)
        kbh, vbh = parity.f64(case.k[b, h, :L]), parity.f64(case.v[b, h, :L])
        for t in range(S // N, C // N):
            pg = [int(x) for x in bt[b, t * ppt:(t + 1) * ppt]]
            layout.write_tile(host, olay, pg, h, codec.encode_tile(kbh[t * N:(t + 1) * N], 4, wl.norm_iters),
                              codec.encode_tile(vbh[t * N:(t + 1) * N], 2, wl.norm_iters))
        pages = torch.from_numpy(bt[b, (S // N) * ppt:(C // N) * ppt]).long().to(DEV)
        cache[pages, h] = torch.from_numpy(host[bt[b, (S // N) * ppt:(C // N) * ppt], h]).to(DEV)
    sink_k, sink_v = case.k[:, :, :S].contiguous(), case.v[:, :, :S].contiguous()
    cap = R + N + Q - 2
    tail_k = torch.zeros((B, Hkv, cap, D), dtype=case.k.dtype, device=DEV)
    tail_v = torch.zeros_like(tail_k)
    for b in range(B):
        L = int(lens[b])
        C = attention.window_committed(L, Q, N, S, R)
        tail_k[b, :, :L - C] = case.k[b, :, C:L]
        tail_v[b, :, :L - C] = case.v[b, :, C:L]
    q = W.verify_queries(wl, Q, device=DEV)
    Lmax = int(lens.max())
    out = torch.empty((B, Q, wl.num_q_heads, D), dtype=torch.float32, device=DEV)
    ws = torch.empty(kv.decode_window_workspace_bytes(lay, B, wl.num_q_heads, Q, Lmax, S, R), dtype=torch.uint8,
                     device=DEV)
    sm = W.default_sm_scale(wl)
    kv.decode_window(q, lay, cache, case.block_table, case.seq_lens, Lmax, out, ws, err, sm, sink_k=sink_k,
                     sink_v=sink_v, recent_tokens=R, tail_k=tail_k, tail_v=tail_v)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    G = wl.group
    rows = [(b, j, h * G + g) for b, h in pairs for j in range(Q) for g in range(G)]
    ref, _ = attention.decode_window(parity.f64(q), host, olay, bt, lens, sm, S, R, parity.f64(sink_k),
                                     parity.f64(sink_v), parity.f64(tail_k), parity.f64(tail_v), rows=rows)
    o = parity.f64(out)
    diff = max(np.abs(o[b, j, hq] - ref[b, j, hq]).max() for b, j, hq in rows)
    print(f"window Q{Q} S{S} R{R}: max |out - oracle| over {len(rows)} sampled rows = {diff:.3e}")
    assert diff <= parity.OUT_ATOL
