"""GPU parity of the decode with raw sink and recent records (the gmlx
record policy) against the oracle, through the C ABI, on pages the oracle
wrote: only the tiles between the sink and the newest records are read from
the pages."""
import numpy as np
import pytest
import torch

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import workloads as W
from oracle import attention, layout
from tests import parity

pytestmark = pytest.mark.gpu

CASES = {
    # name: (workload, overrides, Q, sink, recent, lengths)
    "g8_sink128_recent256": ("dense32b", dict(num_seqs=3, num_q_heads=16, num_kv_heads=2, context=1100), 1, 128, 256,
                             [1100, 700, 300]),
    "g64_q3_sink128_recent100": ("g64", dict(num_seqs=4, num_q_heads=8, num_kv_heads=2, context=900, min_context=1),
                                 3, 128, 100,
                                 [900, 333, 129, 60]),
    "hybrid_q2_bf16": ("hybrid", dict(num_seqs=2, num_q_heads=12, num_kv_heads=2, context=800), 2, 128, 128,
                       [800, 517]),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_kv_cache_kvarn_gb300 import build
    build.build()
    kv.lib()


def _setup(name):
    wname, over, Q, S, R, lens = CASES[name]
    wl = W.WORKLOADS[wname].with_(**over)
    case = W.make_dense(wl, device="cpu")
    N, D, B, Hkv = wl.tile_tokens, wl.head_dim, wl.num_seqs, wl.num_kv_heads
    lens = np.array(lens, np.int32)
    k, v = parity.f64(case.k), parity.f64(case.v)
    lay = layout.DenseLayout(D, N)
    ppt = N // 16
    ends = [attention.window_committed(int(L), Q, N, S, R) for L in lens]
    rows = max(1, max(e // 16 for e in ends))
    bt = np.full((B, rows), -1, np.int32)
    num_pages = max(1, sum((e - S) // 16 for e in ends if e > S))
    order = np.random.default_rng(7).permutation(num_pages)
    off = 0
    for b, e in enumerate(ends):
        for t in range(S // N, e // N):  # pages only for the compressed tiles
            bt[b, t * ppt:(t + 1) * ppt] = order[off:off + ppt]
            off += ppt
    cache = np.zeros((num_pages, Hkv, lay.page_bytes), np.uint8)
    for b, e in enumerate(ends):
        if e > S:
            attention.encode_into_cache(cache, lay, k[b:b + 1, :, S:e], v[b:b + 1, :, S:e], bt[b:b + 1], [S // N])
    dt = W.TORCH_DTYPE[wl.dtype]
    sink_k = torch.zeros((B, Hkv, S, D), dtype=dt)
    sink_v = torch.zeros_like(sink_k)
    cap = R + N + Q - 2
    tail_k = torch.zeros((B, Hkv, cap, D), dtype=dt)
    tail_v = torch.zeros_like(tail_k)
    for b, (L, e) in enumerate(zip(lens, ends)):
        n = min(S, int(L))
        sink_k[b, :, :n], sink_v[b, :, :n] = case.k[b, :, :n], case.v[b, :, :n]
        if L > e:
            tail_k[b, :, :L - e], tail_v[b, :, :L - e] = case.k[b, :, e:L], case.v[b, :, e:L]
    q = W.verify_queries(wl, Q)
    return wl, Q, S, R, lens, bt, cache, sink_k, sink_v, tail_k, tail_v, q


def _run(wl, Q, S, R, lens, bt, cache, sink_k, sink_v, tail_k, tail_v, q, sm, window=True):
    dev = "cuda"
    B, Hq, D = wl.num_seqs, wl.num_q_heads, wl.head_dim
    lay = kv.dense_layout(D, wl.tile_tokens, wl.num_kv_heads, cache.shape[0],
                          kv.BF16 if wl.dtype == "bf16" else kv.FP16)
    Lmax = int(lens.max())
    out = torch.empty((B, Q, Hq, D), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Q, Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_window_workspace_bytes(lay, B, Hq, Q, Lmax, S, R), dtype=torch.uint8, device=dev)
    err = kv.new_error_word(dev)
    args = (q.to(dev), lay, torch.from_numpy(cache).to(dev), torch.from_numpy(bt).to(dev),
            torch.from_numpy(lens).to(dev), Lmax, out, ws, err, sm)
    if window:
        kv.decode_window(*args, sink_k=sink_k.to(dev) if S else None, sink_v=sink_v.to(dev) if S else None,
                         recent_tokens=R, tail_k=tail_k.to(dev), tail_v=tail_v.to(dev), lse=lse)
    else:
        kv.decode_verify(*args, tail_k.to(dev), tail_v.to(dev), lse=lse)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    return out, lse


@pytest.mark.parametrize("name", list(CASES))
def test_window_matches_oracle(name):
    wl, Q, S, R, lens, bt, cache, sink_k, sink_v, tail_k, tail_v, q = _setup(name)
    sm = W.default_sm_scale(wl)
    ref, rlse = attention.decode_window(parity.f64(q), cache, layout.DenseLayout(wl.head_dim, wl.tile_tokens),
                                        bt, lens, sm, S, R, parity.f64(sink_k), parity.f64(sink_v),
                                        parity.f64(tail_k), parity.f64(tail_v))
    out, lse = _run(wl, Q, S, R, lens, bt, cache, sink_k, sink_v, tail_k, tail_v, q, sm)
    out, lse = parity.f64(out), parity.f64(lse)
    diff = np.abs(out - ref).max()
    print(f"\n{name}: lens {lens.tolist()}, max |out - oracle| = {diff:.3e}")
    assert diff <= parity.OUT_ATOL
    fin = np.isfinite(rlse)
    np.testing.assert_array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], rlse[fin], atol=1e-4, rtol=0)


def test_window_without_records_equals_verify_bit_for_bit():
    wl, Q, _, _, lens, _, _, _, _, _, _, q = _setup("g64_q3_sink128_recent100")
    # the same inputs laid out for S = R = 0
    case = W.make_dense(wl, device="cpu")
    N, D = wl.tile_tokens, wl.head_dim
    k, v = parity.f64(case.k), parity.f64(case.v)
    ends = [attention.verify_committed(int(L), Q, N) for L in lens]
    ppt = N // 16
    bt = np.full((wl.num_seqs, max(1, max(e // 16 for e in ends))), -1, np.int32)
    off = 0
    for b, e in enumerate(ends):
        bt[b, :e // 16] = np.arange(off, off + e // 16)
        off += e // 16
    lay = layout.DenseLayout(D, N)
    cache = np.zeros((max(1, off), wl.num_kv_heads, lay.page_bytes), np.uint8)
    for b, e in enumerate(ends):
        if e:
            attention.encode_into_cache(cache, lay, k[b:b + 1, :, :e], v[b:b + 1, :, :e], bt[b:b + 1], [0])
    cap = N + Q - 2
    tk = torch.zeros((wl.num_seqs, wl.num_kv_heads, cap, D), dtype=torch.float16)
    tv = torch.zeros_like(tk)
    for b, (L, e) in enumerate(zip(lens, ends)):
        tk[b, :, :L - e], tv[b, :, :L - e] = case.k[b, :, e:L], case.v[b, :, e:L]
    a, la = _run(wl, Q, 0, 0, lens, bt, cache, None, None, tk, tv, q, 0.1, window=True)
    b_, lb = _run(wl, Q, 0, 0, lens, bt, cache, None, None, tk, tv, q, 0.1, window=False)
    assert torch.equal(a, b_) and torch.equal(la, lb)
