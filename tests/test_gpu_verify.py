"""GPU parity of the speculative-verification decode (several query tokens
per sequence, causal among themselves, tiles committed only once all their
tokens are accepted) against the oracle, through the C ABI, on pages the
oracle wrote."""
import numpy as np
import pytest
import torch

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import workloads as W
from oracle import attention, layout
from tests import parity

pytestmark = pytest.mark.gpu

CASES = {
    # name: (workload, overrides, Q[, (k_bits, v_bits, scale bytes)]). The
    # (head, query) rows of a KV head come in row groups of eight (the mma
    # row tile); the cases cover 1, 2, 3, 4 and 8 row groups, partial ones
    # included, and code widths other than the preset
    "g8_q4": ("dense32b", dict(num_seqs=2, num_q_heads=16, num_kv_heads=2, context=700), 4),
    "g2_q4_one_row_tile": ("dense32b", dict(num_seqs=2, num_q_heads=4, num_kv_heads=2, context=517), 4),
    "g64_q3_ragged": ("g64", dict(num_seqs=3, num_q_heads=16, num_kv_heads=2, context=640, min_context=1), 3),
    "hybrid_q2_bf16": ("hybrid", dict(num_seqs=2, num_q_heads=12, num_kv_heads=2, context=400), 2),
    "g8_q2": ("dense32b", dict(num_seqs=3, num_q_heads=16, num_kv_heads=2, context=900), 2),
    "g8_q8_two_blocks": ("dense32b", dict(num_seqs=2, num_q_heads=8, num_kv_heads=1, context=1000), 8),
    "g4_q5_idle_group": ("dense32b", dict(num_seqs=2, num_q_heads=8, num_kv_heads=2, context=650), 5),
    "k6v6_g8_q4": ("dense32b", dict(num_seqs=2, num_q_heads=16, num_kv_heads=2, context=700), 4, (6, 6, 2)),
    "k8v8_g8_q4_two_warps": ("dense32b", dict(num_seqs=2, num_q_heads=8, num_kv_heads=1, context=600), 4, (8, 8, 2)),
}


def _widths(name):
    c = CASES[name]
    return c[3] if len(c) > 3 else (4, 2, 4)


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_kv_cache_kvarn_gb300 import build
    build.build()
    kv.lib()


def _setup(name, lens_override=None):
    wname, over, Q = CASES[name][:3]
    wl = W.WORKLOADS[wname].with_(**over)
    case = W.make_dense(wl, device="cpu")
    lens = case.seq_lens.numpy().copy() if lens_override is None else np.array(lens_override, np.int32)
    N, D = wl.tile_tokens, wl.head_dim
    k, v = parity.f64(case.k), parity.f64(case.v)
    bt, num_pages = case.block_table.numpy(), case.num_pages
    if lens_override is not None:
        # pages for the committed tiles of the given lengths, placed in reverse
        per = [attention.verify_committed(int(L), Q, N) // 16 for L in lens]
        num_pages = max(1, sum(per))
        bt = np.full((len(lens), max(1, max(per))), -1, np.int32)
        order = np.arange(num_pages)[::-1]
        off = 0
        for b, n in enumerate(per):
            bt[b, :n] = order[off:off + n]
            off += n
    lay = layout.DenseLayout(D, N, *_widths(name))
    cache = np.zeros((num_pages, wl.num_kv_heads, lay.page_bytes), np.uint8)
    cap = N + Q - 2
    tk = np.zeros((wl.num_seqs, wl.num_kv_heads, cap, D))
    tv = np.zeros_like(tk)
    for b, L in enumerate(lens):
        C = attention.verify_committed(int(L), Q, N)
        if C:
            attention.encode_into_cache(cache, lay, k[b:b + 1, :, :C], v[b:b + 1, :, :C], bt[b:b + 1], [0])
        tk[b, :, :L - C] = k[b, :, C:L]
        tv[b, :, :L - C] = v[b, :, C:L]
    q = W.verify_queries(wl, Q)
    return wl, case, Q, lens, cache, tk, tv, q, bt


def _gpu(wl, case, Q, lens, cache, tk, tv, q, bt, widths=(4, 2, 4)):
    dev = "cuda"
    dt = W.TORCH_DTYPE[wl.dtype]
    lay = kv.dense_layout(wl.head_dim, wl.tile_tokens, wl.num_kv_heads, cache.shape[0],
                          kv.BF16 if wl.dtype == "bf16" else kv.FP16, k_bits=widths[0], v_bits=widths[1],
                          fp16_scales=widths[2] == 2)
    B, Hq, D = wl.num_seqs, wl.num_q_heads, wl.head_dim
    Lmax = int(lens.max())
    out = torch.empty((B, Q, Hq, D), dtype=torch.float32, device=dev)
    lse = torch.empty((B, Q, Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_verify_workspace_bytes(lay, B, Hq, Q, Lmax), dtype=torch.uint8, device=dev)
    err = kv.new_error_word(dev)
    kv.decode_verify(q.to(dev), lay, torch.from_numpy(cache).to(dev), torch.from_numpy(np.ascontiguousarray(bt)).to(dev),
                     torch.from_numpy(lens).to(dev), Lmax, out, ws, err, W.default_sm_scale(wl),
                     torch.from_numpy(tk).to(dt).to(dev), torch.from_numpy(tv).to(dt).to(dev), lse=lse)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    return parity.f64(out), parity.f64(lse)


@pytest.mark.parametrize("name", list(CASES))
def test_verify_matches_oracle(name):
    wl, case, Q, lens, cache, tk, tv, q, bt = _setup(name)
    dt = W.TORCH_DTYPE[wl.dtype]
    # the tail goes to the GPU in the storage dtype; the oracle reads the same values
    tk64 = torch.from_numpy(tk).to(dt).double().numpy()
    tv64 = torch.from_numpy(tv).to(dt).double().numpy()
    ref, rlse = attention.decode_verify(parity.f64(q), cache,
                                        layout.DenseLayout(wl.head_dim, wl.tile_tokens, *_widths(name)),
                                        bt, lens, W.default_sm_scale(wl), tk64, tv64)
    out, lse = _gpu(wl, case, Q, lens, cache, tk, tv, q, bt, _widths(name))
    diff = np.abs(out - ref).max()
    print(f"\n{name}: lens {lens.tolist()}, max |out - oracle| = {diff:.3e}, "
          f"max |lse - oracle| = {np.abs(lse - rlse).max():.3e}")
    assert diff <= parity.OUT_ATOL
    np.testing.assert_allclose(lse, rlse, atol=1e-4, rtol=0)


def test_verify_draft_tokens_fill_a_tile():
    """Lengths where the tokens under verification complete a tile (and one
    where the first query token sees nothing committed)."""
    N, Q = 64, 3
    lens = [2 * N + 1, 3 * N, 2]
    wl, case, Q, lens, cache, tk, tv, q, bt = _setup("g64_q3_ragged", lens_override=lens)
    tk64 = torch.from_numpy(tk).half().double().numpy()
    tv64 = torch.from_numpy(tv).half().double().numpy()
    ref, rlse = attention.decode_verify(parity.f64(q), cache, layout.DenseLayout(wl.head_dim, N),
                                        bt, lens, W.default_sm_scale(wl), tk64, tv64)
    out, lse = _gpu(wl, case, Q, lens, cache, tk, tv, q, bt)
    # sequence 2 (L = 2, Q = 3): query token 0 is token -1 and sees nothing
    assert (out[2, 0] == 0).all() and np.isneginf(lse[2, 0]).all()
    assert np.isfinite(lse[2, 1:]).all()
    assert np.abs(out - ref).max() <= parity.OUT_ATOL
    fin = np.isfinite(rlse)
    np.testing.assert_allclose(lse[fin], rlse[fin], atol=1e-4, rtol=0)


def test_verify_with_one_query_equals_decode_bit_for_bit():
    wl, case, _, lens, cache, tk, tv, _, _ = _setup("g8_q4")
    dev = "cuda"
    N, D, B, Hq = wl.tile_tokens, wl.head_dim, wl.num_seqs, wl.num_q_heads
    lay = kv.dense_layout(D, N, wl.num_kv_heads, case.num_pages)
    cache_d = torch.from_numpy(parity.oracle_dense_cache(parity.f64(case.k), parity.f64(case.v),
                                                         case.block_table.numpy(), lens, N, D,
                                                         case.num_pages)).to(dev)
    tail_k = torch.from_numpy(parity.tails(parity.f64(case.k), lens, N)).half().to(dev)
    tail_v = torch.from_numpy(parity.tails(parity.f64(case.v), lens, N)).half().to(dev)
    Lmax = int(lens.max())
    bt, sl = case.block_table.to(dev), torch.from_numpy(lens).to(dev)
    err = kv.new_error_word(dev)
    q = case.q.to(dev)
    o1 = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, B, Hq, Lmax), dtype=torch.uint8, device=dev)
    kv.decode(q, lay, cache_d, bt, sl, Lmax, o1, ws, err, 0.09, tail_k, tail_v)
    o2 = torch.empty((B, 1, Hq, D), dtype=torch.float32, device=dev)
    ws2 = torch.empty(kv.decode_verify_workspace_bytes(lay, B, Hq, 1, Lmax), dtype=torch.uint8, device=dev)
    kv.decode_verify(q[:, None], lay, cache_d, bt, sl, Lmax, o2, ws2, err, 0.09, tail_k, tail_v)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    assert torch.equal(o1, o2[:, 0])
