"""kvarn_append (fused append + commit) against kvarn_encode_tiles, the raw
tokens and the oracle: sequences grow token by token; every tile a token
completes is encoded in the same launch, byte for byte as a separate encode
would, the partial tile stays raw in the tail, the pages agree with the
oracle's encoding of the same tokens, and a decode over the appended cache
and tail agrees with the oracle's decode."""
import numpy as np
import pytest
import torch

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import workloads as W
from oracle import attention, layout
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wname,D,N,dt", [("dense32b", 128, 128, torch.float16), ("g64", 128, 64, torch.float16),
                                          ("hybrid", 256, 128, torch.bfloat16)])
def test_token_by_token_appends_equal_bulk_encode(wname, D, N, dt):
    from quantized_kv_cache_kvarn_gb300 import build
    build.build()
    dev = "cuda"
    B, Hkv, L = 3, 2, 3 * N + 5
    wl = W.WORKLOADS[wname].with_(num_seqs=B, num_q_heads=2 * Hkv, num_kv_heads=Hkv, context=L, min_context=L)
    case = W.make_dense(wl, device=dev)
    k, v, bt = case.k, case.v, case.block_table
    lay = kv.dense_layout(D, N, Hkv, case.num_pages, kv.BF16 if dt == torch.bfloat16 else kv.FP16)
    start = [N - 3, 1, 2 * N - 1]  # tokens already present, at different phases of a tile
    # state before the appends: committed tiles through encode_tiles, partial tile in the tail
    cache = kv.alloc_cache(lay, dev)
    err = kv.new_error_word(dev)
    tail_k = torch.zeros((B, Hkv, N, D), dtype=dt, device=dev)
    tail_v = torch.zeros_like(tail_k)
    z1 = torch.zeros(1, dtype=torch.int32, device=dev)
    for b, s0 in enumerate(start):
        T = s0 // N
        if T:
            kv.encode_tiles(k[b:b + 1], v[b:b + 1], lay, z1, bt[b:b + 1], cache, err, chunk_tokens=T * N)
        tail_k[b, :, :s0 - T * N] = k[b, :, T * N:s0]
        tail_v[b, :, :s0 - T * N] = v[b, :, T * N:s0]
    lens = torch.tensor(start, dtype=torch.int32, device=dev)
    steps = L - min(start)
    for _ in range(steps):
        grow = lens < L
        new_lens = torch.where(grow, lens + 1, torch.zeros_like(lens))  # 0: nothing appended this step
        pos = (new_lens - 1).clamp(min=0).long()
        tok_k = k[torch.arange(B, device=dev), :, pos].contiguous()
        tok_v = v[torch.arange(B, device=dev), :, pos].contiguous()
        kv.append(tok_k, tok_v, new_lens, L, tail_k, tail_v, bt, lay, cache, err)
        lens = torch.where(grow, lens + 1, lens)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    assert lens.tolist() == [L] * B
    # reference: every full tile encoded in one bulk call
    ref = kv.alloc_cache(lay, dev)
    kv.encode_tiles(k, v, lay, torch.zeros(B, dtype=torch.int32, device=dev), bt, ref, err,
                    chunk_tokens=(L // N) * N)
    torch.cuda.synchronize()
    assert torch.equal(cache, ref)
    c = (L // N) * N
    assert torch.equal(tail_k[:, :, :L - c], k[:, :, c:L])
    assert torch.equal(tail_v[:, :, :L - c], v[:, :, c:L])

    # the oracle: its encoding of the same tokens, and its decode over that
    # cache plus the raw tail, against the GPU decode over the appended state
    kf, vf = parity.f64(k), parity.f64(v)
    lens_np = np.full(B, L, dtype=np.int32)
    st_k, st_v = parity.check_dense_pages(cache.cpu().numpy(), kf, vf, bt.cpu().numpy(), lens_np, N, D)
    parity.report(f"append {wname}: K codes {st_k['mismatch']}/{st_k['codes']} and V codes "
                  f"{st_v['mismatch']}/{st_v['codes']} differ from the oracle's float64 chain")
    ocache = parity.oracle_dense_cache(kf, vf, bt.cpu().numpy(), lens_np, N, D, case.num_pages)
    sm = W.default_sm_scale(wl)
    ref, ref_lse = attention.decode(parity.f64(case.q), ocache, layout.DenseLayout(D, N), bt.cpu().numpy(), lens_np,
                                    sm, parity.tails(kf, lens_np, N), parity.tails(vf, lens_np, N))
    out = torch.empty((B, 2 * Hkv, D), dtype=torch.float32, device=dev)
    lse = torch.empty((B, 2 * Hkv), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, B, 2 * Hkv, L), dtype=torch.uint8, device=dev)
    kv.decode(case.q, lay, cache, bt, lens, L, out, ws, err, sm, tail_k, tail_v, lse=lse)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    diff = np.abs(parity.f64(out) - ref).max()
    parity.report(f"append {wname}: decode after {steps} appends, max |out - oracle| = {diff:.3e}")
    assert diff <= parity.OUT_ATOL
    assert np.abs(parity.f64(lse) - ref_lse).max() <= 1e-4
