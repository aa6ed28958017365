"""The step (commit of a filled tile + decode) replays from a captured CUDA
graph: every launch takes its sizes and pointers from host arguments fixed
at capture, so a serving loop can capture it once and replay it with new
query values in the same buffers (turbo-attn page, "Decode": full CUDA-graph
capture with metadata prepared on the host)."""
import pytest
import torch

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_commit_and_decode_replay_bit_identical():
    from quantized_kv_cache_kvarn_gb300 import build
    build.build()
    dev = torch.device("cuda")
    wl = W.WORKLOADS["g64"].with_(num_seqs=3, num_q_heads=16, num_kv_heads=2, context=1000, min_context=200)
    case = W.make_dense(wl, device="cpu")
    N, D, B = wl.tile_tokens, wl.head_dim, wl.num_seqs
    lay = kv.dense_layout(D, N, wl.num_kv_heads, case.num_pages)
    lens = case.seq_lens.tolist()
    bt = case.block_table.to(dev)
    cache = kv.alloc_cache(lay, dev)
    err = kv.new_error_word(dev)
    z1 = torch.zeros(1, dtype=torch.int32, device=dev)
    for b, L in enumerate(lens):  # everything but each sequence's last full tile
        if L // N > 1:
            kv.encode_tiles(case.k[b:b + 1].to(dev), case.v[b:b + 1].to(dev), lay, z1, bt[b:b + 1], cache, err,
                            chunk_tokens=(L // N - 1) * N)
    ts = torch.tensor([L // N - 1 if L // N else -1 for L in lens], dtype=torch.int32, device=dev)
    ck = torch.stack([case.k[b, :, max(L // N - 1, 0) * N:max(L // N - 1, 0) * N + N] for b, L in enumerate(lens)])
    cv = torch.stack([case.v[b, :, max(L // N - 1, 0) * N:max(L // N - 1, 0) * N + N] for b, L in enumerate(lens)])
    ck, cv = ck.contiguous().to(dev), cv.contiguous().to(dev)
    tail_k = torch.zeros((B, wl.num_kv_heads, N, D), dtype=torch.float16, device=dev)
    tail_v = torch.zeros_like(tail_k)
    for b, L in enumerate(lens):
        c = (L // N) * N
        tail_k[b, :, :L - c] = case.k[b, :, c:L].to(dev)
        tail_v[b, :, :L - c] = case.v[b, :, c:L].to(dev)
    Lmax = max(lens)
    q = case.q.to(dev).clone()
    sl = case.seq_lens.to(dev)
    out = torch.empty((B, wl.num_q_heads, D), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, B, wl.num_q_heads, Lmax), dtype=torch.uint8, device=dev)
    sm = W.default_sm_scale(wl)

    def step():
        kv.encode_tiles(ck, cv, lay, ts, bt, cache, err, chunk_tokens=N)
        kv.decode(q, lay, cache, bt, sl, Lmax, out, ws, err, sm, tail_k, tail_v)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # eager, also settles the library's one-time launch set-up
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = out.clone()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)

    # new query values in the captured buffer
    q.copy_(torch.randn(q.shape, generator=torch.Generator().manual_seed(5)).to(q.dtype))
    g.replay()
    torch.cuda.synchronize()
    replayed = out.clone()
    step()
    torch.cuda.synchronize()
    assert torch.equal(replayed, out)
    assert not torch.equal(replayed, eager)
    assert kv.read_error_flags(err) == 0
