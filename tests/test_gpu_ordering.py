"""Stream ordering of the decode call. The decode kernel is launched as a
programmatic dependent of whatever kernel precedes it on the stream and waits
for that kernel's completion before its first global read; these tests issue
the kernels that write the decode's inputs (the commit of the pages, a copy
into the queries) immediately before it, with no synchronisation, and check
that the outputs equal those of a decode run after a full synchronisation,
bit for bit (the decode's schedule and reduction order depend only on the
shapes)."""
import pytest
import torch

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_kv_cache_kvarn_gb300 import build
    build.build()
    kv.lib()


def _setup():
    wl = W.WORKLOADS["dense32b"].with_(num_seqs=4, num_q_heads=16, num_kv_heads=2, context=4 * 128 + 40)
    case = W.make_dense(wl, device="cuda")
    lay = kv.dense_layout(wl.head_dim, wl.tile_tokens, wl.num_kv_heads, case.num_pages, kv.FP16, wl.norm_iters)
    N = wl.tile_tokens
    L = int(case.seq_lens.max())
    tail_k = torch.zeros((wl.num_seqs, wl.num_kv_heads, N, wl.head_dim), dtype=torch.float16, device="cuda")
    tail_v = torch.zeros_like(tail_k)
    for b in range(wl.num_seqs):
        Lb = int(case.seq_lens[b])
        c = (Lb // N) * N
        tail_k[b, :, :Lb - c] = case.k[b, :, c:Lb]
        tail_v[b, :, :Lb - c] = case.v[b, :, c:Lb]
    return wl, case, lay, L, tail_k, tail_v


def _encode_all(wl, case, lay, cache, err):
    tiles = int(case.seq_lens.min()) // wl.tile_tokens
    kv.encode_tiles(case.k, case.v, lay, torch.zeros(wl.num_seqs, dtype=torch.int32, device="cuda"),
                    case.block_table, cache, err, chunk_tokens=tiles * wl.tile_tokens)


def _decode(wl, case, lay, cache, L, tk, tv, q, err):
    out = torch.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
    ws = torch.empty(kv.decode_workspace_bytes(lay, wl.num_seqs, wl.num_q_heads, L), dtype=torch.uint8,
                     device="cuda")
    kv.decode(q, lay, cache, case.block_table, case.seq_lens, L, out, ws, err, W.default_sm_scale(wl), tk, tv)
    return out


def test_decode_right_after_the_commit_sees_its_pages():
    wl, case, lay, L, tk, tv = _setup()
    err = kv.new_error_word("cuda")
    ref_cache = kv.alloc_cache(lay, "cuda")
    _encode_all(wl, case, lay, ref_cache, err)
    torch.cuda.synchronize()
    ref = _decode(wl, case, lay, ref_cache, L, tk, tv, case.q, err)
    torch.cuda.synchronize()
    for _ in range(3):
        cache = torch.zeros_like(ref_cache)
        torch.cuda.synchronize()
        _encode_all(wl, case, lay, cache, err)  # no synchronisation between the two calls
        out = _decode(wl, case, lay, cache, L, tk, tv, case.q, err)
        torch.cuda.synchronize()
        assert kv.read_error_flags(err) == 0
        assert torch.equal(out, ref)


def test_decode_right_after_a_copy_into_its_queries():
    wl, case, lay, L, tk, tv = _setup()
    err = kv.new_error_word("cuda")
    cache = kv.alloc_cache(lay, "cuda")
    _encode_all(wl, case, lay, cache, err)
    q1 = torch.randn(case.q.shape, generator=torch.Generator("cuda").manual_seed(5), device="cuda").to(case.q.dtype)
    torch.cuda.synchronize()
    ref0 = _decode(wl, case, lay, cache, L, tk, tv, case.q, err)
    torch.cuda.synchronize()
    ref1 = _decode(wl, case, lay, cache, L, tk, tv, q1, err)
    torch.cuda.synchronize()
    assert not torch.equal(ref0, ref1)
    q = torch.zeros_like(case.q)
    outs = []
    for src in (q1, case.q, q1):
        q.copy_(src)  # the kernel right before the decode writes its queries
        outs.append(_decode(wl, case, lay, cache, L, tk, tv, q, err))
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    assert torch.equal(outs[0], ref1) and torch.equal(outs[1], ref0) and torch.equal(outs[2], ref1)
