"""The decode kernel's bounded copy waits, driven on the GPU without making a
copy fail (kvarn_set_copy_wait_test): every copy is announced 16 bytes larger
than it is, so that no copy's phase completes, and the wait limit is short
(about half a millisecond). The kernel must flag KVARN_DEVERR_TIMEOUT, wait a
bounded time for the copies it started and return; the context stays usable
and the next call with the default settings is correct."""
import time

import numpy as np
import pytest
import torch

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import workloads as W
from oracle import attention, layout
from tests import parity

pytestmark = pytest.mark.gpu


def test_copy_wait_timeout_is_flagged_and_the_context_survives():
    from quantized_kv_cache_kvarn_gb300 import build
    build.build()
    dev = "cuda"
    wl = W.WORKLOADS["dense32b"].with_(num_seqs=8, num_q_heads=32, num_kv_heads=4, context=2048)
    case = W.make_dense(wl, device=dev)
    lay = kv.dense_layout(128, 128, 4, case.num_pages)
    cache = kv.alloc_cache(lay, dev)
    err = kv.new_error_word(dev)
    kv.encode_tiles(case.k, case.v, lay, torch.zeros(8, dtype=torch.int32, device=dev), case.block_table, cache, err)
    out = torch.empty((8, 32, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(kv.decode_workspace_bytes(lay, 8, 32, 2048), dtype=torch.uint8, device=dev)
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)  # 256 MB, more than the L2
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    kv.set_copy_wait_test(1_000_000, withhold=True)
    try:
        flush.fill_(1.0)
        err.zero_()
        t0 = time.perf_counter()
        kv.decode(case.q, lay, cache, case.block_table, case.seq_lens, 2048, out, ws, err, 0.088)
        torch.cuda.synchronize()
        took = time.perf_counter() - t0
        f = kv.read_error_flags(err)
    finally:
        kv.set_copy_wait_test(0, withhold=False)
    parity.report(f"copy-wait time-out: error word {f:#x} after {took * 1e3:.0f} ms (withheld copies)")
    assert f == kv.DEVERR_TIMEOUT
    # the default limit again: no flag, and the oracle's decode of the same pages
    err.zero_()
    kv.decode(case.q, lay, cache, case.block_table, case.seq_lens, 2048, out, ws, err, 0.088)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    rows = [(b, h) for b in (0, 5) for h in (0, 17, 31)]
    ref, _ = attention.decode(parity.f64(case.q), cache.cpu().numpy(), layout.DenseLayout(128, 128),
                              case.block_table.cpu().numpy(), case.seq_lens.cpu().numpy(), 0.088, heads=rows)
    o = parity.f64(out)
    assert max(np.abs(o[b, h] - ref[b, h]).max() for b, h in rows) <= parity.OUT_ATOL
