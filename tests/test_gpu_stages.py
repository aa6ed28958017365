"""Staged parity of the encoder (the code contract: codes bit-exact except
within 1 fp32 ulp of a rounding boundary). The encoder exports its fp32
intermediates through kvarn_encode_tiles_staged; each stage of the KVarN
review's four-stage paragraph is checked on its own against the float64
oracle, and the round-to-nearest is checked on the GPU's own normalised
values, where the only freedom left is the rounding of one quotient. The
codes against the oracle's whole float64 chain are counted as well (the fp32
rotation and normalisation move a quantiser input by ~1e-5 code units, so a
few flips there are expected and reported, not the contract).
"""
import numpy as np
import pytest
import torch

import quantized_kv_cache_kvarn_gb300 as kv
from quantized_kv_cache_kvarn_gb300 import workloads as W
from oracle import layout
from tests import parity

pytestmark = pytest.mark.gpu

# (name, workload, overrides, k_bits, v_bits, fp16 scales)
CASES = [
    ("toy", "toy", {}, 4, 2, False),
    ("dense_small", "dense32b", dict(num_seqs=2, num_q_heads=16, num_kv_heads=2, context=1152), 4, 2, False),
    ("g64_small", "g64", dict(num_seqs=2, num_q_heads=16, num_kv_heads=2, context=640, min_context=640), 4, 2,
     False),
    ("hybrid_small", "hybrid", dict(num_seqs=1, num_q_heads=12, num_kv_heads=2, context=512), 4, 2, False),
    ("k8v8", "dense32b", dict(num_seqs=1, num_q_heads=8, num_kv_heads=2, context=384), 8, 8, True),
    ("k3v5_g64", "dense32b", dict(num_seqs=1, num_q_heads=8, num_kv_heads=2, context=256, tile_tokens=64), 3, 5,
     True),
    ("k6v2", "dense32b", dict(num_seqs=1, num_q_heads=8, num_kv_heads=2, context=384), 6, 2, True),
    ("d256_k5v5", "hybrid", dict(num_seqs=1, num_q_heads=12, num_kv_heads=2, context=256, k_bits=5, v_bits=5), 5,
     5, True),
]


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_kv_cache_kvarn_gb300 import build
    build.build()
    kv.lib()


def _run(wl, k, v, bt, kb, vb, fp16_scales, dev="cuda"):
    """Staged GPU encode of every whole tile of every sequence (one call,
    chunk = the shortest length's whole tiles)."""
    N, D = wl.tile_tokens, wl.head_dim
    B, Hkv, L = k.shape[:3]
    lay = kv.dense_layout(D, N, Hkv, int(bt.max()) + 1, kv.BF16 if wl.dtype == "bf16" else kv.FP16,
                          wl.norm_iters, k_bits=kb, v_bits=vb, fp16_scales=fp16_scales)
    C = (L // N) * N
    cache = kv.alloc_cache(lay, dev)
    stages = torch.full((kv.encode_stage_floats(lay, B, C),), float("nan"), dtype=torch.float32, device=dev)
    err = kv.new_error_word(dev)
    kv.encode_tiles_staged(k.to(dev), v.to(dev), lay, torch.zeros(B, dtype=torch.int32, device=dev), bt.to(dev),
                           cache, stages, err, chunk_tokens=C)
    torch.cuda.synchronize()
    assert kv.read_error_flags(err) == 0
    # the staged call writes the same pages as the plain one
    plain = kv.alloc_cache(lay, dev)
    kv.encode_tiles(k.to(dev), v.to(dev), lay, torch.zeros(B, dtype=torch.int32, device=dev), bt.to(dev), plain,
                    err, chunk_tokens=C)
    torch.cuda.synchronize()
    assert torch.equal(plain, cache)
    return cache.cpu().numpy(), stages.cpu().numpy(), C // N


def _check_all(name, wl, k, v, bt, kb, vb, fp16_scales):
    N, D = wl.tile_tokens, wl.head_dim
    cache, stages, tiles = _run(wl, k, v, bt, kb, vb, fp16_scales)
    sb = 2 if fp16_scales else 4
    olay = layout.DenseLayout(D, N, kb, vb, sb)
    R = 2 * N * D + 3 * N + D
    B, Hkv = k.shape[:2]
    ppt = N // 16
    kk, vv = parity.f64(k), parity.f64(v)
    stats = {"K": parity.new_stage_stats(), "V": parity.new_stage_stats()}
    for b in range(B):
        for h in range(Hkv):
            for u in range(tiles):
                pages = [int(bt[b, u * ppt + p]) for p in range(ppt)]
                gk, gv = layout.read_tile(cache, olay, pages, h)
                base = ((b * Hkv + h) * tiles + u) * 2 * R
                for side, got, x, bits, off in (("K", gk, kk, kb, 0), ("V", gv, vv, vb, R)):
                    rec = parity.stage_record(stages[base + off:base + off + R], N, D)
                    parity.check_stages(rec, got, x[b, h, u * N:(u + 1) * N], bits, wl.norm_iters, sb, stats[side])
    for side, st in stats.items():
        worst = max(st["max_rel"].values())
        parity.report(f"stages {name} {side}: {st['mismatch']} of {st['codes']} codes differ from the float64 "
                      f"rounding of the GPU's own (z - lo) / delta ({st['within_1ulp']} within 1 fp32 ulp of a "
                      f"boundary); end to end {st['e2e_flips']} flips (max {st['e2e_max_dist']:.2e} code units "
                      f"from a boundary); largest stage error {worst:.2e} "
                      f"({', '.join(f'{k_}={v_:.1e}' for k_, v_ in st['max_rel'].items())})")
        assert worst <= parity.STAGE_RTOL, (side, st)
        assert st["mismatch"] == st["within_1ulp"], (side, st)


@pytest.mark.parametrize("name,wname,over,kb,vb,fp16", CASES, ids=[c[0] for c in CASES])
def test_encode_stages_match_oracle(name, wname, over, kb, vb, fp16):
    wl = W.WORKLOADS[wname].with_(**over)
    case = W.make_dense(wl, device="cpu")
    _check_all(name, wl, case.k, case.v, case.block_table, kb, vb, fp16)


def test_degenerate_tiles_by_stage():
    """Constant, zero, equal-token and constant-channel tiles: a constant
    column or row (all entries equal) keeps sigma = 1 on both sides, a
    zero-range row gets delta = 0 and code 0."""
    wl = W.WORKLOADS["dense32b"].with_(num_seqs=1, num_q_heads=8, num_kv_heads=1, context=640)
    case = W.make_dense(wl, device="cpu")
    k, v = case.k.clone(), case.v.clone()
    k[0, 0, :128] = 3.0
    v[0, 0, :128] = 0.0
    k[0, 0, 128:256, 17] = -2.0
    v[0, 0, 256:384] = v[0, 0, 256:257]
    k[0, 0, 384:512] = k[0, 0, 384:385] * 0.5
    v[0, 0, 512:640, :64] = 1.0
    _check_all("degenerate", wl, k, v, case.block_table, 4, 2, False)
