"""Helpers of the GPU parity tests: run the oracle and the CUDA path on the
same seeded inputs and compare them element by element.

Tolerances (from the problem statement of this codec):
  * codes bit-exact, except elements whose quantiser input x = (z - lo)/delta
    lies within CODE_BAND of a rounding boundary, counted and reported. The
    CUDA path computes z in fp32 through the Hadamard butterflies and 2T
    normalisation passes, about twenty roundings of quantities up to a few
    times the row's std; with delta >= range/15 that moves x by at most
    ~2e-5 code units. CODE_BAND = 2^-13 (1.2e-4) leaves a 5x margin;
  * scales a, b, c to relative 1e-5 (b relative to the larger of |b| and
    the row range |a| (2^bits - 1), its natural scale); with fp16 scales in
    the page, one fp16 step (relative 2^-10): the GPU rounds its fp32 value,
    the oracle its float64 one, and the two may fall either side of a
    rounding point;
  * attention output to max abs 2e-3 (fp32 accumulation).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import attention, codec, layout, mla

CODE_BAND = 2.0 ** -13
SCALE_RTOL = 1e-5
OUT_ATOL = 2e-3


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def compare_tile(gpu: dict, ref: dict, bits: int, stats: dict, sb: int = 4):
    """gpu: codes/a/b/c read back from the GPU pages; ref: oracle encode_tile."""
    mism = gpu["codes"] != ref["codes"]
    if mism.any():
        x = ref["x"][mism]
        lo_code = np.minimum(gpu["codes"][mism], ref["codes"][mism])
        step = np.abs(gpu["codes"][mism] - ref["codes"][mism])
        dist = np.abs(x - (lo_code + 0.5))
        assert (step == 1).all(), "a code differs by more than one step"
        assert dist.max() <= CODE_BAND, f"code mismatch {dist.max():.3g} away from a boundary"
        ulp = np.spacing(np.float32(np.abs(x) + 0.5)).astype(np.float64)
        stats["within_1ulp"] += int((dist <= ulp).sum())
        stats["max_dist"] = max(stats["max_dist"], float(dist.max()))
    stats["mismatch"] += int(mism.sum())
    stats["codes"] += mism.size
    qmax = (1 << bits) - 1
    dt = np.float32 if sb == 4 else np.float16
    ref_a = ref["a"].astype(dt).astype(np.float64)
    for key in ("a", "b", "c"):
        g, r = gpu[key], ref[key].astype(dt).astype(np.float64)
        denom = np.abs(r)
        if key == "b":
            # the row offset lives on the row's quantisation grid: its scale is
            # the row range |a| (2^bits - 1), which also covers an offset that
            # is zero up to rounding (a constant row after rotation)
            denom = np.maximum(denom, np.abs(ref_a) * qmax)
        rel = np.abs(g - r) / np.maximum(denom, 1e-30)
        if sb == 2:
            rel = rel * SCALE_RTOL / 2.0 ** -10  # one fp16 step maps onto the fp32 tolerance
        stats["scale_rel"] = max(stats["scale_rel"], float(rel.max()))


def new_stats():
    return dict(mismatch=0, codes=0, within_1ulp=0, max_dist=0.0, scale_rel=0.0)


def check_dense_pages(cache_gpu: np.ndarray, k, v, bt, lens, N, D, heads=None, T=2, kb=4, vb=2, sb=4):
    """Compare every committed tile of the listed (b, kvh) pairs (all when
    None) of a GPU-written dense cache with the oracle's encoding of the same
    inputs. k, v: float64 [B, Hkv, L, D]."""
    lay = layout.DenseLayout(D, N, kb, vb, sb)
    B, Hkv = k.shape[:2]
    ppt = N // 16
    stats_k, stats_v = new_stats(), new_stats()
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hkv)]
    for b, h in pairs:
        for t in range(int(lens[b]) // N):
            pages = [int(bt[b][t * ppt + p]) for p in range(ppt)]
            gk, gv = layout.read_tile(cache_gpu, lay, pages, h)
            rk = codec.encode_tile(k[b, h, t * N:(t + 1) * N], kb, T)
            rv = codec.encode_tile(v[b, h, t * N:(t + 1) * N], vb, T)
            compare_tile(gk, rk, kb, stats_k, sb)
            compare_tile(gv, rv, vb, stats_v, sb)
    for st in (stats_k, stats_v):
        assert st["scale_rel"] <= SCALE_RTOL, st
        assert st["mismatch"] <= max(4, 1e-3 * st["codes"]), st
    return stats_k, stats_v


def oracle_dense_cache(k, v, bt, lens, N, D, num_pages, T=2, kb=4, vb=2, sb=4):
    lay = layout.DenseLayout(D, N, kb, vb, sb)
    B, Hkv = k.shape[:2]
    cache = np.zeros((num_pages, Hkv, lay.page_bytes), np.uint8)
    for b in range(B):
        tiles = int(lens[b]) // N
        if tiles:
            attention.encode_into_cache(cache, lay, k[b:b + 1, :, :tiles * N], v[b:b + 1, :, :tiles * N],
                                        bt[b:b + 1], [0], T=T)
    return cache


def tails(x: np.ndarray, lens, N):
    """Raw tail rows [B, H, N, D] (zeros past the tail)."""
    B, H, _, D = x.shape
    out = np.zeros((B, H, N, D), x.dtype)
    for b in range(B):
        c = (int(lens[b]) // N) * N
        out[b, :, :int(lens[b]) - c] = x[b, :, c:int(lens[b])]
    return out
