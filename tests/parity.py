"""Helpers of the GPU parity tests: run the oracle and the CUDA path on the
same seeded inputs and compare them element by element.

Tolerances (from the problem statement of this codec):
  * codes bit-exact, except elements within 1 fp32 ulp of a rounding
    boundary, counted and reported. This is enforced stage by stage
    (check_stages): the encoder's own fp32 intermediates are exported, each
    stage is compared with the float64 oracle at 1e-5, and the quantiser is
    checked on the GPU's own normalised values: its codes must equal the
    float64 round-half-to-even of (z - lo) / delta of those fp32 values,
    except within 1 fp32 ulp of a half-way point;
  * end to end (the GPU codes against the float64 oracle's own chain) the
    fp32 arithmetic of the rotation and the 2T normalisation passes moves the
    quantiser input by up to ~2e-5 code units, so a code may flip where the
    float64 input lies that close to a boundary. Those flips are counted and
    reported; as a sanity bound they must be single steps within CODE_BAND =
    2^-13 code units of a boundary. This band is not the contract; the
    staged check is;
  * scales a, b, c to relative 1e-5. b = r lo is measured against the scale
    of its row's values, max(|b|, |a| (2^bits - 1)) = r max(|lo|, hi - lo):
    lo is one of the normalised values of the row, whose fp32 rounding error
    is relative to the row's magnitude, not to |lo| (lo may lie near zero).
    With fp16 scales in the page, one fp16 step (relative 2^-10): the GPU
    rounds its fp32 value, the oracle its float64 one, and the two may fall
    either side of a rounding point;
  * attention output to max abs 2e-3 (fp32 accumulation).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import attention, codec, layout, mla

CODE_BAND = 2.0 ** -13
SCALE_RTOL = 1e-5
STAGE_RTOL = 1e-5
OUT_ATOL = 2e-3

# Count lines printed by the tests; tests/conftest.py repeats them in the
# terminal summary, so that they survive a run without -s.
REPORT: list = []


def report(line: str):
    print(line)
    REPORT.append(line)


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
            # b = r lo: lo is a value of the row, so its rounding error scales
            # with the row's magnitude r max(|lo|, hi - lo), not with |lo|
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


def new_stage_stats():
    return dict(codes=0, mismatch=0, within_1ulp=0, max_rel=dict(Y=0.0, Z=0.0, r=0.0, c=0.0, lo=0.0, delta=0.0),
                e2e_flips=0, e2e_max_dist=0.0)


def stage_record(rec: np.ndarray, N: int, D: int) -> dict:
    """Split one fp32 stage record (kvarn_encode_tiles_staged) into its parts."""
    o = 0
    out = {}
    for name, n, shape in (("Y", N * D, (N, D)), ("Z", N * D, (N, D)), ("r", N, (N,)), ("lo", N, (N,)),
                           ("delta", N, (N,)), ("c", D, (D,))):
        out[name] = rec[o:o + n].reshape(shape)
        o += n
    return out


def check_stages(rec: dict, gpu: dict, x: np.ndarray, bits: int, T: int, sb: int, stats: dict):
    """Staged parity of one tile. rec: the GPU's fp32 stage record
    (stage_record), gpu: codes / a / b / c read back from the GPU's pages,
    x: the input tile (float64 [N, D]).

    (i) every stage's fp32 values against the float64 oracle, each within
        STAGE_RTOL of the magnitude of its row (Y, Z, lo), or relative (r, c,
        delta);
    (ii) the quantiser and the fold on the GPU's own values: the codes are
        the float64 round-half-to-even of (Z - lo) / delta of the exported
        fp32 values, except within 1 fp32 ulp of a half-way point (counted);
        a, b, c in the page are the fp32 products r * delta, r * lo and the
        column scales (rounded to fp16 with fp16 scales), bit for bit;
    (iii) the codes against the oracle's own chain: flips counted (and
        bounded by compare_tile).
    """
    N, D = x.shape
    ref = codec.encode_tile(x, bits, T)
    f = lambda a: np.asarray(a, dtype=np.float64)
    mr = stats["max_rel"]
    for key in ("Y", "Z"):
        row = np.maximum(np.abs(ref[key]).max(axis=1, keepdims=True), 1e-30)
        mr[key] = max(mr[key], float((np.abs(f(rec[key]) - ref[key]) / row).max()))
    zrow = np.maximum(np.abs(ref["Z"]).max(axis=1), 1e-30)
    mr["lo"] = max(mr["lo"], float((np.abs(f(rec["lo"]) - ref["lo"]) / zrow).max()))
    mr["delta"] = max(mr["delta"], float((np.abs(f(rec["delta"]) - ref["delta"]) / zrow).max()))
    for key in ("r", "c"):
        mr[key] = max(mr[key], float((np.abs(f(rec[key]) - ref[key]) / np.abs(ref[key])).max()))
    # (ii) the quantiser on the GPU's own fp32 values
    qmax = (1 << bits) - 1
    z, lo, dl = f(rec["Z"]), f(rec["lo"])[:, None], f(rec["delta"])[:, None]
    xq = np.where(dl > 0, (z - lo) / np.where(dl > 0, dl, 1.0), 0.0)
    q = np.clip(np.rint(xq), 0, qmax).astype(np.int64)
    mism = gpu["codes"] != q
    stats["codes"] += mism.size
    if mism.any():
        xm = xq[mism]
        dist = np.abs(xm - (np.minimum(gpu["codes"][mism], q[mism]) + 0.5))
        ulp = np.spacing(np.float32(xm)).astype(np.float64)
        assert (np.abs(gpu["codes"][mism] - q[mism]) == 1).all(), "a code differs by more than one step"
        stats["within_1ulp"] += int((dist <= ulp).sum())
        stats["mismatch"] += int(mism.sum())
        assert (dist <= ulp).all(), f"code flipped {float((dist / ulp).max()):.3g} ulp from a boundary"
    r32, d32, lo32 = (np.asarray(rec[k], dtype=np.float32) for k in ("r", "delta", "lo"))
    dt = np.float32 if sb == 4 else np.float16
    np.testing.assert_array_equal(gpu["a"], (r32 * d32).astype(dt).astype(np.float64))
    np.testing.assert_array_equal(gpu["b"], (r32 * lo32).astype(dt).astype(np.float64))
    np.testing.assert_array_equal(gpu["c"], np.asarray(rec["c"], dtype=np.float32).astype(dt).astype(np.float64))
    # (iii) end to end against the float64 chain
    st = new_stats()
    compare_tile(gpu, ref, bits, st, sb)
    stats["e2e_flips"] += st["mismatch"]
    stats["e2e_max_dist"] = max(stats["e2e_max_dist"], st["max_dist"])
    assert st["scale_rel"] <= SCALE_RTOL, st
