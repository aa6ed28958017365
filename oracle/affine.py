"""Affine per-token group quantisation, the comparison scheme of the gmlx
page ("The two schemes": mlx-lm's quantized KV cache splits each token's K
and V rows into groups of 64 values and stores N-bit codes with an fp16
scale and offset per group). Test infrastructure only; shares no code with
the CUDA path.

Reading where the page is silent: per group, offset = min and scale =
(max - min) / (2^bits - 1), both rounded to fp16 as stored; codes are
round-half-to-even of (x - offset) / scale with the stored values, clamped
to [0, 2^bits - 1]; a constant group (scale 0) gets code 0.
"""
from __future__ import annotations

import numpy as np


def quantize(x, bits: int, group: int = 64):
    """x [L, D] -> (codes [L, D], scale [L, D/group], offset [L, D/group])."""
    x = np.asarray(x, np.float64)
    L, D = x.shape
    xg = x.reshape(L, D // group, group)
    lo, hi = xg.min(-1), xg.max(-1)
    scale = ((hi - lo) / (2 ** bits - 1)).astype(np.float16).astype(np.float64)
    offset = lo.astype(np.float16).astype(np.float64)
    safe = np.where(scale > 0, scale, 1.0)
    codes = np.clip(np.rint((xg - offset[..., None]) / safe[..., None]), 0, 2 ** bits - 1)
    codes = np.where(scale[..., None] > 0, codes, 0).astype(np.int64)
    return codes.reshape(L, D), scale, offset


def dequantize(codes, scale, offset, group: int = 64):
    L, D = codes.shape
    cg = np.asarray(codes, np.float64).reshape(L, D // group, group)
    return (cg * scale[..., None] + offset[..., None]).reshape(L, D)
