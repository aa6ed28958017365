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


# --------------------------------------------------------------------------
# Affine pages, this library's format for the comparison decode (the page
# says only "N-bit codes plus an fp16 scale and offset per group"). One page
# holds P = 16 tokens of one KV head, in the original (unrotated) basis:
#   K part  K codes in the K plane placement of the kvarn page at k_bits
#           (layout.pack_planes(..., "k")), then per token t its G = D / 64
#           group scales and G group offsets as fp16: 4G bytes at
#           k_sc + 4G t (scale of group g at 2g, offset at 2G + 2g);
#           padded to 16 bytes
#   V part  the same with the V plane placement at v_bits.
# --------------------------------------------------------------------------
P = 16
GROUP = 64


class AffineLayout:
    def __init__(self, D: int, k_bits: int, v_bits: int, group: int = GROUP):
        from oracle import layout
        if k_bits not in layout.PLANES or v_bits not in layout.PLANES or D % group:
            raise ValueError("widths 2, 3, 4, 5, 6, 8; head_dim a multiple of the group")
        self.D, self.k_bits, self.v_bits, self.group = D, k_bits, v_bits, group
        self.G = D // group
        self.k_codes = 0
        self.k_sc = 2 * D * k_bits
        self.v_codes = _align16(self.k_sc + 4 * self.G * P)
        self.v_sc = self.v_codes + 2 * D * v_bits
        self.page_bytes = self.v_codes + _align16(2 * D * v_bits + 4 * self.G * P)


def _align16(x: int) -> int:
    return (x + 15) // 16 * 16


def _sc_bytes(scale, offset) -> np.ndarray:
    """[16, G] scales and offsets as the per-token fp16 records."""
    rec = np.concatenate([np.asarray(scale), np.asarray(offset)], axis=1)
    return rec.astype("<f2").view(np.uint8).ravel()


def write_tokens(cache, lay: AffineLayout, phys_pages, head: int, qk, qv) -> None:
    """Store quantised K and V rows (quantize() results, n*16 tokens) into
    the physical pages ``phys_pages`` of KV head ``head``; cache uint8
    [num_pages, Hkv, page_bytes]."""
    from oracle import layout
    D, G = lay.D, lay.G
    for p, phys in enumerate(phys_pages):
        pg = cache[phys, head]
        rows = slice(p * P, (p + 1) * P)
        pg[lay.k_codes:lay.k_codes + 2 * D * lay.k_bits] = layout.pack_planes(qk[0][rows], lay.k_bits, "k")
        pg[lay.v_codes:lay.v_codes + 2 * D * lay.v_bits] = layout.pack_planes(qv[0][rows], lay.v_bits, "v")
        pg[lay.k_sc:lay.k_sc + 4 * G * P] = _sc_bytes(qk[1][rows], qk[2][rows])
        pg[lay.v_sc:lay.v_sc + 4 * G * P] = _sc_bytes(qv[1][rows], qv[2][rows])


def read_tokens(cache, lay: AffineLayout, phys_pages, head: int):
    """Inverse of write_tokens: ((codes, scale, offset) of K, of V)."""
    from oracle import layout
    D, G = lay.D, lay.G
    out = []
    for side, base, sc, bits in (("k", lay.k_codes, lay.k_sc, lay.k_bits), ("v", lay.v_codes, lay.v_sc, lay.v_bits)):
        codes, scale, offset = [], [], []
        for phys in phys_pages:
            pg = cache[phys, head]
            codes.append(layout.unpack_planes(pg[base:base + 2 * D * bits], D, bits, side))
            rec = np.ascontiguousarray(pg[sc:sc + 4 * G * P]).view("<f2").astype(np.float64).reshape(P, 2 * G)
            scale.append(rec[:, :G])
            offset.append(rec[:, G:])
        out.append((np.concatenate(codes), np.concatenate(scale), np.concatenate(offset)))
    return out[0], out[1]


def encode_into_cache(cache, lay: AffineLayout, k, v, block_table, N: int, tile_start=None):
    """Quantise every whole tile of N tokens of k, v [B, Hkv, C, D] and store
    it (logical tile tile_start[b] + t of sequence b, default 0)."""
    k, v = np.asarray(k, np.float64), np.asarray(v, np.float64)
    B, Hkv, C, _ = k.shape
    ppt = N // P
    for b in range(B):
        t0 = 0 if tile_start is None else int(tile_start[b])
        for t in range(C // N):
            pages = [int(block_table[b][(t0 + t) * ppt + p]) for p in range(ppt)]
            for h in range(Hkv):
                rows = slice(t * N, (t + 1) * N)
                write_tokens(cache, lay, pages, h, quantize(k[b, h, rows], lay.k_bits, lay.group),
                             quantize(v[b, h, rows], lay.v_bits, lay.group))


def decode(q, cache, lay: AffineLayout, block_table, seq_lens, sm_scale, N: int, tail_k=None, tail_v=None):
    """Decode attention over an affine cache by its plain definition: the
    committed tiles [0, floor(L/N) N) dequantised from the pages, the tokens
    after them raw from the tail, then softmax attention (original basis).
    q [B, Hq, D]; returns (out [B, Hq, D], lse [B, Hq])."""
    from oracle import attention
    q = np.asarray(q, np.float64)
    B, Hq, D = q.shape
    Hkv = cache.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), -np.inf)
    ppt = N // P
    for b in range(B):
        L = int(seq_lens[b])
        C = (L // N) * N
        for h in range(Hkv):
            Ks, Vs = [], []
            for t in range(C // N):
                pages = [int(block_table[b][t * ppt + p]) for p in range(ppt)]
                qk, qv = read_tokens(cache, lay, pages, h)
                Ks.append(dequantize(*qk, group=lay.group))
                Vs.append(dequantize(*qv, group=lay.group))
            if L > C:
                Ks.append(np.asarray(tail_k[b, h, :L - C], np.float64))
                Vs.append(np.asarray(tail_v[b, h, :L - C], np.float64))
            if not Ks:
                continue
            K, V = np.concatenate(Ks), np.concatenate(Vs)
            for j in range(G):
                out[b, h * G + j], lse[b, h * G + j] = attention.softmax_attention(q[b, h * G + j], K, V, sm_scale)
    return out, lse
