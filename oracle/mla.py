"""MLA latent cache: codec and decode, restated in float64 (test
infrastructure only).

KVarN review, paragraph on MLA: the compressed KV latent is quantised to int4.
Reading: the same four stages as the dense codec run on each 128-token tile of
the latent (width Dl), at 4 bits, and one code set serves as both key and
value; the rope part (width R) is stored fp16 untouched. A query head scores
token i as sm_scale * (q_latent . latent_i + q_rope . rope_i) and its output is
sum_i p_i latent_i (width Dl), the absorbed-MLA form.
"""
from __future__ import annotations

import numpy as np

from . import codec, layout


def write_tile(cache, lay: layout.LatentLayout, phys_pages, enc: dict, rope) -> None:
    """Store one encoded latent tile and its fp16 rope rows.
    cache: uint8 [num_pages, page_bytes]."""
    Dl, R, cpp = lay.D, lay.R, lay.col_per_page
    P = layout.P
    rope16 = np.asarray(rope, dtype=np.float16)
    for p, phys in enumerate(phys_pages):
        pg = cache[phys]
        rows = slice(p * P, (p + 1) * P)
        pg[lay.codes:lay.codes + 8 * Dl] = layout.pack_codes(enc["codes"][rows], "latent")
        pg[lay.rope:lay.rope + 2 * R * P] = np.ascontiguousarray(rope16[rows]).view(np.uint8).ravel()
        pg[lay.a:lay.a + 4 * P] = layout.f32_bytes(enc["a"][rows])
        pg[lay.b:lay.b + 4 * P] = layout.f32_bytes(enc["b"][rows])
        pg[lay.col:lay.col + 4 * cpp] = layout.f32_bytes(enc["c"][p * cpp:(p + 1) * cpp])


def read_tile(cache, lay: layout.LatentLayout, phys_pages):
    Dl, R, cpp = lay.D, lay.R, lay.col_per_page
    P = layout.P
    codes, a, b, c, rope = [], [], [], [], []
    for phys in phys_pages:
        pg = cache[phys]
        codes.append(layout.unpack_codes(pg[lay.codes:lay.codes + 8 * Dl], Dl, "latent"))
        rope.append(np.ascontiguousarray(pg[lay.rope:lay.rope + 2 * R * P]).view(np.float16)
                    .reshape(P, R).astype(np.float64))
        a.append(layout.f32_from(pg[lay.a:lay.a + 4 * P]))
        b.append(layout.f32_from(pg[lay.b:lay.b + 4 * P]))
        c.append(layout.f32_from(pg[lay.col:lay.col + 4 * cpp]))
    return (dict(codes=np.concatenate(codes), a=np.concatenate(a), b=np.concatenate(b),
                 c=np.concatenate(c)), np.concatenate(rope))


def encode_into_cache(cache, lay: layout.LatentLayout, latent, rope, block_table,
                      tile_start, bits=4, T=2):
    """latent [B, C, Dl], rope [B, C, R] of a chunk (C a multiple of N)."""
    latent = np.asarray(latent, np.float64)
    B, C, _ = latent.shape
    N = lay.N
    ppt = N // layout.P
    for b in range(B):
        for t in range(C // N):
            tile = int(tile_start[b]) + t
            pages = [int(block_table[b][tile * ppt + p]) for p in range(ppt)]
            enc = codec.encode_tile(latent[b, t * N:(t + 1) * N], bits, T)
            write_tile(cache, lay, pages, enc, np.asarray(rope[b, t * N:(t + 1) * N]))


def sequence_latent(cache, lay: layout.LatentLayout, bt_row, seq_len,
                    tail_latent=None, tail_rope=None):
    N = lay.N
    tiles = seq_len // N
    ppt = N // layout.P
    lat, rp = [], []
    for t in range(tiles):
        enc, rope = read_tile(cache, lay, [int(bt_row[t * ppt + p]) for p in range(ppt)])
        lat.append(codec.dequantize(enc["codes"], enc["a"], enc["b"], enc["c"]))
        rp.append(rope)
    tail = seq_len - tiles * N
    if tail:
        lat.append(np.asarray(tail_latent, np.float64)[:tail])
        rp.append(np.asarray(tail_rope, np.float64)[:tail])
    if not lat:
        return np.zeros((0, lay.D)), np.zeros((0, lay.R))
    return np.concatenate(lat), np.concatenate(rp)


def decode(q_latent, q_rope, cache, lay: layout.LatentLayout, block_table, seq_lens,
           sm_scale, tail_latent=None, tail_rope=None, heads=None):
    """Absorbed-MLA decode. Returns (out [B, H, Dl], lse [B, H])."""
    from .attention import softmax_attention
    ql = np.asarray(q_latent, np.float64)
    qr = np.asarray(q_rope, np.float64)
    B, H, Dl = ql.shape
    out = np.full((B, H, Dl), np.nan)
    lse = np.full((B, H), np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    seqs = {}
    for b, h in todo:
        if b not in seqs:
            tl = None if tail_latent is None else tail_latent[b]
            tr = None if tail_rope is None else tail_rope[b]
            seqs[b] = sequence_latent(cache, lay, block_table[b], int(seq_lens[b]), tl, tr)
        lat, rp = seqs[b]
        if lat.shape[0] == 0:
            out[b, h], lse[b, h] = 0.0, -np.inf
            continue
        K = np.concatenate([lat, rp], axis=1)
        qq = np.concatenate([ql[b, h], qr[b, h]])
        out[b, h], lse[b, h] = softmax_attention(qq, K, lat, sm_scale)
    return out, lse
