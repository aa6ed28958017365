"""Decode attention over a KVarN-paged cache, restated in float64 (test
infrastructure only).

Plain definition, no split and no online softmax: dequantise every committed
tile back to the original channel basis, append the raw fp16 tail, take
scores s_i = sm_scale * q . k_i, subtract the maximum, exponentiate, normalise
and form o = sum_i p_i v_i. The library computes the same thing in the
rotated basis; that the two agree is the score-preservation property the
KVarN review (four-stage paragraph: "orthonormal, so attention scores are
preserved") and the turbo-attn page ("How it works": scores on rotated KV
equal scores on unrotated KV when the query is rotated by the same matrix)
rely on.

Commit rule (KVarN review, speculative-decoding paragraph: a block commits
only once all its tokens are accepted): tokens [0, floor(len/N)*N) are read
from the compressed pages; tokens [floor(len/N)*N, len) come from the fp16
tail buffer, in the original basis.
"""
from __future__ import annotations

import numpy as np

from . import codec, layout


def softmax_attention(q, K, V, sm_scale):
    """o = softmax(sm_scale q K^T) V and lse = log sum exp(sm_scale q K^T) for
    one query row q [D] over K [L, D], V [L, Dv]."""
    s = sm_scale * (np.asarray(K, np.float64) @ np.asarray(q, np.float64))
    m = s.max()
    e = np.exp(s - m)
    l = e.sum()
    return (e @ np.asarray(V, np.float64)) / l, m + np.log(l)


def sequence_kv(cache, lay: layout.DenseLayout, bt_row, seq_len, head,
                tail_k=None, tail_v=None):
    """Dequantised K, V [seq_len, D] of one sequence and KV head, in the
    original basis."""
    N = lay.N
    tiles = seq_len // N
    ppt = N // layout.P
    Ks, Vs = [], []
    for t in range(tiles):
        pages = [int(bt_row[t * ppt + p]) for p in range(ppt)]
        ek, ev = layout.read_tile(cache, lay, pages, head)
        Ks.append(codec.dequantize(ek["codes"], ek["a"], ek["b"], ek["c"]))
        Vs.append(codec.dequantize(ev["codes"], ev["a"], ev["b"], ev["c"]))
    tail = seq_len - tiles * N
    if tail:
        Ks.append(np.asarray(tail_k, np.float64)[:tail])
        Vs.append(np.asarray(tail_v, np.float64)[:tail])
    if not Ks:
        return np.zeros((0, lay.D)), np.zeros((0, lay.D))
    return np.concatenate(Ks), np.concatenate(Vs)


def decode(q, cache, lay: layout.DenseLayout, block_table, seq_lens, sm_scale,
           tail_k=None, tail_v=None, heads=None):
    """Decode attention for every (sequence, query head), or for the listed
    ``heads`` = [(b, h), ...] only.

    q           [B, Hq, D]      cache  uint8 [num_pages, Hkv, page_bytes]
    block_table [B, max_pages]  seq_lens [B]
    tail_k/v    [B, Hkv, N, D]  raw tail tokens (positions 0..len%N-1)
    Returns (out [B, Hq, D], lse [B, Hq]); unlisted entries are NaN. A
    sequence of length 0 gives out = 0 and lse = -inf.
    """
    q = np.asarray(q, np.float64)
    B, Hq, D = q.shape
    Hkv = cache.shape[1]
    G = Hq // Hkv
    out = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    kv_cache = {}
    for b, h in todo:
        kvh = h // G
        key = (b, kvh)
        if key not in kv_cache:
            tk = None if tail_k is None else tail_k[b, kvh]
            tv = None if tail_v is None else tail_v[b, kvh]
            kv_cache[key] = sequence_kv(cache, lay, block_table[b], int(seq_lens[b]), kvh, tk, tv)
        K, V = kv_cache[key]
        if K.shape[0] == 0:
            out[b, h], lse[b, h] = 0.0, -np.inf
            continue
        out[b, h], lse[b, h] = softmax_attention(q[b, h], K, V, sm_scale)
    return out, lse


def verify_committed(L: int, Q: int, N: int) -> int:
    """Committed tokens of a sequence of L tokens whose last Q are under
    verification: the whole tiles of the accepted tokens [0, L - Q + 1)."""
    return (max(0, L - Q + 1) // N) * N


def verify_visible(L: int, Q: int, j: int) -> int:
    """Tokens seen by query token j (token L - Q + j): [0, L - Q + 1 + j)."""
    return max(0, L - Q + 1 + j)


def decode_verify(q, cache, lay: layout.DenseLayout, block_table, seq_lens, sm_scale,
                  tail_k=None, tail_v=None, rows=None):
    """Speculative verification: Q query tokens per sequence, causal among
    themselves (gmlx page, "Speed and speculative decoding": a batch
    verifies several tokens per row; KVarN review, speculative-decoding
    paragraph: a block commits only once all its tokens are accepted).

    Sequence b holds L = seq_lens[b] tokens, the last Q under verification;
    query token j is token L - Q + j and attends to tokens [0, L - Q + 1 + j).
    The accepted tokens [0, L - Q + 1) fill the committed tiles
    [0, C), C = floor((L - Q + 1) / N) * N, read from the pages; tokens
    [C, L) are rows 0.. of the raw tail buffer.

    q [B, Q, Hq, D]; tail_k/v [B, Hkv, capacity, D]; rows = [(b, j, h), ...]
    or None for all. Returns (out [B, Q, Hq, D], lse [B, Q, Hq]); a query that
    sees no token gives out = 0 and lse = -inf, unlisted rows NaN.
    """
    q = np.asarray(q, np.float64)
    B, Q, Hq, D = q.shape
    Hkv = cache.shape[1]
    G = Hq // Hkv
    N = lay.N
    out = np.full((B, Q, Hq, D), np.nan)
    lse = np.full((B, Q, Hq), np.nan)
    todo = rows if rows is not None else [(b, j, h) for b in range(B) for j in range(Q) for h in range(Hq)]
    kv_cache = {}
    for b, j, h in todo:
        L = int(seq_lens[b])
        kvh = h // G
        key = (b, kvh)
        if key not in kv_cache:
            C = verify_committed(L, Q, N)
            K, V = sequence_kv(cache, lay, block_table[b], C, kvh)
            if L > C:
                K = np.concatenate([K, np.asarray(tail_k[b, kvh], np.float64)[:L - C]])
                V = np.concatenate([V, np.asarray(tail_v[b, kvh], np.float64)[:L - C]])
            kv_cache[key] = (K, V)
        K, V = kv_cache[key]
        vis = verify_visible(L, Q, j)
        if vis == 0:
            out[b, j, h], lse[b, j, h] = 0.0, -np.inf
            continue
        out[b, j, h], lse[b, j, h] = softmax_attention(q[b, j, h], K[:vis], V[:vis], sm_scale)
    return out, lse


def window_committed(L: int, Q: int, N: int, sink: int, recent: int) -> int:
    """End of the compressed tiles under the raw-record policy of the gmlx
    page ("The two schemes": the first tokens and the newest tokens stay
    fp16): tiles start after the `sink` raw tokens and end before the newest
    `recent` accepted tokens, in whole tiles; never before the sink."""
    return max(sink, (max(0, L - Q + 1 - recent) // N) * N)


def decode_window(q, cache, lay: layout.DenseLayout, block_table, seq_lens, sm_scale, sink, recent,
                  sink_k=None, sink_v=None, tail_k=None, tail_v=None, rows=None):
    """Verification decode (decode_verify) with raw sink and recent records.

    Sequence b of L tokens, the last Q under verification: tokens
    [0, min(sink, L)) are rows of the raw sink buffer, the whole tiles
    [sink, C), C = window_committed(L, Q, N, sink, recent), come from the
    pages (logical tile t holds tokens [tN, tN + N)), and tokens [C, L) are
    rows 0.. of the raw tail buffer. Query token j sees [0, L - Q + 1 + j).

    sink_k/v [B, Hkv, sink, D]; tail_k/v [B, Hkv, capacity, D]. Returns
    (out [B, Q, Hq, D], lse [B, Q, Hq]).
    """
    q = np.asarray(q, np.float64)
    B, Q, Hq, D = q.shape
    Hkv = cache.shape[1]
    G = Hq // Hkv
    N = lay.N
    ppt = N // layout.P
    out = np.full((B, Q, Hq, D), np.nan)
    lse = np.full((B, Q, Hq), np.nan)
    todo = rows if rows is not None else [(b, j, h) for b in range(B) for j in range(Q) for h in range(Hq)]
    kv_cache = {}
    for b, j, h in todo:
        L = int(seq_lens[b])
        kvh = h // G
        key = (b, kvh)
        if key not in kv_cache:
            C = window_committed(L, Q, N, sink, recent)
            Ks, Vs = [], []
            if min(sink, L):
                Ks.append(np.asarray(sink_k[b, kvh], np.float64)[:min(sink, L)])
                Vs.append(np.asarray(sink_v[b, kvh], np.float64)[:min(sink, L)])
            for t in range(sink // N, C // N):
                pages = [int(block_table[b][t * ppt + p]) for p in range(ppt)]
                ek, ev = layout.read_tile(cache, lay, pages, kvh)
                Ks.append(codec.dequantize(ek["codes"], ek["a"], ek["b"], ek["c"]))
                Vs.append(codec.dequantize(ev["codes"], ev["a"], ev["b"], ev["c"]))
            if L > C:
                Ks.append(np.asarray(tail_k[b, kvh], np.float64)[:L - C])
                Vs.append(np.asarray(tail_v[b, kvh], np.float64)[:L - C])
            kv_cache[key] = (np.concatenate(Ks) if Ks else np.zeros((0, D)),
                             np.concatenate(Vs) if Vs else np.zeros((0, D)))
        K, V = kv_cache[key]
        vis = verify_visible(L, Q, j)
        if vis == 0:
            out[b, j, h], lse[b, j, h] = 0.0, -np.inf
            continue
        out[b, j, h], lse[b, j, h] = softmax_attention(q[b, j, h], K[:vis], V[:vis], sm_scale)
    return out, lse


def encode_into_cache(cache, lay: layout.DenseLayout, k, v, block_table, tile_start,
                      bits=None, T=2):
    """Encode every full tile of a chunk and store it.

    k, v [B, Hkv, C, D] values of the chunk (C a multiple of N); tile_start[b]
    is the logical tile index of the chunk's first token in sequence b.
    """
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B, Hkv, C, D = k.shape
    N = lay.N
    bits = (lay.k_bits, lay.v_bits) if bits is None else bits
    ppt = N // layout.P
    for b in range(B):
        for t in range(C // N):
            tile = int(tile_start[b]) + t
            pages = [int(block_table[b][tile * ppt + p]) for p in range(ppt)]
            for h in range(Hkv):
                ek = codec.encode_tile(k[b, h, t * N:(t + 1) * N], bits[0], T)
                ev = codec.encode_tile(v[b, h, t * N:(t + 1) * N], bits[1], T)
                layout.write_tile(cache, lay, pages, h, ek, ev)


def decode_fp16(q, k_cache, v_cache, block_table, seq_lens, sm_scale, heads=None):
    """Plain attention over an uncompressed paged cache (the bypass baseline
    built on the same skeleton): k_cache, v_cache [num_pages, Hkv, P, D]."""
    q = np.asarray(q, np.float64)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    P = k_cache.shape[2]
    out = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in todo:
        L = int(seq_lens[b])
        kvh = h // G
        npg = -(-L // P)
        pages = [int(block_table[b][i]) for i in range(npg)]
        K = np.concatenate([np.asarray(k_cache[p, kvh], np.float64) for p in pages])[:L] if L else None
        V = np.concatenate([np.asarray(v_cache[p, kvh], np.float64) for p in pages])[:L] if L else None
        if not L:
            out[b, h], lse[b, h] = 0.0, -np.inf
            continue
        out[b, h], lse[b, h] = softmax_attention(q[b, h], K, V, sm_scale)
    return out, lse
