"""Pins of the oracle's decode attention: library softmax, closed forms,
the rotated-query identity, the commit rule and block-table invariance."""
import numpy as np
import pytest
import scipy.special

from oracle import attention, codec, layout, mla


def test_softmax_attention_matches_scipy():
    rng = np.random.default_rng(0)
    q, K, V = rng.standard_normal(64), rng.standard_normal((50, 64)) * 3, rng.standard_normal((50, 32))
    o, lse = attention.softmax_attention(q, K, V, 0.125)
    s = 0.125 * K @ q
    np.testing.assert_allclose(o, scipy.special.softmax(s) @ V, rtol=1e-12)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(s), rtol=1e-14)


def test_softmax_attention_two_tokens_by_hand():
    """Scores 0 and log 3 give weights 1/4 and 3/4."""
    q = np.array([1.0, 0.0])
    K = np.array([[0.0, 5.0], [np.log(3), -2.0]])
    V = np.array([[4.0, 0.0], [0.0, 8.0]])
    o, lse = attention.softmax_attention(q, K, V, 1.0)
    np.testing.assert_allclose(o, [1.0, 6.0], rtol=1e-14)
    np.testing.assert_allclose(lse, np.log(4.0), rtol=1e-14)


def _case(B=2, Hkv=2, G=3, D=128, N=128, lens=(256, 300), seed=0):
    rng = np.random.default_rng(seed)
    lay = layout.DenseLayout(D, N)
    Lmax = max(lens)
    k = rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float16).astype(np.float64)
    v = rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float16).astype(np.float64)
    k[..., 5] *= 20
    v[..., 77] *= 20
    q = rng.standard_normal((B, Hkv * G, D)).astype(np.float16).astype(np.float64)
    ppt = N // 16
    tiles = [L // N for L in lens]
    num_pages = sum(tiles) * ppt + 3
    perm = rng.permutation(num_pages)
    bt = np.full((B, Lmax // 16 + 1), -1)
    off = 0
    for b in range(B):
        n = tiles[b] * ppt
        bt[b, :n] = perm[off:off + n]
        off += n
    cache = np.zeros((num_pages, Hkv, lay.page_bytes), np.uint8)
    for b in range(B):
        attention.encode_into_cache(cache, lay, k[b:b + 1, :, :tiles[b] * N], v[b:b + 1, :, :tiles[b] * N],
                                    bt[b:b + 1], [0])
    tail_k = np.full((B, Hkv, N, D), np.nan)
    tail_v = np.full((B, Hkv, N, D), np.nan)
    for b, L in enumerate(lens):
        t = L - tiles[b] * N
        tail_k[b, :, :t] = k[b, :, tiles[b] * N:L]
        tail_v[b, :, :t] = v[b, :, tiles[b] * N:L]
    return dict(lay=lay, k=k, v=v, q=q, bt=bt, cache=cache, lens=np.array(lens),
                tail_k=tail_k, tail_v=tail_v, G=G)


def test_decode_equals_rotated_space_computation():
    """The library's rotated-basis formulation (q' = qH scored against the
    rotated dequantised keys, output un-rotated once at the end) equals the
    oracle's plain definition in the original basis."""
    c = _case()
    lay, D = c["lay"], 128
    sm = 1 / np.sqrt(D)
    out, lse = attention.decode(c["q"], c["cache"], lay, c["bt"], c["lens"], sm, c["tail_k"], c["tail_v"])
    H = codec.hadamard(D)
    for b in range(2):
        L = c["lens"][b]
        T = L // 128
        for h in range(6):
            kvh = h // c["G"]
            Kr, Vr = [], []
            for t in range(T):
                pages = [int(c["bt"][b, t * 8 + p]) for p in range(8)]
                ek, ev = layout.read_tile(c["cache"], lay, pages, kvh)
                Kr.append(codec.dequantize_rotated(ek["codes"], ek["a"], ek["b"], ek["c"]))
                Vr.append(codec.dequantize_rotated(ev["codes"], ev["a"], ev["b"], ev["c"]))
            Kr, Vr = np.concatenate(Kr), np.concatenate(Vr)
            qr = c["q"][b, h] @ H
            s = sm * np.concatenate([Kr @ qr, c["tail_k"][b, kvh, :L - T * 128] @ c["q"][b, h]])
            p = scipy.special.softmax(s)
            o = (p[:T * 128] @ Vr) @ H + p[T * 128:] @ c["tail_v"][b, kvh, :L - T * 128]
            np.testing.assert_allclose(out[b, h], o, rtol=1e-10, atol=1e-10)
            np.testing.assert_allclose(lse[b, h], scipy.special.logsumexp(s), rtol=1e-12)


def test_tail_only_sequence_is_plain_attention():
    """len < N: nothing is committed, the fp16 tail is read as is."""
    c = _case(lens=(100, 5))
    out, _ = attention.decode(c["q"], c["cache"], c["lay"], c["bt"], c["lens"], 0.1, c["tail_k"], c["tail_v"])
    for b, L in enumerate((100, 5)):
        for h in range(6):
            s = 0.1 * c["k"][b, h // 3, :L] @ c["q"][b, h]
            np.testing.assert_allclose(out[b, h], scipy.special.softmax(s) @ c["v"][b, h // 3, :L], rtol=1e-12, atol=1e-14)


def test_full_tiles_never_read_the_tail():
    """len a multiple of N: the tail buffer (all NaN here) is not touched."""
    c = _case(lens=(256, 128))
    out, lse = attention.decode(c["q"], c["cache"], c["lay"], c["bt"], c["lens"], 0.1, c["tail_k"], c["tail_v"])
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_block_table_permutation_invariance():
    """Moving pages to other physical slots (and the table with them) changes
    nothing."""
    c = _case(lens=(256, 384), seed=3)
    out1, _ = attention.decode(c["q"], c["cache"], c["lay"], c["bt"], c["lens"], 0.1, c["tail_k"], c["tail_v"])
    rng = np.random.default_rng(9)
    perm = rng.permutation(c["cache"].shape[0])
    cache2 = np.empty_like(c["cache"])
    cache2[perm] = c["cache"]
    bt2 = np.where(c["bt"] >= 0, perm[np.maximum(c["bt"], 0)], -1)
    out2, _ = attention.decode(c["q"], cache2, c["lay"], bt2, c["lens"], 0.1, c["tail_k"], c["tail_v"])
    np.testing.assert_array_equal(out1, out2)


def test_k4v2_decode_beats_plain_rtn():
    """At the k4v2 widths, decode over the KVarN cache is closer to exact
    attention on the raw tokens than decode over a plain per-token RTN cache
    with the same widths, on tiles with outlier channels (KVarN review:
    rotation spreads outliers, normalisation keeps any token or channel from
    dominating). On uncorrelated synthetic V a 2-bit cache cannot be close in
    absolute terms, so the comparison is relative."""
    c = _case(lens=(1024, 1024), seed=5)
    sm = 1 / np.sqrt(128)
    out, _ = attention.decode(c["q"], c["cache"], c["lay"], c["bt"], c["lens"], sm)
    err_kvarn, err_plain = [], []
    for b in range(2):
        for h in range(6):
            K, V = c["k"][b, h // 3], c["v"][b, h // 3]
            o, _ = attention.softmax_attention(c["q"][b, h], K, V, sm)
            Kp = np.concatenate([codec.rtn_plain_rows(K[i:i + 128], 4) for i in range(0, 1024, 128)])
            Vp = np.concatenate([codec.rtn_plain_rows(V[i:i + 128], 2) for i in range(0, 1024, 128)])
            op, _ = attention.softmax_attention(c["q"][b, h], Kp, Vp, sm)
            err_kvarn.append(np.linalg.norm(out[b, h] - o))
            err_plain.append(np.linalg.norm(op - o))
    assert np.mean(err_kvarn) < 0.5 * np.mean(err_plain), (err_kvarn, err_plain)


def test_empty_sequence():
    c = _case(lens=(0, 128))
    out, lse = attention.decode(c["q"], c["cache"], c["lay"], c["bt"], c["lens"], 0.1)
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()


def test_decode_fp16_is_plain_attention():
    rng = np.random.default_rng(1)
    kc = rng.standard_normal((6, 2, 16, 32))
    vc = rng.standard_normal((6, 2, 16, 32))
    q = rng.standard_normal((1, 4, 32))
    bt = np.array([[4, 1, 5]])
    out, _ = attention.decode_fp16(q, kc, vc, bt, [40], 0.2)
    K = np.concatenate([kc[4, 1], kc[1, 1], kc[5, 1]])[:40]
    V = np.concatenate([vc[4, 1], vc[1, 1], vc[5, 1]])[:40]
    np.testing.assert_allclose(out[0, 3], scipy.special.softmax(0.2 * K @ q[0, 3]) @ V, rtol=1e-12, atol=1e-14)


def test_mla_decode_rope_and_shared_latent():
    """MLA: the score adds the rope dot product to the latent one, and the
    value is the (dequantised) latent itself."""
    rng = np.random.default_rng(2)
    lay = layout.LatentLayout(512, 64, 128)
    L = 128 + 20
    lat = rng.standard_normal((1, L, 512)).astype(np.float16).astype(np.float64)
    rope = rng.standard_normal((1, L, 64)).astype(np.float16).astype(np.float64)
    cache = np.zeros((8, lay.page_bytes), np.uint8)
    bt = np.array([[3, 0, 7, 1, 6, 2, 5, 4]])
    mla.encode_into_cache(cache, lay, lat[:, :128], rope[:, :128], bt, [0])
    tail_lat = np.zeros((1, 128, 512))
    tail_rope = np.zeros((1, 128, 64))
    tail_lat[0, :20] = lat[0, 128:]
    tail_rope[0, :20] = rope[0, 128:]
    ql = rng.standard_normal((1, 3, 512))
    qr = rng.standard_normal((1, 3, 64))
    sm = 1 / np.sqrt(576)
    out, lse = mla.decode(ql, qr, cache, lay, bt, [L], sm, tail_lat, tail_rope)
    enc, rope_rd = mla.read_tile(cache, lay, list(bt[0]))
    np.testing.assert_array_equal(rope_rd, rope[0, :128])   # rope stays fp16
    latent_hat = np.concatenate([codec.dequantize(enc["codes"], enc["a"], enc["b"], enc["c"]), lat[0, 128:]])
    K = np.concatenate([latent_hat, rope[0]], 1)
    for h in range(3):
        s = sm * K @ np.concatenate([ql[0, h], qr[0, h]])
        np.testing.assert_allclose(out[0, h], scipy.special.softmax(s) @ latent_hat, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse[0, h], scipy.special.logsumexp(s), rtol=1e-12)


# ---------------------------------------------------------------- verify
def _verify_case(lens, Q, B=None, Hkv=2, G=2, D=128, N=64, seed=3):
    """Cache with the accepted tiles committed and the rest in a raw tail of
    N + Q - 2 rows, built from the commit rule's definition."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    lay = layout.DenseLayout(D, N)
    Lmax = max(lens)
    k = rng.standard_normal((B, Hkv, Lmax, D))
    v = rng.standard_normal((B, Hkv, Lmax, D))
    k[..., 9] *= 15
    q = rng.standard_normal((B, Q, Hkv * G, D))
    ppt = N // 16
    C = [(max(0, L - Q + 1) // N) * N for L in lens]
    num_pages = sum(c // N for c in C) * ppt + 2
    bt = np.full((B, Lmax // 16 + 2), -1)
    off = 0
    for b in range(B):
        n = C[b] // N * ppt
        bt[b, :n] = np.arange(off, off + n)[::-1]
        off += n
    cache = np.zeros((num_pages, Hkv, lay.page_bytes), np.uint8)
    for b in range(B):
        if C[b]:
            attention.encode_into_cache(cache, lay, k[b:b + 1, :, :C[b]], v[b:b + 1, :, :C[b]], bt[b:b + 1], [0])
    cap = N + Q - 2
    tk = np.full((B, Hkv, cap, D), np.nan)
    tv = np.full((B, Hkv, cap, D), np.nan)
    for b, L in enumerate(lens):
        tk[b, :, :L - C[b]] = k[b, :, C[b]:L]
        tv[b, :, :L - C[b]] = v[b, :, C[b]:L]
    return dict(lay=lay, k=k, v=v, q=q, bt=bt, cache=cache, lens=np.array(lens), tk=tk, tv=tv, C=C, G=G)


def test_verify_with_one_query_is_decode():
    c = _verify_case([200, 64, 130], Q=1)
    out, lse = attention.decode_verify(c["q"], c["cache"], c["lay"], c["bt"], c["lens"], 0.1, c["tk"], c["tv"])
    ref, rlse = attention.decode(c["q"][:, 0], c["cache"], c["lay"], c["bt"], c["lens"], 0.1,
                                 c["tk"][:, :, :64], c["tv"][:, :, :64])
    np.testing.assert_array_equal(out[:, 0], ref)
    np.testing.assert_array_equal(lse[:, 0], rlse)


def test_verify_without_committed_tiles_is_causal_softmax():
    """Nothing committed (L - Q + 1 < N): query j is plain softmax attention
    over the raw tokens 0 .. L - Q + j, by scipy."""
    L, Q = 40, 4
    c = _verify_case([L], Q)
    assert c["C"] == [0]
    out, lse = attention.decode_verify(c["q"], c["cache"], c["lay"], c["bt"], c["lens"], 0.07, c["tk"], c["tv"])
    for j in range(Q):
        for h in range(4):
            K, V = c["k"][0, h // 2, :L - Q + 1 + j], c["v"][0, h // 2, :L - Q + 1 + j]
            s = 0.07 * K @ c["q"][0, j, h]
            np.testing.assert_allclose(out[0, j, h], scipy.special.softmax(s) @ V, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(lse[0, j, h], scipy.special.logsumexp(s), rtol=1e-12)


def test_verify_is_causal():
    """Changing the last token under verification changes only the last
    query token's output."""
    L, Q = 150, 3
    c = _verify_case([L], Q)
    a, _ = attention.decode_verify(c["q"], c["cache"], c["lay"], c["bt"], c["lens"], 0.1, c["tk"], c["tv"])
    tk, tv = c["tk"].copy(), c["tv"].copy()
    last = L - 1 - c["C"][0]
    tk[0, :, last] *= -3.0
    tv[0, :, last] += 5.0
    b, _ = attention.decode_verify(c["q"], c["cache"], c["lay"], c["bt"], c["lens"], 0.1, tk, tv)
    np.testing.assert_array_equal(a[0, :Q - 1], b[0, :Q - 1])
    assert np.abs(a[0, Q - 1] - b[0, Q - 1]).max() > 1e-3


def test_verify_keeps_a_tile_filled_by_drafts_raw():
    """The tokens under verification complete a tile (L - Q + 1 < 2N <= L):
    that tile is not committed, so every query reads its tokens raw; query 0
    equals plain decode at length L - Q + 1, whose commit point is the same."""
    N, Q = 64, 4
    L = 2 * N + 1  # accepted: 2N - 2 tokens, one committed tile
    c = _verify_case([L], Q, N=N)
    assert c["C"] == [N]
    out, _ = attention.decode_verify(c["q"], c["cache"], c["lay"], c["bt"], c["lens"], 0.1, c["tk"], c["tv"])
    ref, _ = attention.decode(c["q"][:, 0], c["cache"], c["lay"], c["bt"], np.array([L - Q + 1]), 0.1,
                              c["tk"][:, :, :N], c["tv"][:, :, :N])
    np.testing.assert_allclose(out[:, 0], ref, rtol=1e-12, atol=1e-13)
    # the last query: dequantised first tile, then 2N + 1 - N = N + 1 raw tokens
    K0, V0 = attention.sequence_kv(c["cache"], c["lay"], c["bt"][0], N, 0)
    K = np.concatenate([K0, c["k"][0, 0, N:L]])
    V = np.concatenate([V0, c["v"][0, 0, N:L]])
    s = 0.1 * K @ c["q"][0, Q - 1, 0]
    np.testing.assert_allclose(out[0, Q - 1, 0], scipy.special.softmax(s) @ V, rtol=1e-10, atol=1e-12)


def test_verify_queries_before_the_first_token_see_nothing():
    c = _verify_case([2], Q=4)
    out, lse = attention.decode_verify(c["q"], c["cache"], c["lay"], c["bt"], c["lens"], 0.1, c["tk"], c["tv"])
    assert (out[0, :2] == 0).all() and np.isneginf(lse[0, :2]).all()
    assert np.isfinite(lse[0, 2:]).all()


# ------------------------------------------------------- sink + recent records
def test_window_commit_points_by_hand():
    """(L, Q, N, sink, recent) -> end of the compressed tiles, worked by hand:
    accepted = L - Q + 1; whole tiles of [0, accepted - recent); not before
    the sink."""
    cases = [((1000, 1, 128, 128, 256), 640),   # 744 -> 5 tiles
             ((300, 1, 128, 128, 256), 128),    # 44 -> 0 tiles, clamped to the sink
             ((100, 1, 128, 128, 256), 128),    # shorter than the sink
             ((2050, 4, 64, 128, 1024), 960),   # 2047 - 1024 = 1023 -> 15 whole tiles of 64
             ((1151, 1, 128, 0, 1024), 0),      # 127 -> 0
             ((1152, 1, 128, 0, 1024), 128),    # 128 -> 1 tile
             ((1154, 3, 128, 0, 1024), 128)]    # accepted 1152 -> 128 -> 1 tile
    for args, want in cases:
        assert attention.window_committed(*args) == want, (args, want)


def test_window_without_records_is_verify():
    c = _verify_case([200, 64, 130], Q=2)
    a, la = attention.decode_verify(c["q"], c["cache"], c["lay"], c["bt"], c["lens"], 0.1, c["tk"], c["tv"])
    b, lb = attention.decode_window(c["q"], c["cache"], c["lay"], c["bt"], c["lens"], 0.1, 0, 0,
                                    tail_k=c["tk"], tail_v=c["tv"])
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_window_all_raw_is_causal_softmax():
    """L - Q + 1 <= sink + recent: every token is raw (sink rows, then tail
    rows from the sink's end); scipy softmax over the causally visible ones."""
    rng = np.random.default_rng(11)
    N, S, R, Q, D, L = 64, 64, 100, 2, 128, 150
    lay = layout.DenseLayout(D, N)
    k, v = rng.standard_normal((L, D)), rng.standard_normal((L, D))
    k[:, 3] *= 30  # an outlier channel stays exact in the raw records
    q = rng.standard_normal((1, Q, 2, D))
    assert attention.window_committed(L, Q, N, S, R) == S
    sk, sv = k[None, None, :S], v[None, None, :S]
    cap = R + N + Q - 2
    tk = np.zeros((1, 1, cap, D)); tv = np.zeros((1, 1, cap, D))
    tk[0, 0, :L - S], tv[0, 0, :L - S] = k[S:], v[S:]
    cache = np.zeros((1, 1, lay.page_bytes), np.uint8)
    out, lse = attention.decode_window(q, cache, lay, np.zeros((1, 8), int), np.array([L]), 0.09, S, R,
                                       sk, sv, tk, tv)
    for j in range(Q):
        for h in range(2):
            vis = L - Q + 1 + j
            s = 0.09 * k[:vis] @ q[0, j, h]
            np.testing.assert_allclose(out[0, j, h], scipy.special.softmax(s) @ v[:vis], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(lse[0, j, h], scipy.special.logsumexp(s), rtol=1e-12)


def test_window_reads_the_sink_raw_and_the_middle_from_pages():
    """Sink of one tile, one compressed tile, a raw tail: the output moves
    with a change to the raw sink row and not with a change to the tokens of
    the sink tile in the pages' source (they are never read)."""
    rng = np.random.default_rng(12)
    N, S, R, Q, D = 64, 64, 70, 1, 128
    L = 200  # accepted 200 - 70 = 130 -> 2 tiles -> C = 128: tile 1 compressed, tail [128, 200)
    lay = layout.DenseLayout(D, N)
    assert attention.window_committed(L, Q, N, S, R) == 128
    k, v = rng.standard_normal((L, D)), rng.standard_normal((L, D))
    q = rng.standard_normal((1, Q, 2, D))
    bt = np.arange(8)[None, :]
    cache = np.zeros((8, 1, lay.page_bytes), np.uint8)
    attention.encode_into_cache(cache, lay, k[None, None, :2 * N], v[None, None, :2 * N], bt, [0])
    sk, sv = k[None, None, :S].copy(), v[None, None, :S].copy()
    tk = np.zeros((1, 1, R + N + Q - 2, D)); tv = np.zeros_like(tk)
    tk[0, 0, :L - 128], tv[0, 0, :L - 128] = k[128:], v[128:]
    a, _ = attention.decode_window(q, cache, lay, bt, np.array([L]), 0.1, S, R, sk, sv, tk, tv)
    cache2 = cache.copy()
    cache2[bt[0, :4]] = 0  # the pages of tile 0 are not read under a one-tile sink
    b, _ = attention.decode_window(q, cache2, lay, bt, np.array([L]), 0.1, S, R, sk, sv, tk, tv)
    np.testing.assert_array_equal(a, b)
    sv2 = sv.copy(); sv2[0, 0, 5] += 4.0
    c, _ = attention.decode_window(q, cache, lay, bt, np.array([L]), 0.1, S, R, sk, sv2, tk, tv)
    assert np.abs(c - a).max() > 1e-4
    cache3 = cache.copy()
    cache3[bt[0, 4:8]] = 0  # the compressed tile 1 is read
    d, _ = attention.decode_window(q, cache3, lay, bt, np.array([L]), 0.1, S, R, sk, sv, tk, tv)
    assert np.abs(d - a).max() > 1e-4
