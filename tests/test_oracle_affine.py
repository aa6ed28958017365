"""Pins of the oracle's affine comparison pages (test infrastructure; CPU
only): the page format stated in include/kvarn.h, restated independently in
oracle/affine.py, and the affine decode by its plain definition (gmlx page,
"The two schemes": groups of 64 values per token, an fp16 scale and offset
per group)."""
import numpy as np

from oracle import affine, attention, layout


def test_page_offsets_by_hand():
    # K part: 2*128*4 = 1024 code bytes, then 16 tokens x 8 bytes of records
    # (1152, already 16-aligned); V part the same: 2304 bytes
    lay = affine.AffineLayout(128, 4, 4)
    assert (lay.k_sc, lay.v_codes, lay.v_sc, lay.page_bytes) == (1024, 1152, 2176, 2304)
    lay = affine.AffineLayout(128, 3, 3)
    assert (lay.k_sc, lay.v_codes, lay.v_sc, lay.page_bytes) == (768, 896, 1664, 1792)
    assert affine.AffineLayout(128, 8, 8).page_bytes == 4352


def test_token_record_bytes_by_hand():
    """Token 3 with K group scales (1, 2) and offsets (-0.5, 0.25): fp16
    0x3C00, 0x4000, 0xB800, 0x3400, little-endian, at byte 1024 + 8 * 3 of
    the K part; V records likewise at 1152 + 1024 + 8 t."""
    lay = affine.AffineLayout(128, 4, 4)
    cache = np.zeros((1, 1, lay.page_bytes), np.uint8)
    z = np.zeros((16, 128), np.int64)
    ks, ko = np.zeros((16, 2)), np.zeros((16, 2))
    ks[3], ko[3] = [1.0, 2.0], [-0.5, 0.25]
    vs, vo = np.zeros((16, 2)), np.zeros((16, 2))
    vs[15], vo[15] = [0.5, 4.0], [1.0, -2.0]
    affine.write_tokens(cache, lay, [0], 0, (z, ks, ko), (z, vs, vo))
    pg = cache[0, 0]
    assert list(pg[1024 + 24:1024 + 32]) == [0x00, 0x3C, 0x00, 0x40, 0x00, 0xB8, 0x00, 0x34]
    # V token 15: 0.5 = 0x3800, 4 = 0x4400, 1 = 0x3C00, -2 = 0xC000
    assert list(pg[2176 + 120:2176 + 128]) == [0x00, 0x38, 0x00, 0x44, 0x00, 0x3C, 0x00, 0xC0]
    assert int(pg[:1024].sum()) == 0 and int(pg[1152:2176].sum()) == 0


def test_codes_use_the_dense_plane_placement():
    """The codes of an affine page sit exactly where the dense page's K / V
    codes of the same width sit (the pinned layout of oracle/layout.py)."""
    rng = np.random.default_rng(3)
    for bits in (2, 3, 4, 6, 8):
        lay = affine.AffineLayout(128, bits, bits)
        codes_k = rng.integers(0, 2 ** bits, size=(16, 128))
        codes_v = rng.integers(0, 2 ** bits, size=(16, 128))
        cache = np.zeros((1, 1, lay.page_bytes), np.uint8)
        one = np.ones((16, 2))
        affine.write_tokens(cache, lay, [0], 0, (codes_k, one, one), (codes_v, one, one))
        pg = cache[0, 0]
        np.testing.assert_array_equal(pg[:2 * 128 * bits], layout.pack_planes(codes_k, bits, "k"))
        np.testing.assert_array_equal(pg[lay.v_codes:lay.v_codes + 2 * 128 * bits],
                                      layout.pack_planes(codes_v, bits, "v"))


def test_write_read_roundtrip():
    rng = np.random.default_rng(5)
    lay = affine.AffineLayout(128, 6, 6)
    x = rng.standard_normal((32, 128)) * 3
    y = rng.standard_normal((32, 128))
    qk, qv = affine.quantize(x, 6), affine.quantize(y, 6)
    cache = np.zeros((3, 2, lay.page_bytes), np.uint8)
    affine.write_tokens(cache, lay, [2, 0], 1, qk, qv)
    rk, rv = affine.read_tokens(cache, lay, [2, 0], 1)
    for a, b in zip(qk + qv, rk + rv):
        np.testing.assert_array_equal(a, b)


def test_decode_is_attention_over_the_dequantised_rows():
    """Two tiles through the pages (permuted block table) and a 37-token raw
    tail: equal to softmax attention over the rows dequantised straight from
    quantize(), and the raw tail rows."""
    rng = np.random.default_rng(11)
    N, L, D = 128, 2 * 128 + 37, 128
    k = rng.standard_normal((1, 1, L, D))
    v = rng.standard_normal((1, 1, L, D))
    q = rng.standard_normal((1, 4, D))
    lay = affine.AffineLayout(D, 4, 4)
    bt = np.array([[5, 3, 12, 0, 7, 9, 1, 15, 2, 4, 6, 8, 10, 11, 13, 14]])
    cache = np.zeros((16, 1, lay.page_bytes), np.uint8)
    affine.encode_into_cache(cache, lay, k[:, :, :256], v[:, :, :256], bt, N)
    tk = np.zeros((1, 1, N, D))
    tv = np.zeros((1, 1, N, D))
    tk[0, 0, :37], tv[0, 0, :37] = k[0, 0, 256:], v[0, 0, 256:]
    out, lse = affine.decode(q, cache, lay, bt, [L], 0.1, N, tk, tv)
    K = np.concatenate([affine.dequantize(*affine.quantize(k[0, 0, :256], 4)), k[0, 0, 256:]])
    V = np.concatenate([affine.dequantize(*affine.quantize(v[0, 0, :256], 4)), v[0, 0, 256:]])
    for h in range(4):
        ref, rl = attention.softmax_attention(q[0, h], K, V, 0.1)
        np.testing.assert_allclose(out[0, h], ref, rtol=0, atol=1e-12)
        assert abs(lse[0, h] - rl) < 1e-12


def test_decode_tail_only_and_empty():
    rng = np.random.default_rng(2)
    lay = affine.AffineLayout(128, 4, 4)
    cache = np.zeros((1, 1, lay.page_bytes), np.uint8)
    k = rng.standard_normal((1, 1, 128, 128))
    q = rng.standard_normal((2, 2, 128))
    bt = np.zeros((2, 8), np.int64)
    out, lse = affine.decode(q, cache, lay, bt, [40, 0], 0.2, 128, np.concatenate([k, k]), np.concatenate([k, k]))
    ref, _ = attention.softmax_attention(q[0, 1], k[0, 0, :40], k[0, 0, :40], 0.2)
    np.testing.assert_allclose(out[0, 1], ref, atol=1e-12)
    assert (out[1] == 0).all() and np.isneginf(lse[1]).all()
