"""Pins of the oracle's page packing: hand-derived bytes of the documented
format, round trips, sizes and the capacity ratios the pages quote."""
import os

import numpy as np
import pytest

from oracle import layout

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _page_fixture():
    rows = []
    with open(os.path.join(GOLDEN, "page_bytes.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                kind, off, val, _ = [p.strip() for p in line.split("|")]
                rows.append((kind, int(off), int(val, 16)))
    return rows


def test_page_bytes_hand_derived():
    D = 128
    tau, j = np.meshgrid(np.arange(16), np.arange(D), indexing="ij")
    kc = (j + j // 16 + 3 * tau) % 16
    nc = j // 8
    vc = (j % 8 + nc * (nc + 1) // 2 + tau) % 4
    kb = layout.pack_codes(kc, "k")
    vb = layout.pack_codes(vc, "v")
    assert kb.size == 1024 and vb.size == 512
    for kind, off, val in _page_fixture():
        got = (kb if kind == "k" else vb)[off]
        assert got == val, (kind, off, hex(got), hex(val))


@pytest.mark.parametrize("D", [128, 256, 512])
def test_code_positions_are_a_bijection(D):
    kinds = [("k", 8 * D, 4), ("v", 4 * D, 2)] + ([("latent", 8 * D, 4)] if D >= 256 else [])
    fn = {"k": layout.k_code_position, "v": layout.v_code_position, "latent": layout.latent_code_position}
    for kind, nbytes, width in kinds:
        seen = set()
        for tau in range(16):
            for j in range(D):
                pos = fn[kind](D, tau, j)
                assert 0 <= pos[0] < nbytes and pos[1] % width == 0
                seen.add(pos)
        assert len(seen) == 16 * D


def test_latent_code_positions_hand_derived():
    """Latent width 512: token 0 keeps the K placement's unit order with the
    lane chunks interleaved; token 1 is shifted by four units (64 bytes).
    Channel 0 is lane chunk 0, word 0, nibble 0; channel 1 nibble 4 (byte 2);
    channel 8 nibble 1 (shift 4); channel 2 lane chunk 1 (unit 1); channel
    130 lane chunk 1, word 4 (unit 4 * 1 + 1 = 5)."""
    cases = {(0, 0): (0, 0), (1, 0): (256 + 64, 0), (0, 1): (2, 0), (1, 1): (256 + 66, 0),
             (0, 8): (0, 4), (1, 8): (256 + 64, 4), (0, 2): (16, 0), (1, 2): (256 + 80, 0),
             (0, 130): (80, 0), (1, 130): (256 + 16, 0)}
    for (tau, j), want in cases.items():
        assert layout.latent_code_position(512, tau, j) == want, (tau, j)


@pytest.mark.parametrize("D", [128, 256, 512])
def test_pack_unpack_roundtrip(D):
    rng = np.random.default_rng(D)
    for kind, q in (("k", 16), ("v", 4)) + ((("latent", 16),) if D >= 256 else ()):
        codes = rng.integers(0, q, (16, D))
        np.testing.assert_array_equal(layout.unpack_codes(layout.pack_codes(codes, kind), D, kind), codes)


@pytest.mark.parametrize("D,N,expected", [(128, 128, 1920), (128, 64, 2048), (256, 128, 3584),
                                          (512, 128, 6912)])
def test_dense_page_sizes(D, N, expected):
    lay = layout.DenseLayout(D, N)
    assert lay.page_bytes == expected
    for off in (lay.v_codes, lay.k_a, lay.k_col, lay.v_col, lay.page_bytes):
        assert off % 16 == 0


def test_latent_page_size():
    assert layout.LatentLayout(512, 64, 128).page_bytes == 6528


def test_capacity_ratios_match_pages():
    """KVarN review: roughly 4x KV capacity for k4v2_g128 on a dense model,
    within the 3-5x headline range; 2.77x for the int4 MLA latent. Our page
    format gives 4.27x and 2.82x."""
    dense = 2 * 2 * 128 / (layout.DenseLayout(128, 128).page_bytes / 16)
    assert 3.0 <= dense <= 5.0 and abs(dense - 4.0) < 0.3
    g64 = 2 * 2 * 128 / (layout.DenseLayout(128, 64).page_bytes / 16)
    assert g64 < dense  # the 64-token variant costs a little capacity
    mla = 2 * (512 + 64) / (layout.LatentLayout(512, 64, 128).page_bytes / 16)
    assert abs(mla - 2.77) / 2.77 < 0.03


def test_write_read_tile_roundtrip():
    lay = layout.DenseLayout(128, 128)
    rng = np.random.default_rng(0)
    cache = np.zeros((20, 2, lay.page_bytes), np.uint8)
    enc_k = dict(codes=rng.integers(0, 16, (128, 128)), a=rng.random(128), b=-rng.random(128),
                 c=rng.random(128) + 0.5)
    enc_v = dict(codes=rng.integers(0, 4, (128, 128)), a=rng.random(128), b=-rng.random(128),
                 c=rng.random(128) + 0.5)
    pages = [17, 3, 9, 0, 12, 5, 19, 8]
    layout.write_tile(cache, lay, pages, 1, enc_k, enc_v)
    assert (cache[:, 0] == 0).all()  # the other head is untouched
    k, v = layout.read_tile(cache, lay, pages, 1)
    for enc, got in ((enc_k, k), (enc_v, v)):
        np.testing.assert_array_equal(got["codes"], enc["codes"])
        for key in "abc":
            np.testing.assert_array_equal(got[key], enc[key].astype(np.float32).astype(np.float64))


# ------------------------------------------------ other widths (code planes)
def test_plane_positions_hand_derived():
    """D = 128. K plane: lane 4g + t, fragment 2kc + e, 8/w fragments per word,
    units of min(4, 2w) words; V plane: fragment nc, units of w words; element
    (h, e') of fragment f at bit 4f + 8e' + 16h (w = 4), 8f + 2h + 4e' (w = 2),
    f + 8h + 16e' (w = 1) (see the layout module)."""
    cases = {
        # (side, w, tau, j): (byte, shift)
        ("k", 1, 0, 0): (0, 0),
        ("k", 1, 9, 0): (32, 1),      # g1 t0 -> lane 4, e1 -> fragment 1 of word 0; units of 2 words (8 B)
        ("k", 1, 0, 112): (4, 6),     # kc7 -> fragment 14 = word 1, slot 6
        ("k", 1, 7, 127): (255, 6),   # lane 31, fragment 14, h1 e'1 -> bit 30
        ("k", 2, 8, 0): (1, 0),       # e1 -> fragment 1 = byte 1
        ("k", 2, 0, 16): (2, 0),      # kc1 -> fragment 2 = byte 2
        ("k", 2, 0, 32): (4, 0),      # kc2 -> word 1
        ("k", 2, 0, 8): (0, 2),       # h1 -> bit 2
        ("k", 2, 0, 1): (0, 4),       # e'1 -> bit 4
        ("k", 2, 15, 127): (511, 6),  # lane 31, fragment 15 = word 3 byte 3, h1 e'1 -> bit 30
        ("k", 4, 0, 1): (1, 0),       # e'1 -> byte 1
        ("k", 4, 0, 8): (2, 0),       # h1 -> half-word 1
        ("k", 4, 8, 0): (0, 4),       # e1 -> fragment 1, the high nibble
        ("v", 1, 0, 8): (0, 1),       # block 1 -> slot 1
        ("v", 1, 8, 0): (1, 0),       # h1 -> bit 8
        ("v", 1, 1, 0): (2, 0),       # e'1 -> bit 16
        ("v", 1, 2, 3): (52, 0),      # t1 g3 -> lane 13, 4-byte units
        ("v", 1, 15, 127): (255, 7),  # block 15 = word 1 slot 7, lane 31, bit 31
        ("v", 4, 0, 8): (0, 4),       # block 1 -> slot 1
        ("v", 4, 0, 16): (4, 0),      # block 2 -> word 1
        ("v", 4, 15, 127): (1023, 4),  # block 15 = word 7 = word 3 of unit 1, lane 31, bit 28
        ("v", 4, 1, 0): (1, 0),       # token 1: e'1 -> byte 1
        ("v", 4, 8, 0): (2, 0),       # token 8: h1 -> half-word 1
    }
    for (side, w, tau, j), want in cases.items():
        f = layout.k_plane_position if side == "k" else layout.v_plane_position
        assert f(128, tau, j, w) == want, (side, w, tau, j, f(128, tau, j, w), want)
    # the 4-bit K and 2-bit V placements are the w = 4 and w = 2 cases
    for tau in range(16):
        for j in range(128):
            assert layout.k_plane_position(128, tau, j, 4) == layout.k_code_position(128, tau, j)
            assert layout.v_plane_position(128, tau, j, 2) == layout.v_code_position(128, tau, j)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("side,w", [("k", 1), ("k", 2), ("v", 1), ("v", 4)])
def test_plane_positions_are_a_bijection(D, side, w):
    f = layout.k_plane_position if side == "k" else layout.v_plane_position
    seen = set()
    for tau in range(16):
        for j in range(D):
            byte, sh = f(D, tau, j, w)
            assert 0 <= byte < 2 * D * w and sh % w == 0 and sh + w <= 8
            seen.add((byte, sh))
    assert len(seen) == 16 * D


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_planes_roundtrip(bits):
    rng = np.random.default_rng(bits)
    for side in ("k", "v"):
        codes = rng.integers(0, 2 ** bits, (16, 128))
        region = layout.pack_planes(codes, bits, side)
        assert region.size == 2 * 128 * bits
        np.testing.assert_array_equal(layout.unpack_planes(region, 128, bits, side), codes)


def test_six_bit_fp16_scale_record_is_about_40_percent_of_fp16():
    """gmlx page, "The two schemes": at 6 bits a record takes about 40% of
    the memory of fp16. Here: K and V at 6 bits with fp16 scales."""
    lay = layout.DenseLayout(128, 128, 6, 6, scale_bytes=2)
    per_token = lay.page_bytes / 16
    assert lay.page_bytes == 3264
    assert abs(per_token / (2 * 2 * 128) - 0.40) < 0.01


@pytest.mark.parametrize("D,N,kb,vb,expected", [(128, 128, 8, 4, 3264), (256, 64, 2, 6, 4480)])
def test_mixed_width_page_bytes_hand_derived(D, N, kb, vb, expected):
    """Keys and values at their own widths (gmlx page, GMLX_KVARN_BITS), fp16
    scales. By hand, K8V4 at D 128, N 128: K part 2*128*8 codes + 2*16*2 of
    a, b + 128*16/128*2 of column slice = 2048 + 64 + 32 = 2144, V part
    1024 + 64 + 32 = 1120, 3264 in all (the same as K6V6: the code bits per
    token are equal). K2V6 at D 256, N 64: 1024 + 64 + 128 = 1216 and
    3072 + 64 + 128 = 3264, 4480 in all."""
    assert layout.DenseLayout(D, N, kb, vb, scale_bytes=2).page_bytes == expected


@pytest.mark.parametrize("D,kb,vb,sb", [(128, 6, 6, 2), (128, 3, 3, 2), (128, 8, 8, 2), (128, 4, 2, 2), (128, 5, 5, 4),
                                        (128, 8, 4, 2), (128, 2, 6, 2), (128, 5, 3, 2), (256, 6, 6, 2),
                                        (256, 3, 8, 2)])
def test_write_read_tile_roundtrip_other_widths(D, kb, vb, sb):
    lay = layout.DenseLayout(D, 64, kb, vb, scale_bytes=sb)
    rng = np.random.default_rng(kb * 10 + vb + D)
    cache = np.zeros((8, 1, lay.page_bytes), np.uint8)
    enc_k = dict(codes=rng.integers(0, 2 ** kb, (64, D)), a=rng.random(64), b=-rng.random(64), c=rng.random(D))
    enc_v = dict(codes=rng.integers(0, 2 ** vb, (64, D)), a=rng.random(64), b=-rng.random(64), c=rng.random(D))
    layout.write_tile(cache, lay, [5, 1, 7, 2], 0, enc_k, enc_v)
    k, v = layout.read_tile(cache, lay, [5, 1, 7, 2], 0)
    dt = np.float32 if sb == 4 else np.float16
    for enc, got in ((enc_k, k), (enc_v, v)):
        np.testing.assert_array_equal(got["codes"], enc["codes"])
        for key in "abc":
            np.testing.assert_array_equal(got[key], enc[key].astype(dt).astype(np.float64))
