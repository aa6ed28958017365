"""Byte layout of one cache page of one KV head, restated from the library's
documented format (test infrastructure only; shares no code with the CUDA
path).

The pages fix the tile (128 tokens, or 64 for the finer variant: KVarN review,
paragraph on kvarn_k4v2_g128), 4-bit keys and 2-bit values (same paragraph),
and a paged cache (vLLM block tables). Everything below the tile is this
library's own format. A page holds P = 16 tokens of one KV head:

  K codes   8*D bytes   4-bit. Lane L = 4g + t (g, t in 0..7, 0..3) owns,
                        for every 16-channel k-chunk kc, one 32-bit word;
                        its byte m = e + 2h holds channel
                        16kc + 2t + e + 8h of token g in the low nibble and
                        of token 8 + g in the high nibble. Words are stored
                        as 16-byte units of four k-chunks: the word of
                        (kc, L) sits at byte 16*(32*(kc//4) + L) + 4*(kc%4).
  V codes   4*D bytes   2-bit. Lane L = 4g + t owns, for every four 8-channel
                        blocks nc = 4w + c, one 32-bit word whose byte c is
                        channel 8nc + g; token 2t + e + 8h of that channel
                        sits at bit 2h + 4e of the byte.
                        Words are stored as 8-byte units of two: the word w
                        of lane L sits at byte 8*(32*(w//2) + L) + 4*(w%2).
  The page is two parts, each contiguous: the K part (K codes, then K a[16],
  K b[16] fp32 row scales, then the K column-scale slice, D*P/N fp32), then
  the V part (V codes, V a[16], V b[16], V column-scale slice).
The page at logical index l of a sequence carries the column scales of
channels [(l mod N/P) * D*P/N, +D*P/N) of its tile; all words little-endian.

Other widths (gmlx page, "The two schemes": kvarn widths 2, 3, 4, 5, 6 and 8,
separate for keys and values). A b-bit code is stored as one or two planes,
b = 2: [2], 3: [2, 1], 4: [4], 5: [4, 1], 6: [4, 2], 8: [4, 4], the code
being plane0 + 2^w0 plane1; each plane region (2*D*w bytes per page, the
planes in order) follows one rule for a plane of width w in {1, 2, 4}: lane
L = 4g + t owns words of 8/w fragments each;
fragment f of a word holds two operand registers h = 0, 1 of two elements
e' = 0, 1 each, element (h, e') at bit
    w = 4:  4f + 8e' + 16h   (register h = half-word h, element = byte)
    w = 2:  8f + 2h + 4e'    (fragment = byte f)
    w = 1:  f + 8h + 16e'.
  K plane: fragment 2*kc + e (k-chunk kc, token block e: tokens 8e + g);
           element (h, e') is channel 16kc + 2t + e' + 8h. Words go in
           units of U = min(4, D*w/64) words: word i of lane L at byte
           4U*(32*(i//U) + L) + 4*(i%U).
  V plane: fragment nc (8-channel block); element (h, e') is channel
           8nc + g of token 2t + e' + 8h. Words go in units of w
           words (eight blocks): word i of lane L at 4w*(32*(i//w) + L) +
           4*(i%w).
The 4-bit K and 2-bit V placements above are the w = 4 and w = 2 cases. The
scales are fp32 ("S32") or fp16 ("S16"): a[16], b[16], col as 2-byte values.
"""
from __future__ import annotations

import functools

import numpy as np

P = 16  # tokens per page


PLANES = {2: (2,), 3: (2, 1), 4: (4,), 5: (4, 1), 6: (4, 2), 8: (4, 4)}


def _align16(x: int) -> int:
    return (x + 15) // 16 * 16


class DenseLayout:
    def __init__(self, D: int, N: int, k_bits: int = 4, v_bits: int = 2, scale_bytes: int = 4):
        if k_bits not in PLANES or v_bits not in PLANES or scale_bytes not in (2, 4):
            raise ValueError("widths 2, 3, 4, 5, 6, 8 and fp32 or fp16 scales")
        if N % P:
            raise ValueError("tile must be a whole number of pages")
        self.D, self.N, self.k_bits, self.v_bits, self.sb = D, N, k_bits, v_bits, scale_bytes
        sb = scale_bytes
        self.col_per_page = D * P // N
        self.k_codes = 0
        self.k_a = 2 * D * k_bits
        self.k_b = self.k_a + sb * P
        self.k_col = self.k_b + sb * P
        self.v_codes = _align16(self.k_col + sb * self.col_per_page)   # start of the V part
        self.v_a = self.v_codes + 2 * D * v_bits
        self.v_b = self.v_a + sb * P
        self.v_col = self.v_b + sb * P
        self.page_bytes = _align16(self.v_col + sb * self.col_per_page)


def k_code_position(D: int, tau: int, j: int):
    """(byte offset inside the K-code region, bit shift) of token tau, channel j."""
    kc, r = divmod(j, 16)
    t, e, h = (r % 8) // 2, r % 2, r // 8
    g, upper = tau % 8, tau // 8
    lane = 4 * g + t
    word = 16 * (32 * (kc // 4) + lane) + 4 * (kc % 4)
    return word + e + 2 * h, 4 * upper


def v_code_position(D: int, tau: int, j: int):
    """(byte offset inside the V-code region, bit shift) of token tau, channel j."""
    nc, g = divmod(j, 8)
    t, e, h = (tau % 8) // 2, tau % 2, tau // 8
    w, c = divmod(nc, 4)
    lane = 4 * g + t
    bit = 8 * c + 2 * h + 4 * e
    return 8 * (32 * (w // 2) + lane) + 4 * (w % 2) + bit // 8, bit % 8


def plane_bit(w: int, f: int, h: int, ep: int) -> int:
    """Bit of element (h, e') of fragment f in a plane word of width w."""
    if w == 4:
        return 4 * f + 8 * ep + 16 * h
    if w == 2:
        return 8 * f + 2 * h + 4 * ep
    return f + 8 * h + 16 * ep


def k_plane_position(D: int, tau: int, j: int, w: int):
    """(byte, bit shift) of token tau, channel j inside a K plane of width w."""
    F = 8 // w
    kc, r = divmod(j, 16)
    t, ep, h = (r % 8) // 2, r % 2, r // 8
    g, e = tau % 8, tau // 8
    lane = 4 * g + t
    word, f = divmod(2 * kc + e, F)
    U = min(4, D * w // 64)
    bit = plane_bit(w, f, h, ep)
    return 4 * U * (32 * (word // U) + lane) + 4 * (word % U) + bit // 8, bit % 8


def v_plane_position(D: int, tau: int, j: int, w: int):
    """(byte, bit shift) of token tau, channel j inside a V plane of width w."""
    F = 8 // w
    nc, g = divmod(j, 8)
    t, ep, h = (tau % 8) // 2, tau % 2, tau // 8
    lane = 4 * g + t
    word, f = divmod(nc, F)
    bit = plane_bit(w, f, h, ep)
    return 4 * w * (32 * (word // w) + lane) + 4 * (word % w) + bit // 8, bit % 8


def _latent_word_position(D: int, tau: int, j: int):
    """Word content of the latent page before its 16-byte units are
    reordered: token-major rows of D/2 bytes made of four lane chunks of D/8
    bytes; chunk t holds, for every 16-channel k-chunk kc, channels
    16kc + {2t, 2t+1, 2t+8, 2t+9}; word w of a chunk serves kc = 2w, 2w+1 and
    its nibble n holds channel 16(2w + (n%4)//2) + 2t + 8(n%2) + n//4."""
    kc, r = divmod(j, 16)
    t = (r % 8) // 2
    e = r % 2
    h = r // 8
    w, kp = divmod(kc, 2)
    n = 2 * kp + h + 4 * e
    byte = tau * (D // 2) + t * (D // 8) + 4 * w + n // 2
    return byte, 4 * (n % 2)


def latent_code_position(D: int, tau: int, j: int):
    """(byte offset inside the latent-code region, bit shift) of token tau,
    channel j. The word content of _latent_word_position, with the 16-byte
    units of a token row (unit 4t + q holds words 4q..4q+3 of lane chunk t)
    stored at unit (4q + t) XOR 4*(tau%2): lane chunks interleaved, odd
    tokens shifted by four units."""
    byte, shift = _latent_word_position(D, tau, j)
    r = byte - tau * (D // 2)
    t, rem = divmod(r, D // 8)
    q, within = divmod(rem, 16)
    unit = (4 * q + t) ^ (4 * (tau % 2))
    return tau * (D // 2) + 16 * unit + within, shift


@functools.lru_cache(maxsize=None)
def _maps(D: int):
    pos = {"k": k_code_position, "v": v_code_position, "latent": latent_code_position}
    for w in (1, 2, 4):
        pos[f"k{w}"] = functools.partial(k_plane_position, w=w)
        pos[f"v{w}"] = functools.partial(v_plane_position, w=w)
    out = {}
    for kind, f in pos.items():
        if kind == "latent" and D // 32 < 8:
            continue  # the latent order needs at least 8 units per token row
        byte = np.zeros((P, D), dtype=np.int64)
        shift = np.zeros((P, D), dtype=np.int64)
        for tau in range(P):
            for j in range(D):
                byte[tau, j], shift[tau, j] = f(D, tau, j)
        out[kind] = (byte, shift)
    return out


_WIDTH = {"k": (4, 8), "latent": (4, 8), "v": (2, 4),   # bits, bytes per channel of a page
          "k1": (1, 2), "k2": (2, 4), "k4": (4, 8), "v1": (1, 2), "v2": (2, 4), "v4": (4, 8)}


def pack_codes(codes: np.ndarray, kind: str) -> np.ndarray:
    """Pack a [16, D] code block of one page into its region bytes."""
    D = codes.shape[1]
    byte, shift = _maps(D)[kind]
    out = np.zeros(_WIDTH[kind][1] * D, dtype=np.int64)
    np.bitwise_or.at(out, byte.ravel(), (codes.astype(np.int64) << shift).ravel())
    return out.astype(np.uint8)


def unpack_codes(region: np.ndarray, D: int, kind: str) -> np.ndarray:
    byte, shift = _maps(D)[kind]
    mask = (1 << _WIDTH[kind][0]) - 1
    return (region.astype(np.int64)[byte] >> shift) & mask


def pack_planes(codes: np.ndarray, bits: int, side: str) -> np.ndarray:
    """A [16, D] block of `bits`-bit codes of K (side "k") or V ("v") as its
    plane regions in order. The K4 / V2 planes are the "k" / "v" kinds."""
    out, rest = [], codes.astype(np.int64)
    for w in PLANES[bits]:
        plane = rest & ((1 << w) - 1)
        rest = rest >> w
        kind = {("k", 4): "k", ("v", 2): "v"}.get((side, w), f"{side}{w}")
        out.append(pack_codes(plane, kind))
    return np.concatenate(out)


def unpack_planes(region: np.ndarray, D: int, bits: int, side: str) -> np.ndarray:
    codes, off, shift = 0, 0, 0
    for w in PLANES[bits]:
        kind = {("k", 4): "k", ("v", 2): "v"}.get((side, w), f"{side}{w}")
        n = 2 * D * w
        codes = codes + (unpack_codes(region[off:off + n], D, kind) << shift)
        off += n
        shift += w
    return codes


def f32_bytes(x) -> np.ndarray:
    return np.asarray(x, dtype="<f4").view(np.uint8)


def f32_from(region: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(region).view("<f4").astype(np.float64)


def scale_bytes(x, sb: int) -> np.ndarray:
    return np.asarray(x, dtype="<f4" if sb == 4 else "<f2").view(np.uint8)


def scale_from(region: np.ndarray, sb: int) -> np.ndarray:
    return np.ascontiguousarray(region).view("<f4" if sb == 4 else "<f2").astype(np.float64)


def write_tile(cache: np.ndarray, lay: DenseLayout, phys_pages, head: int,
               enc_k: dict, enc_v: dict) -> None:
    """Store the encodings of one K tile and one V tile (N tokens) into the
    N/P physical pages ``phys_pages`` of KV head ``head``.

    cache: uint8 [num_pages, Hkv, page_bytes].
    """
    D, N, cpp, sb = lay.D, lay.N, lay.col_per_page, lay.sb
    for p, phys in enumerate(phys_pages):
        pg = cache[phys, head]
        rows = slice(p * P, (p + 1) * P)
        cols = slice(p * cpp, (p + 1) * cpp)
        pg[lay.k_codes:lay.k_codes + 2 * D * lay.k_bits] = pack_planes(enc_k["codes"][rows], lay.k_bits, "k")
        pg[lay.v_codes:lay.v_codes + 2 * D * lay.v_bits] = pack_planes(enc_v["codes"][rows], lay.v_bits, "v")
        pg[lay.k_a:lay.k_a + sb * P] = scale_bytes(enc_k["a"][rows], sb)
        pg[lay.k_b:lay.k_b + sb * P] = scale_bytes(enc_k["b"][rows], sb)
        pg[lay.v_a:lay.v_a + sb * P] = scale_bytes(enc_v["a"][rows], sb)
        pg[lay.v_b:lay.v_b + sb * P] = scale_bytes(enc_v["b"][rows], sb)
        pg[lay.k_col:lay.k_col + sb * cpp] = scale_bytes(enc_k["c"][cols], sb)
        pg[lay.v_col:lay.v_col + sb * cpp] = scale_bytes(enc_v["c"][cols], sb)


def read_tile(cache: np.ndarray, lay: DenseLayout, phys_pages, head: int):
    """Inverse of write_tile: returns (K dict, V dict) of codes [N, D] and
    float64 copies of the stored a [N], b [N], c [D] (fp32 or fp16)."""
    D, cpp, sb = lay.D, lay.col_per_page, lay.sb
    out = {}
    for kind in ("k", "v"):
        codes, a, b, c = [], [], [], []
        base, bits = (lay.k_codes, lay.k_bits) if kind == "k" else (lay.v_codes, lay.v_bits)
        oa, ob, oc = (lay.k_a, lay.k_b, lay.k_col) if kind == "k" else (lay.v_a, lay.v_b, lay.v_col)
        for phys in phys_pages:
            pg = cache[phys, head]
            codes.append(unpack_planes(pg[base:base + 2 * D * bits], D, bits, kind))
            a.append(scale_from(pg[oa:oa + sb * P], sb))
            b.append(scale_from(pg[ob:ob + sb * P], sb))
            c.append(scale_from(pg[oc:oc + sb * cpp], sb))
        out[kind] = dict(codes=np.concatenate(codes), a=np.concatenate(a),
                         b=np.concatenate(b), c=np.concatenate(c))
    return out["k"], out["v"]


# --------------------------------------------------------------------------
# MLA latent page: one shared latent of width Dl (4-bit codes, K = V) plus an
# fp16 rope part of width R, 16 tokens per page.
#   latent codes  8*Dl bytes   latent word content, 16-byte units reordered
#                              (latent_code_position)
#   rope          2*R*P bytes  fp16, token-major
#   a[16], b[16]  fp32
#   col           Dl*P/N fp32  column-scale slice, as for the dense page
# --------------------------------------------------------------------------
class LatentLayout:
    def __init__(self, Dl: int, R: int, N: int):
        self.D, self.R, self.N = Dl, R, N
        self.codes = 0
        self.rope = 8 * Dl
        self.a = self.rope + 2 * R * P
        self.b = self.a + 4 * P
        self.col_per_page = Dl * P // N
        self.col = self.b + 4 * P
        self.page_bytes = self.col + 4 * self.col_per_page
