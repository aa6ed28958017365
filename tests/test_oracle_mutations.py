"""The oracle's pins must catch plausible mistakes in the oracle itself.

Each case below plants one mistake in the oracle (a dropped term, a wrong sign
or index, a swapped operand or order) by patching a function of the oracle
package, runs the pin tests of test_oracle_codec, test_oracle_layout and
test_oracle_attention, and expects at least one pin to fail. Everything runs
on the CPU; nothing here touches the CUDA path.
"""
import numpy as np
import pytest

from oracle import attention, codec, layout
from tests import test_oracle_attention as ta
from tests import test_oracle_codec as tc
from tests import test_oracle_layout as tl

PINS = [
    (tc.test_hadamard_matches_scipy_sylvester, dict(D=128)),
    (tc.test_hadamard_orthonormal_and_symmetric, dict(D=128)),
    (tc.test_rotation_preserves_scores, dict(D=128)),
    (tc.test_rotation_tiny_by_hand, {}),
    (tc.test_sinkhorn_closed_form, {}),
    (tc.test_normalize_reconstructs_exactly, {}),
    (tc.test_normalize_rows_have_unit_std, dict(T=2)),
    (tc.test_column_pass_gives_unit_column_std, {}),
    (tc.test_normalize_columns_converge_toward_one, {}),
    (tc.test_normalize_constant_vectors_keep_unit_scale, {}),
    (tc.test_normalize_tiny_spread_is_not_constant, {}),
    (tc.test_rtn_hand_worked_rows, {}),
    (tc.test_rtn_range_endpoints_and_error_bound, dict(bits=4)),
    (tc.test_reconstruction_error_shrinks_with_bits, {}),
    (tc.test_dequantize_roundtrip_is_exact_without_rounding, {}),
    (tl.test_page_bytes_hand_derived, {}),
    (tl.test_write_read_tile_roundtrip, {}),
    (tl.test_plane_positions_hand_derived, {}),
    (tl.test_mixed_width_page_bytes_hand_derived, dict(D=128, N=128, kb=8, vb=4, expected=3264)),
    (ta.test_softmax_attention_matches_scipy, {}),
    (ta.test_softmax_attention_two_tokens_by_hand, {}),
    (ta.test_decode_equals_rotated_space_computation, {}),
    (ta.test_tail_only_sequence_is_plain_attention, {}),
    (ta.test_mla_decode_rope_and_shared_latent, {}),
    (ta.test_verify_without_committed_tiles_is_causal_softmax, {}),
    (ta.test_verify_keeps_a_tile_filled_by_drafts_raw, {}),
    (ta.test_window_commit_points_by_hand, {}),
    (ta.test_window_all_raw_is_causal_softmax, {}),
]


def _pins_fail():
    for fn, kw in PINS:
        try:
            fn(**kw)
        except AssertionError:
            return fn.__name__
    return None


def _hadamard_unscaled(orig):
    return lambda D: orig(D) * np.sqrt(D)


def _hadamard_wrong_sign(orig):
    def H(D):
        M = np.ones((1, 1))
        while M.shape[0] < D:
            M = np.block([[M, M], [-M, M]])
        return M / np.sqrt(D)
    return H


def _normalize_row_first(orig):
    def vn(Y, T):
        Z = np.array(Y, dtype=np.float64)
        lr, lc = np.zeros(Z.shape[0]), np.zeros(Z.shape[1])
        for _ in range(T):
            Z, a = codec.row_pass(Z)
            lr += a
            Z, b = codec.column_pass(Z)
            lc += b
        return Z, np.exp(lr), np.exp(lc)
    return vn


def _normalize_swap_scales(orig):
    def vn(Y, T):
        Z, r, c = orig(Y, T)
        return Z, np.resize(c, r.size), np.resize(r, c.size)
    return vn


def _std_sample(orig):
    def s(Z, axis):
        v = np.std(Z, axis=axis, ddof=1)
        return np.where(np.isfinite(v) & (v > 0), v, 1.0)
    return s


def _std_relative_threshold(orig):
    # a near-constant vector (std <= 2^-20 |mean|) treated as constant
    def s(Z, axis):
        v = np.std(Z, axis=axis, ddof=0)
        mu = np.abs(np.mean(Z, axis=axis))
        return np.where(np.isfinite(v) & (v > 2.0 ** -20 * mu), v, 1.0)
    return s


def _std_zero_only(orig):
    # only sigma == 0 in float64 counts as constant: the rounding residue of
    # the mean of an exactly constant vector is divided out as spread
    def s(Z, axis):
        v = np.std(Z, axis=axis, ddof=0)
        return np.where(np.isfinite(v) & (v > 0), v, 1.0)
    return s


def _rtn_floor(orig):
    def rtn(Z, bits):
        codes, lo, delta, x = orig(Z, bits)
        return np.clip(np.floor(x), 0, 2 ** bits - 1).astype(np.int64), lo, delta, x
    return rtn


def _rtn_levels_off_by_one(orig):
    return _rtn_levels


def _rtn_levels(Z, bits):
    lo, hi = Z.min(1), Z.max(1)
    delta = (hi - lo) / (2 ** bits)
    safe = np.where(delta > 0, delta, 1.0)
    x = (Z - lo[:, None]) / safe[:, None]
    return np.clip(np.rint(x), 0, 2 ** bits - 1).astype(np.int64), lo, delta, x


def _dequant_drop_b(orig):
    return lambda codes, a, b, c: orig(codes, a, np.zeros_like(np.asarray(b, float)), c)


def _dequant_no_unrotate(orig):
    return lambda codes, a, b, c: codec.dequantize_rotated(codes, a, b, c)


def _attention_no_scale(orig):
    return lambda q, K, V, sm_scale: orig(q, K, V, 1.0)


def _k_nibble_order(orig):
    # the pair element and the upper-eight flag trade places in the byte index
    def pos(D, tau, j):
        kc, r = divmod(j, 16)
        t, e, h = (r % 8) // 2, r % 2, r // 8
        lane = 4 * (tau % 8) + t
        return 16 * (32 * (kc // 4) + lane) + 4 * (kc % 4) + h + 2 * e, 4 * (tau // 8)
    return pos


def _v_pair_order(orig):
    # tokens 8 apart and tokens 1 apart trade their bit offsets
    def pos(D, tau, j):
        nc, g = divmod(j, 8)
        t, e, h = (tau % 8) // 2, tau % 2, tau // 8
        w, c = divmod(nc, 4)
        bit = 8 * c + 4 * h + 2 * e
        return 8 * (32 * (w // 2) + 4 * g + t) + 4 * (w % 2) + bit // 8, bit % 8
    return pos


def _wrong_kv_head(orig):
    def skv(cache, lay, bt_row, seq_len, head, tail_k=None, tail_v=None):
        return orig(cache, lay, bt_row, seq_len, (head + 1) % cache.shape[1], tail_k, tail_v)
    return skv


def _tail_off_by_one(orig):
    def skv(cache, lay, bt_row, seq_len, head, tail_k=None, tail_v=None):
        tk = None if tail_k is None else np.roll(np.asarray(tail_k), -1, axis=0)
        return orig(cache, lay, bt_row, seq_len, head, tk, tail_v)
    return skv


def _commit_from_full_length(orig):
    return lambda L, Q, N: (L // N) * N


def _visible_off_by_one(orig):
    return lambda L, Q, j: max(0, L - Q + j)


def _plane_halves_swapped(orig):
    # the pair element and the second-register flag trade bit offsets
    def pos(D, tau, j, w):
        F = 8 // w
        kc, r = divmod(j, 16)
        t, ep, h = (r % 8) // 2, r % 2, r // 8
        word, f = divmod(2 * kc + tau // 8, F)
        U = min(4, D * w // 64)
        bit = layout.plane_bit(w, f, ep, h)
        return 4 * U * (32 * (word // U) + 4 * (tau % 8) + t) + 4 * (word % U) + bit // 8, bit % 8
    return pos


def _recent_ignored(orig):
    return lambda L, Q, N, sink, recent: orig(L, Q, N, sink, 0)


def _v_region_at_key_width(orig):
    # the V codes sized by the key width (separate widths mixed up)
    class Mut(orig):
        def __init__(self, D, N, k_bits=4, v_bits=2, scale_bytes=4):
            super().__init__(D, N, k_bits, v_bits, scale_bytes)
            self.v_a = self.v_codes + 2 * D * k_bits
            self.v_b = self.v_a + scale_bytes * layout.P
            self.v_col = self.v_b + scale_bytes * layout.P
            self.page_bytes = layout._align16(self.v_col + scale_bytes * self.col_per_page)
    return Mut


MUTATIONS = [
    ("hadamard without 1/sqrt(D)", codec, "hadamard", _hadamard_unscaled),
    ("hadamard with a wrong sign", codec, "hadamard", _hadamard_wrong_sign),
    ("row pass before column pass", codec, "variance_normalize", _normalize_row_first),
    ("row and column scales swapped", codec, "variance_normalize", _normalize_swap_scales),
    ("sample std instead of population std", codec, "pop_std", _std_sample),
    ("constant test with a relative threshold", codec, "pop_std", _std_relative_threshold),
    ("constant test on the float64 std alone", codec, "pop_std", _std_zero_only),
    ("floor instead of round-to-nearest", codec, "rtn_rows", _rtn_floor),
    ("2^bits levels instead of 2^bits - 1", codec, "rtn_rows", _rtn_levels_off_by_one),
    ("offset term b dropped at dequantisation", codec, "dequantize_rotated", _dequant_drop_b),
    ("output left in the rotated basis", codec, "dequantize", _dequant_no_unrotate),
    ("softmax scale ignored", attention, "softmax_attention", _attention_no_scale),
    ("K nibbles in the wrong order", layout, "k_code_position", _k_nibble_order),
    ("V token halves swapped", layout, "v_code_position", _v_pair_order),
    ("query head mapped to the wrong KV head", attention, "sequence_kv", _wrong_kv_head),
    ("tail read one token off", attention, "sequence_kv", _tail_off_by_one),
    ("verify commits tiles the drafts filled", attention, "verify_committed", _commit_from_full_length),
    ("verify query sees one token too few", attention, "verify_visible", _visible_off_by_one),
    ("recent raw records ignored", attention, "window_committed", _recent_ignored),
    ("plane register halves swapped", layout, "k_plane_position", _plane_halves_swapped),
    ("V codes sized by the key width", layout, "DenseLayout", _v_region_at_key_width),
]


@pytest.mark.parametrize("label,module,name,make", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(monkeypatch, label, module, name, make):
    assert _pins_fail() is None  # the clean oracle passes every pin
    monkeypatch.setattr(module, name, make(getattr(module, name)))
    layout._maps.cache_clear()
    try:
        caught = _pins_fail()
    finally:
        layout._maps.cache_clear()
    assert caught is not None, f"no pin caught: {label}"
