"""Pins of the oracle's codec against facts the pages and the mathematics fix.

Every test here checks the oracle against something other than itself: a
library routine, a closed form worked by hand, an invariant, or a hand-worked
fixture under tests/golden/.
"""
import os

import numpy as np
import pytest
import scipy.linalg

from oracle import codec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append([p.strip() for p in line.split("|")])
    return out


# ---------------------------------------------------------------- rotation
@pytest.mark.parametrize("D", [1, 2, 4, 8, 16, 64, 128, 256, 512])
def test_hadamard_matches_scipy_sylvester(D):
    """scipy.linalg.hadamard builds the same Sylvester matrix (unscaled)."""
    np.testing.assert_array_equal(codec.hadamard(D) * np.sqrt(D), scipy.linalg.hadamard(D))


@pytest.mark.parametrize("D", [2, 128, 256, 512])
def test_hadamard_orthonormal_and_symmetric(D):
    """KVarN review, four-stage paragraph: the rotation is orthonormal."""
    H = codec.hadamard(D)
    np.testing.assert_allclose(H @ H.T, np.eye(D), atol=1e-12)
    np.testing.assert_array_equal(H, H.T)
    np.testing.assert_allclose(H @ H, np.eye(D), atol=1e-12)   # its own inverse


@pytest.mark.parametrize("D", [128, 512])
def test_rotation_preserves_scores(D):
    """Scores on rotated keys equal scores on raw keys when the query is
    rotated by the same matrix (turbo-attn, "How it works")."""
    rng = np.random.default_rng(1)
    q = rng.standard_normal(D)
    K = rng.standard_normal((37, D)) * rng.exponential(3, D)
    np.testing.assert_allclose(codec.rotate(K) @ codec.rotate(q), K @ q, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(np.linalg.norm(codec.rotate(K), axis=1),
                               np.linalg.norm(K, axis=1), rtol=1e-12)


def test_rotation_tiny_by_hand():
    """D = 2: H = [[1, 1], [1, -1]] / sqrt 2, so (3, 1) -> (4, 2) / sqrt 2."""
    np.testing.assert_allclose(codec.rotate(np.array([[3.0, 1.0]])),
                               [[4 / np.sqrt(2), 2 / np.sqrt(2)]], rtol=1e-15)


def test_rotation_spreads_outlier_channel():
    """A channel 20x larger than the rest (the toy workload's outliers) is
    spread: the peak-to-rms ratio of each token drops (KVarN review:
    the rotation "spreads out per-channel outliers")."""
    rng = np.random.default_rng(2)
    X = rng.standard_normal((128, 128))
    X[:, 31] *= 20
    crest = lambda A: (np.abs(A).max(1) / np.sqrt((A ** 2).mean(1))).mean()
    assert crest(codec.rotate(X)) < 0.5 * crest(X)


# ----------------------------------------------------------- normalisation
def test_sinkhorn_closed_form():
    rows = dict((r[0], np.array(r[1].split(), dtype=float)) for r in _rows("sinkhorn_closed_form.txt"))
    rho, gamma = rows["rho"], rows["gamma"]
    i, j = np.meshgrid(np.arange(4), np.arange(4), indexing="ij")
    S = (-1.0) ** (i + j)
    Y = rho[:, None] * gamma[None, :] * S
    for T in (1, 2, 5):
        Z, r, c = codec.variance_normalize(Y, T)
        np.testing.assert_allclose(Z, S, atol=1e-14)
        np.testing.assert_allclose(r, rows["r"], rtol=1e-14)
        np.testing.assert_allclose(c, rows["c"], rtol=1e-14)


def test_normalize_reconstructs_exactly():
    """Y = diag(r) Z diag(c): the scales carry everything the normalisation
    removed."""
    rng = np.random.default_rng(3)
    Y = rng.standard_t(3, (128, 128)) * rng.exponential(2, 128)
    Z, r, c = codec.variance_normalize(Y, 2)
    np.testing.assert_allclose(r[:, None] * Z * c[None, :], Y, rtol=1e-12, atol=1e-12)


def test_normalize_T0_is_identity():
    Y = np.random.default_rng(4).standard_normal((64, 128))
    Z, r, c = codec.variance_normalize(Y, 0)
    np.testing.assert_array_equal(Z, Y)
    np.testing.assert_array_equal(r, np.ones(64))
    np.testing.assert_array_equal(c, np.ones(128))


@pytest.mark.parametrize("T", [1, 2, 3])
def test_normalize_rows_have_unit_std(T):
    """The last pass of every iteration is the row pass, so each token ends
    with population std exactly 1."""
    Y = np.random.default_rng(5).standard_normal((128, 256)) * 7
    Z, _, _ = codec.variance_normalize(Y, T)
    np.testing.assert_allclose(Z.std(axis=1), 1.0, rtol=1e-12)


def test_column_pass_gives_unit_column_std():
    Y = np.random.default_rng(6).standard_normal((128, 128)) * np.arange(1, 129)
    Z, ls = codec.column_pass(Y)
    np.testing.assert_allclose(Z.std(axis=0), 1.0, rtol=1e-12)
    np.testing.assert_allclose(np.exp(ls) * Z, Y, rtol=1e-12)


def test_normalize_columns_converge_toward_one():
    """Row and column stds converge toward 1 as iterations grow (the
    Sinkhorn-like alternation); measured on a heavy-tailed tile with
    per-channel and per-token scale spread."""
    rng = np.random.default_rng(7)
    Y = codec.rotate(rng.standard_t(3, (128, 128)) * rng.lognormal(0, 1, 128)
                     * rng.lognormal(0, 1, (128, 1)))
    dev = []
    for T in (1, 2, 4, 8):
        Z, _, _ = codec.variance_normalize(Y, T)
        dev.append(np.abs(Z.std(axis=0) - 1).max())
    assert all(b <= a * 1.0001 for a, b in zip(dev, dev[1:])), dev
    assert dev[-1] < 0.25 * dev[0]


def test_normalize_scale_equivariance():
    """Scaling the tile by alpha scales the product of the scales by alpha and
    leaves Z unchanged."""
    Y = np.random.default_rng(8).standard_normal((32, 64))
    Z1, r1, c1 = codec.variance_normalize(Y, 2)
    Z2, r2, c2 = codec.variance_normalize(Y * 8.0, 2)
    np.testing.assert_allclose(Z1, Z2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(np.outer(r2, c2), 8.0 * np.outer(r1, c1), rtol=1e-12)


def test_normalize_constant_vectors_keep_unit_scale():
    """A constant column (any value) and a constant row are left unscaled;
    the rounding residue of the mean does not count as spread."""
    rng = np.random.default_rng(13)
    Y = rng.standard_normal((128, 64))
    Y[:, 5] = 0.1 * 3 + 1e-3          # constant column, value not exact in binary
    Z, ls = codec.column_pass(Y)
    assert ls[5] == 0.0 and np.all(Z[:, 5] == Y[:, 5])
    R = np.tile(np.array([[7.3]]), (4, 32))
    Zr, lr = codec.row_pass(R)
    np.testing.assert_array_equal(lr, 0.0)
    np.testing.assert_array_equal(Zr, R)


def test_normalize_tiny_spread_is_not_constant():
    """Only an exactly constant vector keeps sigma = 1: a column or row whose
    entries differ by a relative 1e-9 has a genuine (tiny) standard deviation
    and is divided by it, so it leaves the pass with unit std like any other
    (the std definition of the four-stage paragraph of the KVarN review has
    no threshold)."""
    base = 5.0
    col = base * (1.0 + 1e-9 * np.array([-1.0, 1.0] * 8))  # population std 5e-9, mean 5
    Y = np.random.default_rng(17).standard_normal((16, 8))
    Y[:, 2] = col
    Z, ls = codec.column_pass(Y)
    s = np.std(col)
    assert s > 0 and ls[2] == np.log(s)
    np.testing.assert_allclose(np.std(Z[:, 2]), 1.0, rtol=1e-6)
    R = np.tile(col, (3, 2))
    Zr, lr = codec.row_pass(R)
    np.testing.assert_allclose(lr, np.log(s), rtol=1e-12)
    np.testing.assert_allclose(np.std(Zr, axis=1), 1.0, rtol=1e-6)


def test_normalize_zero_column_stays_finite():
    Y = np.random.default_rng(9).standard_normal((16, 8))
    Y[:, 3] = 0.0
    Z, r, c = codec.variance_normalize(Y, 2)
    assert np.isfinite(Z).all() and np.isfinite(r).all() and np.isfinite(c).all()
    assert (Z[:, 3] == 0).all() and c[3] == 1.0


# --------------------------------------------------------------- quantiser
def test_rtn_hand_worked_rows():
    for bits, vals, codes, lo, delta in _rows("rtn_rows.txt"):
        z = np.array(vals.split(), dtype=float)[None, :]
        c, l, d, _ = codec.rtn_rows(z, int(bits))
        np.testing.assert_array_equal(c[0], np.array(codes.split(), dtype=int))
        assert l[0] == float(lo)
        np.testing.assert_allclose(d[0], float(delta), rtol=1e-15)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_rtn_range_endpoints_and_error_bound(bits):
    Z = np.random.default_rng(bits).standard_normal((64, 128))
    codes, lo, delta, _ = codec.rtn_rows(Z, bits)
    qmax = 2 ** bits - 1
    assert codes.min() == 0 and codes.max() == qmax
    np.testing.assert_array_equal(codes[np.arange(64), Z.argmin(1)], 0)
    np.testing.assert_array_equal(codes[np.arange(64), Z.argmax(1)], qmax)
    err = np.abs(lo[:, None] + delta[:, None] * codes - Z)
    assert (err <= delta[:, None] / 2 * (1 + 1e-12)).all()
    # monotone: a larger value never gets a smaller code
    order = np.argsort(Z, axis=1)
    assert (np.diff(np.take_along_axis(codes, order, 1), axis=1) >= 0).all()


def test_reconstruction_error_shrinks_with_bits():
    """Reconstruction error falls as the width grows (gmlx page: widths 2..8;
    the two schemes converge at 8 bits)."""
    rng = np.random.default_rng(10)
    X = rng.standard_normal((128, 128))
    X[:, [7, 31, 64, 100]] *= 20
    errs = []
    for bits in (2, 3, 4, 5, 6, 8):
        e = codec.encode_tile(X, bits, 2)
        Xh = codec.dequantize(e["codes"], e["a"], e["b"], e["c"])
        errs.append(np.linalg.norm(Xh - X) / np.linalg.norm(X))
    assert all(b < a for a, b in zip(errs, errs[1:])), errs
    assert errs[-1] < 0.02


def test_dequantize_roundtrip_is_exact_without_rounding():
    """With the codes replaced by the exact quantiser input x, dequantisation
    returns the tile itself: the fold a = r delta, b = r lo and the inverse
    rotation lose nothing."""
    rng = np.random.default_rng(11)
    X = rng.standard_normal((128, 128)) * rng.lognormal(0, 1, 128)
    e = codec.encode_tile(X, 4, 2)
    np.testing.assert_allclose(codec.dequantize(e["x"], e["a"], e["b"], e["c"]), X,
                               rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("bits", [2, 4])
def test_kvarn_beats_plain_rtn_on_outliers(bits):
    """On tiles with outlier channels, rotation plus normalisation gives a
    smaller reconstruction error than plain per-token RTN at the same width
    (the point of the method: KVarN review, four-stage paragraph)."""
    rng = np.random.default_rng(12)
    X = rng.standard_normal((128, 128))
    X[:, rng.choice(128, 3, replace=False)] *= 20
    e = codec.encode_tile(X, bits, 2)
    err_kvarn = np.linalg.norm(codec.dequantize(e["codes"], e["a"], e["b"], e["c"]) - X)
    err_plain = np.linalg.norm(codec.rtn_plain_rows(X, bits) - X)
    assert err_kvarn < 0.8 * err_plain
