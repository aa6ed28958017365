"""KVarN per-tile codec, restated in float64 (test infrastructure only).

Sources. "KVarN ... vLLM KV cache quantization" review, paragraph on the
four-stage quantisation. Restated: a tile of raw keys or values is turned by
an orthonormal Hadamard matrix acting on its channels (scores do not change,
and the energy of an outlier channel is shared among all channels); its
columns and rows are then rescaled in turn by their standard deviations, a
Sinkhorn-style alternation whose scales are accumulated as logarithms;
finally every row is rounded to the nearest level of an asymmetric grid, and
the scales are multiplied back in when the cache is read. The gmlx "KV cache
quantization" page, section "The two schemes", describes the same codec as a
Hadamard rotation of each head followed by 128-token records whose scaling
keeps any single token or channel from dominating.

Readings where the pages leave a step open (each also listed in the design
notes):
  * H is the Sylvester Hadamard matrix in natural order scaled by 1/sqrt(D):
    symmetric and orthonormal, so H @ H = I and the inverse rotation is H.
  * One normalisation iteration is a column pass then a row pass. A pass
    divides by the population standard deviation (ddof=0) about the mean and
    adds log(sigma) to the running log-scale; scales leave log space once, at
    the end. A constant vector (all of its entries equal, so that its
    standard deviation is zero by definition) or one whose sigma is not
    finite keeps sigma = 1. The test is exact: a vector whose entries differ
    at all is normalised, however small its spread.
  * Quantisation is per token row of the normalised tile: lo = min, hi = max,
    delta = (hi - lo) / (2^bits - 1), code = clamp(rint((z - lo) / delta)),
    rint being round-half-to-even. A row with hi == lo gets delta = 0 and all
    codes 0. The row scale r folds into a = r * delta and b = r * lo; the
    column scale c stays separate, so the dequantised rotated value is
    y_hat[i, j] = c[j] * (a[i] * code[i, j] + b[i]).
"""
from __future__ import annotations

import numpy as np


def hadamard(D: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order D (a power of two), scaled by 1/sqrt(D).

    KVarN review, four-stage paragraph (stage two, the orthonormal rotation of
    the channels). Built by the doubling rule H_2n = [[H, H], [H, -H]] from
    H_1 = [1].
    """
    if D < 1 or D & (D - 1):
        raise ValueError("Hadamard order must be a power of two")
    H = np.ones((1, 1), dtype=np.float64)
    while H.shape[0] < D:
        H = np.block([[H, H], [H, -H]])
    return H / np.sqrt(D)


def rotate(X: np.ndarray) -> np.ndarray:
    """Y = X H: every token row rotated across its D channels (same review,
    stage two). Works on [..., D]."""
    X = np.asarray(X, dtype=np.float64)
    return X @ hadamard(X.shape[-1])


def pop_std(Z: np.ndarray, axis: int) -> np.ndarray:
    """Population standard deviation along ``axis``; 1 for a constant vector
    (max == min: its standard deviation is zero by definition, whatever
    rounding residue the float64 mean leaves) or a non-finite std."""
    s = np.std(Z, axis=axis, ddof=0)
    constant = np.max(Z, axis=axis) == np.min(Z, axis=axis)
    return np.where(np.isfinite(s) & ~constant & (s > 0), s, 1.0)


def column_pass(Z: np.ndarray):
    """Divide every channel (column) by its std over the tile's tokens.
    Returns (Z', log sigma_c)."""
    s = pop_std(Z, axis=0)
    return Z / s[None, :], np.log(s)


def row_pass(Z: np.ndarray):
    """Divide every token (row) by its std over the channels.
    Returns (Z', log sigma_r)."""
    s = pop_std(Z, axis=1)
    return Z / s[:, None], np.log(s)


def variance_normalize(Y: np.ndarray, T: int):
    """Sinkhorn-like alternation of column- and row-wise std normalisation with
    the scales kept in log space (KVarN review, stage three; T iterations, one
    iteration = column pass then row pass).

    Returns (Z, r, c) with Y = diag(r) Z diag(c).
    """
    Z = np.array(Y, dtype=np.float64)
    N, D = Z.shape
    log_r = np.zeros(N)
    log_c = np.zeros(D)
    for _ in range(T):
        Z, lc = column_pass(Z)
        log_c += lc
        Z, lr = row_pass(Z)
        log_r += lr
    return Z, np.exp(log_r), np.exp(log_c)


def rtn_rows(Z: np.ndarray, bits: int):
    """Asymmetric round-to-nearest of every row to ``bits``-bit codes (KVarN
    review, stage four). Returns (codes int64, lo, delta, x) where
    x = (z - lo) / delta is the quantiser input before rounding (kept for the
    boundary-distance bookkeeping of the parity tests)."""
    qmax = (1 << bits) - 1
    lo = Z.min(axis=1)
    hi = Z.max(axis=1)
    delta = (hi - lo) / qmax
    safe = np.where(delta > 0, delta, 1.0)
    x = (Z - lo[:, None]) / safe[:, None]
    x = np.where(delta[:, None] > 0, x, 0.0)
    codes = np.clip(np.rint(x), 0, qmax).astype(np.int64)
    return codes, lo, np.where(delta > 0, delta, 0.0), x


def encode_tile(X: np.ndarray, bits: int, T: int) -> dict:
    """All four stages on one N x D tile of one KV head.

    Returns a dict with the stored quantities (codes, a, b, c, all float64
    before the page stores a, b, c as fp32) and the intermediates Y, Z, r,
    lo, delta and x.
    """
    Y = rotate(X)
    Z, r, c = variance_normalize(Y, T)
    codes, lo, delta, x = rtn_rows(Z, bits)
    return dict(codes=codes, a=r * delta, b=r * lo, c=c,
                Y=Y, Z=Z, r=r, lo=lo, delta=delta, x=x)


def dequantize_rotated(codes, a, b, c) -> np.ndarray:
    """y_hat[i, j] = c[j] * (a[i] * code[i, j] + b[i]): the scales folded back
    in at read time (KVarN review, stage four), still in the rotated basis."""
    codes = np.asarray(codes, dtype=np.float64)
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    return c[None, :] * (a[:, None] * codes + b[:, None])


def dequantize(codes, a, b, c) -> np.ndarray:
    """Dequantised tile back in the original channel basis: y_hat H (H is its
    own inverse)."""
    Yh = dequantize_rotated(codes, a, b, c)
    return Yh @ hadamard(Yh.shape[-1])


def rtn_plain_rows(X: np.ndarray, bits: int) -> np.ndarray:
    """Plain per-token asymmetric RTN without rotation or normalisation, used
    only by the fidelity tests as the no-KVarN baseline. Returns the
    reconstruction."""
    codes, lo, delta, _ = rtn_rows(np.asarray(X, dtype=np.float64), bits)
    return lo[:, None] + delta[:, None] * codes
