"""Rank-r key side codes (fp64 oracle): one mechanism behind two of the pages' methods.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

* [HeadQ] technical summary, section 3 (and 2.1): keys are read through logits, so the
  cache keeps, next to the base code of each key, a low-rank side code of its residual
  in a basis U_h (d x r, per head) learned by PCA of calibration queries. Cache write:
  e_j = k_j - k_hat_base_j, z_j = Q_q(U_h^T e_j). Cache read: the logit is
  q^T k_hat_base_j / sqrt(d) + q^T U_h z_hat_j / sqrt(d).
* [KVQuant++] "Core innovation 4" (低秩误差修正): the quantisation residual K - K_hat has
  its energy in a few singular directions; a rank-4 or rank-8 SVD reconstruction is
  added back (reported MSE -11 % / -19 %, about 6.3 % extra storage).

Both store per token the r coordinates of the residual in a per-head orthonormal basis
and add U_h z_hat back -- to the reconstruction (KVQuant++), hence to every logit
(HeadQ); they differ only in where the basis comes from: the principal directions of
calibration queries (HeadQ) or of the residuals themselves (KVQuant++, whose top right
singular vectors are the principal directions of the residual rows).

Readings where the pages are silent:

* the side quantiser Q_q is rounding to float16 (2r bytes per token): at r = 8 that is
  16 bytes against a 256-byte bf16 key, the 6.3 % KVQuant++ reports;
* "PCA" is taken about the origin (the principal directions of sum_j x_j x_j^T, no mean
  removed): the logit is linear in q, so a shared mean of the queries is a direction the
  correction must serve like any other;
* the sign of each basis vector is fixed so that its component of largest magnitude is
  positive (eigenvectors are defined up to sign; the convention makes U a function of the
  calibration data);
* side codes apply to unsketched key roles (the KV and KQV schemes), whose base
  reconstruction is nu D^T H^T c[idx] (or nu c[idx] unrotated).
"""

import numpy as np

from . import turboquant as tq


def principal_basis(X: np.ndarray, r: int) -> np.ndarray:
    """[d, r]: the r leading eigenvectors of X^T X (rows of X are samples), orthonormal
    columns ordered by decreasing eigenvalue, each signed so that its largest-magnitude
    component is positive."""
    X = np.asarray(X, dtype=np.float64)
    C = X.T @ X
    w, V = np.linalg.eigh(C)
    order = np.argsort(w)[::-1][:r]
    U = V[:, order]
    for j in range(r):
        i = int(np.argmax(np.abs(U[:, j])))
        if U[i, j] < 0:
            U[:, j] = -U[:, j]
    return U


def side_codes(x: np.ndarray, x_hat_base: np.ndarray, U: np.ndarray) -> np.ndarray:
    """[N, r] float16: Q_q(U^T (x - x_hat_base)) for each row."""
    e = np.asarray(x, dtype=np.float64) - np.asarray(x_hat_base, dtype=np.float64)
    return (e @ U).astype(np.float16)


def corrected(x_hat_base: np.ndarray, z: np.ndarray, U: np.ndarray) -> np.ndarray:
    """x_hat_base + U z_hat for each row (the side-corrected reconstruction)."""
    return np.asarray(x_hat_base, dtype=np.float64) + np.asarray(z, dtype=np.float64) @ U.T


def encode_keys(k: np.ndarray, role: "tq.Role", params: "tq.Params", U: np.ndarray):
    """Base code of the keys (as ``turboquant.encode``) plus their side codes."""
    if role.qjl:
        raise ValueError("side codes apply to unsketched key roles")
    enc = tq.encode(k, role, params)
    base = tq.decode(enc, params)
    return enc, side_codes(k, base, U)


def decode_keys(enc: "tq.Encoded", z: np.ndarray, params: "tq.Params", U: np.ndarray) -> np.ndarray:
    return corrected(tq.decode(enc, params), z, U)
