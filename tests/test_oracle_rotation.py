"""Pins of the oracle's dense SO(d) rotation (oracle/rotation.py) against what the
pages and the mathematics fix ([KVQuant++] "Rotation-invariance guarantee":
determinant +1; "Rate-distortion performance": QR or Hadamard rotation, the same
distortion). CPU only."""

import math

import numpy as np
import pytest
from scipy import stats

from oracle import codebook as cb
from oracle import rng
from oracle import rotation as rot
from oracle import turboquant as tq


def _gram_schmidt(G):
    """Columns of G orthonormalised in order (classical Gram-Schmidt, each column
    projected twice): the Q of G = QR with a positive diagonal, computed a second way."""
    d = G.shape[0]
    Q = np.zeros_like(G)
    for j in range(d):
        v = G[:, j].copy()
        for _ in range(2):
            v -= Q[:, :j] @ (Q[:, :j].T @ v)
        Q[:, j] = v / np.linalg.norm(v)
    return Q


def test_gaussian_entries_follow_the_counter_recipe():
    # entry k of the matrix is Box-Muller (cosine branch) on words 2k, 2k+1 of stream 3
    G = rot.gaussian_matrix(5, 8)
    for k in (0, 9, 63):
        w1, w2 = rng.draw(5, 3, 2 * k), rng.draw(5, 3, 2 * k + 1)
        u1 = ((w1 >> 11) + 1) * 2.0 ** -53
        u2 = (w2 >> 11) * 2.0 ** -53
        assert G.reshape(-1)[k] == math.sqrt(-2 * math.log(u1)) * math.cos(2 * math.pi * u2)
    assert rot.STREAM_ROTATION not in (rng.STREAM_DIAG, rng.STREAM_SKETCH)


@pytest.mark.parametrize("d", [8, 128])
def test_rotation_is_special_orthogonal(d):
    M = rot.dense_rotation(7, d)
    np.testing.assert_allclose(M.T @ M, np.eye(d), atol=1e-13)
    np.testing.assert_allclose(M @ M.T, np.eye(d), atol=1e-13)
    assert abs(np.linalg.det(M) - 1.0) < 1e-12
    x = np.random.default_rng(1).standard_normal((50, d))
    np.testing.assert_allclose(np.linalg.norm(x @ M.T, axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)


@pytest.mark.parametrize("seed", [0, 1, 2, 3, 11])
def test_rotation_is_the_sign_fixed_qr_of_the_seeded_gaussian(seed):
    # M^T's columns are Gram-Schmidt's basis of G's columns, except that the last one is
    # negated exactly when that basis is a reflection (det G < 0)
    d = 16
    G = rot.gaussian_matrix(seed, d)
    Q = _gram_schmidt(G)
    M = rot.dense_rotation(seed, d)
    np.testing.assert_allclose(M.T[:, :-1], Q[:, :-1], atol=1e-11)
    flip = -1.0 if np.linalg.det(G) < 0 else 1.0
    np.testing.assert_allclose(M.T[:, -1], flip * Q[:, -1], atol=1e-11)


def test_rotations_over_seeds_are_haar_on_so_d():
    # a fixed direction lands uniformly on the sphere: its coordinates follow the
    # Beta((d-1)/2, (d-1)/2) marginal the codebook is fitted to; about half of the draws
    # needed the reflection fixed; every determinant is +1
    d, n = 16, 1500
    e1 = np.zeros(d)
    e1[0] = 1.0
    ys, flips = [], 0
    for s in range(n):
        M = rot.dense_rotation(1000 + s, d)
        assert abs(np.linalg.det(M) - 1.0) < 1e-12
        ys.append(M @ e1)
        flips += np.linalg.det(rot.gaussian_matrix(1000 + s, d)) < 0
    ys = np.array(ys)
    a = (d - 1) / 2
    for j in (0, 5, d - 1):
        assert stats.kstest((ys[:, j] + 1) / 2, stats.beta(a, a).cdf).pvalue > 1e-3
    assert abs(flips / n - 0.5) < 4 * math.sqrt(0.25 / n)
    np.testing.assert_allclose(np.mean(ys ** 2, axis=0), 1 / d, atol=6 * math.sqrt(2 / (d * d * n)))


def test_dense_rotation_gives_the_codebook_distortion_like_the_hadamard():
    # "QR or Hadamard": after either rotation the per-vector MSE is the sphere-marginal
    # Lloyd-Max distortion (vectors with very unequal channel scales, where no rotation
    # would leave the marginal far from the fitted one)
    g = np.random.default_rng(8)
    x = g.standard_normal((3000, 128)) * np.exp(g.standard_normal(128))[None, :]
    u = x / np.linalg.norm(x, axis=1, keepdims=True)
    for rotation in ("wht", "dense"):
        p = tq.make_params(128, 4, "KQV", 21, rotation=rotation)
        for bits in (2, 3, 4):
            e = tq.encode(x, tq.Role(bits, True, False), p)
            xh = tq.decode(e, p) / e.norm.astype(np.float64)[:, None]
            err = np.sum((u - xh) ** 2, axis=1)
            want = cb.lloyd_max(128, bits).mse_per_vector()
            assert abs(err.mean() - want) < 0.1 * want, (rotation, bits)


def test_dense_params_rotate_and_unrotate_are_inverse_and_differ_from_the_hadamard():
    p = tq.make_params(128, 3, "QKQV", 5, rotation="dense")
    w = tq.make_params(128, 3, "QKQV", 5)
    x = np.random.default_rng(2).standard_normal((10, 128))
    np.testing.assert_allclose(p.unrotate(p.rotate(x)), x, atol=1e-13)
    assert np.max(np.abs(p.rotate(x) - w.rotate(x))) > 0.1
    # the sketched reconstruction stays unbiased through the dense rotation
    role = tq.Role(2, True, True)
    e = tq.encode(x, role, p)
    assert e.signs is not None and np.all(np.isfinite(tq.decode(e, p)))
