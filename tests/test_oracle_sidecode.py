"""Pins of the oracle's rank-r key side codes (oracle/sidecode.py) against what the
mathematics fixes: the principal basis against an SVD, the exact logit recovery when
queries lie in the basis ([HeadQ] section 3), the Eckart-Young residual of the
low-rank correction ([KVQuant++] "Core innovation 4"), and the "wrong sign" control
of [HeadQ] "Main contributions". CPU only."""

import numpy as np
import pytest

from oracle import sidecode as sc
from oracle import turboquant as otq
from quantised_kv_cache_gb300 import workloads as wl


def test_principal_basis_is_the_svd_right_basis():
    g = np.random.default_rng(0)
    X = g.standard_normal((500, 16)) @ np.diag(np.linspace(3, 0.1, 16)) @ np.linalg.qr(g.standard_normal((16, 16)))[0]
    U = sc.principal_basis(X, 5)
    _, _, Vt = np.linalg.svd(X, full_matrices=False)
    np.testing.assert_allclose(U.T @ U, np.eye(5), atol=1e-12)
    for j in range(5):
        v = Vt[j] * np.sign(Vt[j][np.argmax(np.abs(Vt[j]))])
        np.testing.assert_allclose(U[:, j], v, atol=1e-10)
        assert U[np.argmax(np.abs(U[:, j])), j] > 0


def test_principal_basis_recovers_an_exact_rank_r_row_space():
    g = np.random.default_rng(1)
    B = np.linalg.qr(g.standard_normal((32, 4)))[0]
    X = g.standard_normal((200, 4)) @ B.T
    U = sc.principal_basis(X, 4)
    np.testing.assert_allclose(U @ U.T, B @ B.T, atol=1e-10)  # the same subspace


@pytest.mark.parametrize("scheme,n", [("KQV", 2), ("KV", 2), ("KQV", 4)])
def test_queries_in_the_basis_recover_the_exact_logits(scheme, n):
    # HeadQ's correction with U spanning the queries: q^T (k_hat + U U^T (k - k_hat)) = q^T k,
    # up to the float16 rounding of the side code
    g = np.random.default_rng(2)
    d, N = 128, 400
    basis = np.linalg.qr(g.standard_normal((d, 4)))[0]
    q = g.standard_normal((50, 4)) @ basis.T
    k = g.standard_normal((N, d)) * 2.0
    p = otq.make_params(d, n, scheme, 3)
    role = p.roles()[0]
    U = sc.principal_basis(q, 4)
    enc, z = sc.encode_keys(k, role, p, U)
    kc = sc.decode_keys(enc, z, p, U)
    base = otq.decode(enc, p)
    exact = q @ k.T
    err_base = np.abs(q @ base.T - exact).max()
    err_corr = np.abs(q @ kc.T - exact).max()
    # fp16 rounding of z: |z| <= ||e||, relative 2^-11
    bound = np.max(np.linalg.norm(q, axis=1)) * np.max(np.linalg.norm(k - base, axis=1)) * 2.0 ** -10
    assert err_corr <= bound
    assert err_corr < 0.01 * err_base


def test_low_rank_correction_meets_eckart_young():
    # with U the top-r right singular vectors of the residual matrix E, the corrected
    # residual E - E U U^T has squared Frobenius norm sum_{i > r} sigma_i^2 (exact codes);
    # the float16 codes add at most their own rounding
    w = wl.WORKLOADS[3]
    _, k, _ = wl.generate(w, "cpu", seed=7, key_dist="lowrank", batch=1, heads_kv=1, heads_q=1, seq=2000)
    k = k[0, 0].double().numpy()
    p = otq.make_params(128, 2, "KQV", 9)
    role = p.roles()[0]
    enc = otq.encode(k, role, p)
    E = k - otq.decode(enc, p)
    s = np.linalg.svd(E, compute_uv=False)
    for r in (4, 8):
        U = sc.principal_basis(E, r)
        Ec = E - (E @ U) @ U.T
        np.testing.assert_allclose(np.sum(Ec ** 2), np.sum(s[r:] ** 2), rtol=1e-9)
        enc2, z = sc.encode_keys(k, role, p, U)
        got = k - sc.decode_keys(enc2, z, p, U)
        assert abs(np.sum(got ** 2) - np.sum(s[r:] ** 2)) <= 1e-3 * np.sum(E ** 2)
        assert np.sum(got ** 2) < np.sum(E ** 2)


def test_wrong_sign_correction_hurts_and_right_sign_helps():
    # [HeadQ]: flipping the sign of the correction is catastrophic; the right sign cuts the
    # attention KL. Rank-4 keys with 64 queries of their subspace (one seed, one basis):
    # queries 1..63 calibrate a rank-4 basis, query 0 is evaluated; 2-bit KQV keys
    w = wl.WORKLOADS[3]
    q, k, _ = wl.generate(w, "cpu", seed=11, key_dist="lowrank", batch=1, heads_kv=1, heads_q=64, seq=1024)
    qs = q[0].double().numpy()
    k64 = k[0, 0].double().numpy()
    p = otq.make_params(128, 2, "KQV", 5)
    U = sc.principal_basis(qs[1:], 4)
    enc, z = sc.encode_keys(k64, p.roles()[0], p, U)
    base = otq.decode(enc, p)

    def kl(Kh):
        s, sh = k64 @ qs[0] / np.sqrt(128), Kh @ qs[0] / np.sqrt(128)
        pp = np.exp(s - s.max())
        pp /= pp.sum()
        ph = np.exp(sh - sh.max())
        ph /= ph.sum()
        return float(np.sum(pp * np.log(pp / ph)))
    k_base, k_right, k_wrong = kl(base), kl(sc.decode_keys(enc, z, p, U)), kl(sc.decode_keys(enc, -z, p, U))
    assert k_right < 0.01 * k_base, (k_right, k_base)
    assert k_wrong > k_base, (k_wrong, k_base)
