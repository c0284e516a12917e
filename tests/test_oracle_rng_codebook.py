"""Pins for the oracle's method randomness and Lloyd-Max codebook (CPU only).

Each check compares the oracle with something other than itself: a published
test vector, an independent quadrature, a closed form, a textbook table or a
bound the pages print.
"""

import math

import numpy as np
import pytest
from scipy import integrate, special, stats

from conftest import read_golden
from oracle import codebook as cb
from oracle import rng


# ---------------------------------------------------------------- SplitMix64

def test_splitmix64_published_stream():
    want = [int(r[0]) for r in read_golden("splitmix64_seed1234567.txt")]
    # stream 0, counters 1..5 from seed 1234567 are the sequential outputs
    got = [rng.draw(1234567, 0, i) for i in range(5)]
    assert got == want


def test_counter_form_equals_sequential_generator():
    seed = 0xDEADBEEF12345678
    state = seed
    seq = []
    for _ in range(40):
        state = (state + rng.GAMMA) & ((1 << 64) - 1)
        seq.append(rng.mix64(state))
    assert [rng.draw(seed, 0, i) for i in range(40)] == seq


def test_diagonal_is_balanced_rademacher():
    d = 128
    D = np.stack([rng.rademacher_diagonal(s, d) for s in range(64)])
    assert set(np.unique(D).tolist()) == {-1, 1}
    # mean of 8192 fair signs: |mean| < 4 / sqrt(8192)
    assert abs(D.mean()) < 4 / math.sqrt(D.size)
    # different seeds give different diagonals
    assert len({D[i].tobytes() for i in range(64)}) == 64


def test_sketch_is_standard_gaussian():
    S = rng.gaussian_sketch(42, 128).astype(np.float64).ravel()
    assert S.size == 128 * 128
    assert abs(S.mean()) < 4 / math.sqrt(S.size)
    assert abs(S.var() - 1.0) < 4 * math.sqrt(2.0 / S.size)
    assert stats.kstest(S, "norm").pvalue > 1e-3


# ---------------------------------------------------------------- codebook

@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_lloyd_max_fixed_point_by_independent_quadrature(d, bits):
    """Each centroid is the conditional mean of its cell, each boundary a midpoint.

    The conditional means are recomputed with adaptive Gauss-Kronrod quadrature
    of the density itself (not the incomplete beta / closed form the fit uses).
    """
    C = cb.lloyd_max(d, bits)
    c, b = C.centroids, C.bounds
    assert np.all(np.diff(c) > 0)
    np.testing.assert_allclose(b, 0.5 * (c[:-1] + c[1:]), rtol=0, atol=1e-15)
    edges = np.concatenate(([-1.0], b, [1.0]))
    f = lambda t: cb.density(t, d)
    for i in range(C.levels):
        lo, hi = edges[i], edges[i + 1]
        mass = integrate.quad(f, lo, hi, epsabs=1e-17, epsrel=1e-13, limit=200)[0]
        mom = integrate.quad(lambda t: t * f(t), lo, hi, epsabs=1e-17, epsrel=1e-13, limit=200)[0]
        assert abs(mom / mass - c[i]) < 1e-12 * max(1.0, abs(c[i]) * 10)
        assert abs(mass - C.masses[i]) < 1e-12


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_is_odd_symmetric(bits):
    C = cb.lloyd_max(128, bits)
    np.testing.assert_array_equal(C.centroids, -C.centroids[::-1])
    np.testing.assert_array_equal(C.centroids32, -C.centroids32[::-1])
    assert C.bounds[C.levels // 2 - 1] == 0.0


@pytest.mark.parametrize("d", [16, 128, 1024])
def test_one_bit_closed_form(d):
    """E[t | t > 0] = Gamma(d/2) / (sqrt(pi) Gamma((d+1)/2)) for the sphere marginal."""
    want = math.exp(special.gammaln(d / 2) - special.gammaln((d + 1) / 2)) / math.sqrt(math.pi)
    C = cb.lloyd_max(d, 1)
    assert abs(C.centroids[1] - want) < 1e-14
    if d == 128:
        assert abs(math.sqrt(d) * want - 0.79944) < 1e-5


@pytest.mark.parametrize("row", read_golden("max1960_gaussian.txt"))
def test_large_d_limit_is_max_gaussian_table(row):
    bits = int(row[0])
    want = np.array([float(x) for x in row[1:]])
    C = cb.lloyd_max(16384, bits)
    got = math.sqrt(16384) * C.centroids[C.levels // 2:]
    # the marginal differs from the Gaussian by O(1/d); Max's table has 4 digits
    np.testing.assert_allclose(got, want, atol=2e-3)


def test_mse_within_the_pages_rate_distortion_bound():
    claims = {r[0]: float(r[1]) for r in read_golden("page_claims.txt")}
    read = claims["mse_bound_constant_read"]
    for d in (64, 128, 256, 1024):
        for bits in (1, 2, 3, 4):
            mse = cb.lloyd_max(d, bits).mse_per_vector()
            assert 0 < mse <= read * 4.0 ** -bits, (d, bits, mse)
    # the constant as literally printed, sqrt(3 pi / 2), holds only for b <= 2 at d = 128
    lit = claims["mse_bound_constant_literal"]
    holds = [cb.lloyd_max(128, b).mse_per_vector() <= lit * 4.0 ** -b for b in (1, 2, 3, 4)]
    assert holds == [True, True, False, False]


def test_mse_matches_monte_carlo_of_the_quantiser():
    """E||u - Q(u)||^2 from the cell masses equals a Monte-Carlo average over sphere points."""
    g = np.random.default_rng(5)
    d = 128
    u = g.standard_normal((40000, d))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    for bits in (2, 4):
        C = cb.lloyd_max(d, bits)
        idx = np.searchsorted(C.bounds, u, side="right")
        err = np.sum((u - C.centroids[idx]) ** 2, axis=1)
        assert abs(err.mean() - C.mse_per_vector()) < 5 * err.std() / math.sqrt(len(err))


def test_entropy_saving_matches_the_pages_claim():
    claims = {r[0]: float(r[1]) for r in read_golden("page_claims.txt")}
    H = cb.lloyd_max(128, 4).cell_entropy_bits()
    saving = 1.0 - H / 4.0
    assert abs(H - 3.774) < 1e-3
    # "about 5%": the exact cell entropy leaves 5.7% to an ideal entropy coder
    assert abs(saving - claims["entropy_saving_4bit_d128"]) < 0.01


def test_marginal_beta_law_monte_carlo():
    """Coordinates of uniform sphere points: (t+1)/2 ~ Beta((d-1)/2, (d-1)/2)."""
    g = np.random.default_rng(11)
    d = 128
    u = g.standard_normal((20000, d))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    t = u[:, 3]
    a = (d - 1) / 2
    assert stats.kstest((t + 1) / 2, stats.beta(a, a).cdf).pvalue > 1e-3
    assert abs(t.mean()) < 4 * math.sqrt(1 / d / len(t))
    assert abs(t.var() - 1 / d) < 0.05 / d
    # the oracle's mass function is that law's CDF
    x = np.linspace(-0.3, 0.3, 13)
    np.testing.assert_allclose(cb.cell_mass(np.full_like(x, -1.0), x, d), stats.beta(a, a).cdf((x + 1) / 2),
                               atol=1e-13)
