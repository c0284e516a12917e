"""Lloyd-Max scalar codebook fitted to the unit-sphere coordinate marginal.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

[KVQuant++] "Codebook design": the codebook is fitted to the true marginal of a
coordinate of a uniform point on the unit sphere, f(t) proportional to
(1 - t^2)^((d-3)/2) on [-1, 1]. [TQ-stats] "Theoretical framework" states the
same law as (t + 1)/2 ~ Beta((d-1)/2, (d-1)/2). [TQ-stats] "Quantisation
schemes" names the quantiser: scalar MSE (Lloyd-Max).

The fit is the textbook Lloyd iteration (Lloyd 1957 / Max 1960):
boundaries are midpoints of adjacent centroids, and each centroid is the
conditional mean of its cell. Cell masses come from the regularised incomplete
beta function (scipy.special.betainc, a library primitive). The cell first
moment has the closed form

    int_a^b t f(t) dt = C * ((1 - a^2)^((d-1)/2) - (1 - b^2)^((d-1)/2)) / (d - 1),
    C = 1 / B(1/2, (d-1)/2).

Initial centroids: the (i + 1/2)/L quantiles of N(0, 1/d). Iteration stops when
no centroid moves by more than 1e-15 (or, at very large d, when the step has
stopped shrinking at the fp64 noise floor); the result is then made exactly odd
(c[L-1-i] = -c[i]) so the middle boundary is exactly 0.

Storage reading (pages silent): the library holds the codebook in float32, the
fp64 values rounded to nearest; quantisation compares against the stored
float32 boundaries and reconstruction uses the stored float32 centroids. The
oracle does the same (``Codebook.centroids32`` / ``bounds32``), evaluated in
fp64 arithmetic.

Pinned by: fixed-point residuals checked with independent adaptive quadrature,
the 1-bit closed form, the large-d Gaussian limit (Max's table) and the
rate-distortion bound of [KVQuant++] "Rate-distortion performance"
(tests/test_oracle_codebook.py).
"""

from dataclasses import dataclass
from functools import lru_cache

import numpy as np
from scipy import special, stats


@dataclass(frozen=True)
class Codebook:
    d: int
    bits: int
    centroids: np.ndarray    # fp64, ascending, length 2^bits
    bounds: np.ndarray       # fp64, length 2^bits - 1 (midpoints)
    centroids32: np.ndarray  # float32 copies
    bounds32: np.ndarray
    masses: np.ndarray       # cell probabilities under f
    iterations: int

    @property
    def levels(self) -> int:
        return 1 << self.bits

    def mse_per_vector(self) -> float:
        """E||u - Q(u)||^2 for u uniform on S^{d-1}, coordinatewise Q.

        E[t^2] = 1/d per coordinate; with centroid = conditional mean the
        per-coordinate distortion is 1/d - sum_i P_i c_i^2, times d coordinates.
        """
        return float(1.0 - self.d * np.sum(self.masses * self.centroids ** 2))

    def cell_entropy_bits(self) -> float:
        p = self.masses[self.masses > 0]
        return float(-np.sum(p * np.log2(p)))


def _upper_tail(t: np.ndarray, d: int) -> np.ndarray:
    """P(T >= t) for the sphere marginal, via (1 - t)/2 ~ Beta(a, a)."""
    a = 0.5 * (d - 1)
    return special.betainc(a, a, np.clip((1.0 - t) * 0.5, 0.0, 1.0))


def cell_mass(lo: np.ndarray, hi: np.ndarray, d: int) -> np.ndarray:
    """P(lo <= T < hi), evaluated on the side of 0 that keeps precision."""
    lo = np.asarray(lo, dtype=np.float64)
    hi = np.asarray(hi, dtype=np.float64)
    pos = lo >= 0
    neg = hi <= 0
    mid = ~(pos | neg)
    out = np.empty(np.broadcast(lo, hi).shape)
    out[pos] = _upper_tail(lo[pos], d) - _upper_tail(hi[pos], d)
    out[neg] = _upper_tail(-hi[neg], d) - _upper_tail(-lo[neg], d)
    out[mid] = 1.0 - _upper_tail(hi[mid], d) - _upper_tail(-lo[mid], d)
    return out


def cell_first_moment(lo: np.ndarray, hi: np.ndarray, d: int) -> np.ndarray:
    """int_lo^hi t f(t) dt (closed form, see module docstring)."""
    e = 0.5 * (d - 1)
    log_c = -special.betaln(0.5, e)
    glo = np.power(np.maximum(1.0 - np.asarray(lo) ** 2, 0.0), e)
    ghi = np.power(np.maximum(1.0 - np.asarray(hi) ** 2, 0.0), e)
    return np.exp(log_c) * (glo - ghi) / (d - 1)


def density(t: np.ndarray, d: int) -> np.ndarray:
    """f(t) = (1 - t^2)^((d-3)/2) / B(1/2, (d-1)/2) on [-1, 1]."""
    t = np.asarray(t, dtype=np.float64)
    e = 0.5 * (d - 3)
    return np.exp(-special.betaln(0.5, 0.5 * (d - 1))) * np.power(np.maximum(1.0 - t * t, 0.0), e)


@lru_cache(maxsize=None)
def lloyd_max(d: int, bits: int, tol: float = 1e-15, max_iter: int = 400000) -> Codebook:
    """Fit the 2^bits-level Lloyd-Max quantiser for the dimension-d marginal."""
    if d < 4 or bits < 1 or bits > 8:
        raise ValueError("need d >= 4 and 1 <= bits <= 8")
    L = 1 << bits
    c = stats.norm.ppf((np.arange(L) + 0.5) / L) / np.sqrt(d)
    it = 0
    best, since_best = np.inf, 0
    for it in range(1, max_iter + 1):
        b = 0.5 * (c[:-1] + c[1:])
        edges = np.concatenate(([-1.0], b, [1.0]))
        m = cell_mass(edges[:-1], edges[1:], d)
        c_new = cell_first_moment(edges[:-1], edges[1:], d) / m
        step = np.max(np.abs(c_new - c))
        c = c_new
        if step < tol:
            break
        # at very large d the step can reach the fp64 noise floor of the
        # incomplete-beta differences before it reaches tol: stop there
        if step < best:
            best, since_best = step, 0
        else:
            since_best += 1
            if since_best > 2000:
                break
    c = 0.5 * (c - c[::-1])  # exact odd symmetry
    b = 0.5 * (c[:-1] + c[1:])
    b[L // 2 - 1] = 0.0
    edges = np.concatenate(([-1.0], b, [1.0]))
    masses = cell_mass(edges[:-1], edges[1:], d)
    c.setflags(write=False)
    b.setflags(write=False)
    return Codebook(d=d, bits=bits, centroids=c, bounds=b,
                    centroids32=c.astype(np.float32), bounds32=b.astype(np.float32),
                    masses=masses, iterations=it)
