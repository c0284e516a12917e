"""TurboQuant-style vector quantisation of K/V cache vectors (fp64 oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What each step follows:

* normalise, keep the norm in float32 -- [TQ-stats] "Theoretical framework"
  (the codebook is defined for unit-sphere coordinates) and [KVQuant++]
  "Codebook design";
* randomised Walsh-Hadamard rotation y = H_d D u, D a seeded +/-1 diagonal,
  H_d the orthonormal Sylvester Hadamard matrix in natural order --
  [TQ-stats] "Quantisation schemes" (KQV and QKQV apply a WHT to both K and V)
  and "Low-rank pathology" (the WHT makes the marginals Beta-shaped);
* scalar Lloyd-Max codes, found by counting the boundaries at or below each
  coordinate (bucketize, [KVQuant++] "Fast codebook lookup");
* the 1-bit QJL sketch sign(S r) of the residual r = y - c[idx], with S a
  seeded Gaussian d x d matrix and the residual norm stored --
  [TQ-stats] "Quantisation schemes" and "Main contribution 1" (the estimator
  of <., r> has variance (pi/2) ||r||^2 / d, so the sketch has m = d rows);
* the three equal-budget schemes of [TQ-stats] "Quantisation schemes":
  KV   -- K and V: n-bit Lloyd-Max, no rotation, no sketch;
  KQV  -- WHT on both; K n-bit; V (n-1)-bit + 1-bit QJL;
  QKQV -- WHT on both; K and V (n-1)-bit + 1-bit QJL.

Readings where the pages are silent:

* n bits are per coordinate; norms are float32 side data.
* KV uses the same sphere-marginal codebook on unrotated unit coordinates.
* ties go to the upper cell (idx = #{j : y >= b_j}); sign(0) = +1.
* the sign is taken of S applied to the unit-domain residual; the stored
  residual norm is rho = ||x|| * ||r_unit||, so a token's QJL weight is
  p_j * rho_j.
* dequantisation does not renormalise: x_hat = nu * D H c[idx]
  (+ rho sqrt(pi/2)/m * D H S^T sigma for sketched vectors).
* a zero vector stores nu = 0, the codes of y = 0, all sign bits 1, rho = 0.

Storage format (the library's, stated in include/tq.h and restated here): the
vector's d coordinates form d/2 pairs (2p, 2p+1); pair p = 4n + t (t = p mod 4)
sits in slot (d/8) t + n, so coordinate i = 8n + 2t + e (e = i mod 2) has its
b-bit code at bit offset b ((d/4) t + 2n + e) of the record's little-endian
bit string (string bit k is bit k % 8 of byte k // 8). Sign bits use the same
offsets with b = 1. For d = 8 this is the natural order.
"""

from dataclasses import dataclass
from typing import Optional

import math

import numpy as np
from scipy.linalg import hadamard as _scipy_hadamard

from . import codebook as _cb
from . import rng as _rng
from . import rotation as _rot

SCHEMES = ("KV", "KQV", "QKQV")
SQRT_HALF_PI = math.sqrt(math.pi / 2.0)


def hadamard(d: int) -> np.ndarray:
    """Orthonormal Sylvester Hadamard H_d (natural order): H_{ij} = (-1)^{popcount(i&j)} / sqrt(d)."""
    return _scipy_hadamard(d).astype(np.float64) / math.sqrt(d)


@dataclass(frozen=True)
class Role:
    """How one of K or V is coded under a scheme."""
    bits: int
    rotate: bool
    qjl: bool


def scheme_roles(scheme: str, n: int):
    """(K role, V role) for an n-bit-per-coordinate budget ([TQ-stats] "Quantisation schemes")."""
    if scheme == "KV":
        r = Role(n, False, False)
        return r, r
    if scheme == "KQV":
        return Role(n, True, False), Role(n - 1, True, True)
    if scheme == "QKQV":
        r = Role(n - 1, True, True)
        return r, r
    raise ValueError(scheme)


@dataclass(frozen=True)
class Params:
    """The quantiser state a context holds: D, S, the rotation and the codebooks it needs."""
    d: int
    n: int
    scheme: str
    seed: int
    D: np.ndarray   # int8 +/-1, length d
    S: np.ndarray   # float32, d x d
    rotation: str = "wht"             # "wht": y = H D u; "dense": y = M u, M in SO(d)
    M: Optional[np.ndarray] = None    # the dense rotation (fp64), rotation == "dense"

    def codebook(self, bits: int) -> _cb.Codebook:
        return _cb.lloyd_max(self.d, bits)

    def roles(self):
        return scheme_roles(self.scheme, self.n)

    def rotate(self, u: np.ndarray) -> np.ndarray:
        """Rows u -> rows y of the rotated roles."""
        if self.rotation == "dense":
            return u @ self.M.T
        H = hadamard(self.d)
        return (u * self.D.astype(np.float64)[None, :]) @ H.T

    def unrotate(self, y: np.ndarray) -> np.ndarray:
        """Rows y -> rows of the original domain (the transpose of `rotate`)."""
        if self.rotation == "dense":
            return y @ self.M
        H = hadamard(self.d)
        return (y @ H.T) * self.D.astype(np.float64)[None, :]


def make_params(d: int, n: int, scheme: str, seed: int, rotation: str = "wht") -> Params:
    if scheme not in SCHEMES:
        raise ValueError(scheme)
    if d & (d - 1) or d < 4:
        raise ValueError("d must be a power of two")
    if not 2 <= n <= 4:
        raise ValueError("budget n must be 2..4 (the sketched schemes need n-1 >= 1)")
    if rotation not in ("wht", "dense"):
        raise ValueError(rotation)
    M = _rot.dense_rotation(seed, d) if rotation == "dense" else None
    return Params(d=d, n=n, scheme=scheme, seed=seed,
                  D=_rng.rademacher_diagonal(seed, d), S=_rng.gaussian_sketch(seed, d), rotation=rotation, M=M)


@dataclass
class Encoded:
    """Quantised vectors: norms, integer codes, optional QJL signs and residual norms."""
    role: Role
    norm: np.ndarray                    # float32 [N]
    idx: np.ndarray                     # int64 [N, d]
    signs: Optional[np.ndarray] = None  # bool [N, d] (True = +1)
    rnorm: Optional[np.ndarray] = None  # float32 [N]
    # fp64 values at which each decision was taken (for the boundary-band rule)
    y: Optional[np.ndarray] = None      # the coordinates that were bucketized
    z: Optional[np.ndarray] = None      # S @ r_unit, whose signs were kept


def encode(x: np.ndarray, role: Role, params: Params) -> Encoded:
    """Quantise the rows of x (any float dtype; taken exactly into fp64)."""
    x = np.asarray(x, dtype=np.float64)
    N, d = x.shape
    assert d == params.d
    cb = params.codebook(role.bits)
    nu = np.sqrt(np.sum(x * x, axis=1))
    zero = nu == 0.0
    u = np.zeros_like(x)
    u[~zero] = x[~zero] / nu[~zero, None]
    if role.rotate:
        y = params.rotate(u)
    else:
        y = u
    bounds = cb.bounds32.astype(np.float64)
    idx = np.sum(y[:, :, None] >= bounds[None, None, :], axis=2).astype(np.int64)
    enc = Encoded(role=role, norm=nu.astype(np.float32), idx=idx, y=y)
    if role.qjl:
        c = cb.centroids32.astype(np.float64)
        r = y - c[idx]
        z = r @ params.S.astype(np.float64).T
        signs = z >= 0.0
        rho = nu * np.sqrt(np.sum(r * r, axis=1))
        signs[zero] = True
        rho[zero] = 0.0
        enc.signs = signs
        enc.rnorm = rho.astype(np.float32)
        enc.z = z
    return enc


def decode(enc: Encoded, params: Params) -> np.ndarray:
    """Reconstruct fp64 vectors from codes, norms and (optionally) signs."""
    role = enc.role
    d = params.d
    cb = params.codebook(role.bits)
    c = cb.centroids32.astype(np.float64)
    yhat = enc.norm.astype(np.float64)[:, None] * c[enc.idx]
    if role.qjl:
        sig = np.where(enc.signs, 1.0, -1.0)
        m = params.S.shape[0]
        yhat = yhat + (SQRT_HALF_PI / m) * enc.rnorm.astype(np.float64)[:, None] * (sig @ params.S.astype(np.float64))
    if role.rotate:
        yhat = params.unrotate(yhat)
    return yhat


# ----------------------------------------------------------------------------
# storage format
# ----------------------------------------------------------------------------

def slot_order(d: int) -> np.ndarray:
    """Position (in units of one code) of coordinate i in the record: (d/4) t + 2n + e."""
    if d % 8:
        raise ValueError("d must be a multiple of 8")
    i = np.arange(d)
    n, t, e = i >> 3, (i >> 1) & 3, i & 1
    return (d // 4) * t + 2 * n + e


def pack_codes(idx: np.ndarray, bits: int) -> np.ndarray:
    """[N, d] integer codes -> [N, bits*d/8] bytes in the slot order above."""
    idx = np.asarray(idx, dtype=np.int64)
    N, d = idx.shape
    pos = slot_order(d)
    stream = np.zeros((N, d * bits), dtype=np.uint8)
    for k in range(bits):
        stream[:, bits * pos + k] = (idx >> k) & 1
    return np.packbits(stream, axis=1, bitorder="little")


def unpack_codes(packed: np.ndarray, bits: int, d: int) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    stream = np.unpackbits(packed, axis=1, bitorder="little")[:, : d * bits].astype(np.int64)
    pos = slot_order(d)
    return sum(stream[:, bits * pos + k] << k for k in range(bits))


def pack_signs(signs: np.ndarray) -> np.ndarray:
    signs = np.asarray(signs, dtype=np.uint8)
    stream = np.zeros_like(signs)
    stream[:, slot_order(signs.shape[1])] = signs
    return np.packbits(stream, axis=1, bitorder="little")


def unpack_signs(packed: np.ndarray, d: int) -> np.ndarray:
    stream = np.unpackbits(np.asarray(packed, dtype=np.uint8), axis=1, bitorder="little")[:, :d]
    return stream[:, slot_order(d)].astype(bool)


def encoded_from_storage(role: Role, norm, codes_packed, d, signs_packed=None, rnorm=None) -> Encoded:
    """Rebuild an Encoded record from packed storage (e.g. bytes a GPU produced)."""
    enc = Encoded(role=role, norm=np.asarray(norm, dtype=np.float32).reshape(-1),
                  idx=unpack_codes(np.asarray(codes_packed).reshape(len(np.asarray(norm).reshape(-1)), -1),
                                   role.bits, d))
    if role.qjl:
        enc.signs = unpack_signs(np.asarray(signs_packed).reshape(enc.idx.shape[0], -1), d)
        enc.rnorm = np.asarray(rnorm, dtype=np.float32).reshape(-1)
    return enc


def record_bytes(role: Role, d: int) -> int:
    """Algorithmic bytes of one stored vector: codes + float32 norm (+ signs + float32 rho)."""
    b = role.bits * d // 8 + 4
    if role.qjl:
        b += d // 8 + 4
    return b
