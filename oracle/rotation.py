"""Dense random rotation in SO(d): the alternative to the randomised Walsh-Hadamard
transform (fp64 oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

[KVQuant++] "Rotation-invariance guarantee" (旋转不变性保证): a random rotation taken
from a QR factorisation may come out as a reflection (determinant -1); the method
requires a matrix of the special orthogonal group SO(d), determinant +1. [KVQuant++]
"Rate-distortion performance" (率失真性能) and "Core innovation 5": the rotation may be
a QR rotation or a Hadamard transform; after either, the coordinates of a unit vector
follow the sphere marginal the codebook is fitted to.

Steps, in that order:

1. G: a d x d Gaussian matrix from the method's counter generator, stream 3 (row-major
   entry k = row * d + col, the Box-Muller recipe of ``rng.gaussian_sketch`` kept in
   fp64 rather than rounded to float32);
2. G = Q R with R's diagonal made positive (Q's columns times the signs of diag(R)), the
   unique factorisation with that convention -- column j of Q is the unit vector of
   column j of G orthogonal to the columns before it (Gram-Schmidt);
3. if det Q = -1, the last column of Q changes sign (a reflection becomes a rotation);
4. the rotation applied to a unit vector u is y = Q^T u (its coordinates in the basis
   Q's columns form); reconstruction applies Q.

Readings where the pages are silent: the generator stream and the positive-diagonal
convention (which makes the factorisation, hence the rotation, a function of the seed);
y = Q^T u rather than Q u (either is a Haar rotation; this one reads as "coordinates in
the random basis"); one rotation per context, shared by keys, values and queries, as D
is for the Walsh-Hadamard transform.
"""

import math

import numpy as np

from . import rng as _rng

STREAM_ROTATION = 3


def gaussian_matrix(seed: int, d: int) -> np.ndarray:
    """G in R^{d x d}, row-major entry k = row * d + col, from stream 3:
    u1 = ((w_{2k} >> 11) + 1) 2^-53, u2 = (w_{2k+1} >> 11) 2^-53,
    G_k = sqrt(-2 ln u1) cos(2 pi u2) in fp64."""
    out = np.empty(d * d, dtype=np.float64)
    scale = 2.0 ** -53
    for k in range(d * d):
        w1 = _rng.draw(seed, STREAM_ROTATION, 2 * k)
        w2 = _rng.draw(seed, STREAM_ROTATION, 2 * k + 1)
        u1 = ((w1 >> 11) + 1) * scale
        u2 = (w2 >> 11) * scale
        out[k] = math.sqrt(-2.0 * math.log(u1)) * math.cos(2.0 * math.pi * u2)
    return out.reshape(d, d)


def dense_rotation(seed: int, d: int) -> np.ndarray:
    """The d x d matrix M with y = M u: M = Q^T for the sign-fixed Q of G = Q R, with
    det M = +1."""
    G = gaussian_matrix(seed, d)
    Q, R = np.linalg.qr(G)
    Q = Q * np.sign(np.diag(R))[None, :]
    if np.linalg.det(Q) < 0:
        Q[:, -1] = -Q[:, -1]
    return Q.T.copy()
