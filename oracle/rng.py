"""Seeded method randomness: the +/-1 diagonal D and the Gaussian sketch S.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The pages draw a "seeded +/-1 diagonal" for the randomised Walsh-Hadamard
rotation and a Gaussian d x d matrix S for the QJL sketch ([TQ-stats],
technical summary, "Quantisation schemes" and "Main contribution 1"), but fix
no generator. Both sides therefore implement one counter-based generator from
its published definition: SplitMix64 (Steele, Lea, Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), evaluated at counter
``stream * 2**32 + i + 1`` so that any element can be drawn independently.
The Gaussian is the cosine branch of the Box-Muller transform (Box & Muller
1958), evaluated in double precision with the platform libm and rounded to
float32.

Pinned by: the published SplitMix64 output stream for seed 1234567, and the
statistics of the draws (tests/test_oracle_rng.py).
"""

import math

import numpy as np

_MASK = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15  # SplitMix64 golden-ratio increment

STREAM_DIAG = 1
STREAM_SKETCH = 2


def mix64(z: int) -> int:
    """SplitMix64 output function (variant 13 finaliser) on a 64-bit word."""
    z &= _MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
    return z ^ (z >> 31)


def draw(seed: int, stream: int, i: int) -> int:
    """The i-th 64-bit word of ``stream`` for ``seed``.

    Equals the (stream*2**32 + i + 1)-th output of a SplitMix64 generator
    whose state starts at ``seed``.
    """
    counter = (stream << 32) + i + 1
    return mix64((seed + counter * GAMMA) & _MASK)


def rademacher_diagonal(seed: int, d: int) -> np.ndarray:
    """D_i = -1 if the top bit of draw(seed, 1, i) is set, else +1 (int8)."""
    return np.array([-1 if (draw(seed, STREAM_DIAG, i) >> 63) else 1
                     for i in range(d)], dtype=np.int8)


def gaussian_sketch(seed: int, d: int, m: int = None) -> np.ndarray:
    """S in R^{m x d} (m = d by default), row-major entry k = row*d + col.

    u1 = ((w_{2k} >> 11) + 1) * 2^-53 in (0, 1], u2 = (w_{2k+1} >> 11) * 2^-53,
    S_k = float32( sqrt(-2 ln u1) * cos(2 pi u2) ).
    """
    if m is None:
        m = d
    out = np.empty(m * d, dtype=np.float32)
    scale = 2.0 ** -53
    for k in range(m * d):
        w1 = draw(seed, STREAM_SKETCH, 2 * k)
        w2 = draw(seed, STREAM_SKETCH, 2 * k + 1)
        u1 = ((w1 >> 11) + 1) * scale
        u2 = (w2 >> 11) * scale
        out[k] = np.float32(math.sqrt(-2.0 * math.log(u1)) * math.cos(2.0 * math.pi * u2))
    return out.reshape(m, d)
