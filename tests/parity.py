"""Helpers shared by the GPU parity tests: read a cache's planes back to the host
and hand them to the oracle, and apply the boundary-band rule.

The rule (taken from the parity bar this library is held to): packed codes and
sign bits must be bit-exact except where the oracle's fp64 value lies within
1e-6 of a decision boundary; such mismatches are counted and must stay under
1e-5 of all codes or bits. Codes live next to the rotated unit coordinate y,
signs next to (S r)_i, KIVI codes next to the half-integers of (x - zero)/step.
"""

import math

import numpy as np
import torch

from oracle import attention as oatt
from oracle import kivi as okivi
from oracle import turboquant as otq

BAND = 1e-6
MISMATCH_FRACTION = 1e-5

D = 128
U24 = 2.0 ** -24  # unit roundoff of float32 (round to nearest)
U23 = 2.0 ** -23  # one ulp: a bound for any faithful rounding (e.g. truncating accumulation)


def norm_rtol(through_rotation_mma: bool) -> float:
    """Largest relative difference allowed between the stored float32 norm and the
    oracle's fp64 ||x||, from a rounding-error bound of the library's arithmetic (not
    from observed errors).

    Direct paths compute s = sum_i x_i^2 with float32 FMAs in some order, then
    sqrt(s). For an inner product evaluated in any order, |fl(x.x) - x.x| <= gamma_d
    x.x with gamma_d = d u / (1 - d u) (Higham, "Accuracy and Stability of Numerical
    Algorithms", 2nd ed., Lemma 3.1 and eq. (3.5)); the square root halves that relative
    error and adds one rounding, so |nu_hat / nu - 1| <= d u / 2 + u + O(u^2). The inputs
    reach the kernels exactly (bf16 and fp32 are exact in float32), so with
    u = 2^-24, d = 128: (d/2 + 2) u = 3.93e-6.

    The bf16 bulk path reads the norm off the rotation instead: the tensor cores form
    y' = H' D x (H' the +/-1 Hadamard matrix, so ||y'|| = sqrt(d) ||x||) with exact
    products and float32 accumulation, then nu = ||y'|| / sqrt(d). Each y'_n is a sum
    of d terms of magnitude |x_j|, so |y'_n_hat - y'_n| <= gamma_{d-1} ||x||_1 with the
    accumulation's rounding taken as merely faithful (u = 2^-23); hence
    ||y'_hat - y'|| <= sqrt(d) gamma_{d-1} ||x||_1 <= d gamma_{d-1} ||x||_2, a relative
    error of at most sqrt(d) gamma_{d-1} in ||y'||, plus the sum of squares, the square
    root and the 1/sqrt(d) factor as above: sqrt(d) (d - 1) 2^-23 + (d/2 + 3) 2^-24 =
    1.72e-4. Any plausible mistake (a dropped coordinate moves the norm by ~1/d of its
    square) is orders of magnitude above either bound."""
    direct = (D / 2 + 2) * U24
    if not through_rotation_mma:
        return direct
    g = (D - 1) * U23 / (1 - (D - 1) * U23)
    return math.sqrt(D) * g + (D / 2 + 3) * U24


def bulk_bf16_path(dtype, vectors_per_tensor: int, role) -> bool:
    """True when an append of this many bf16 vectors on this role takes the bulk
    tensor-map kernel, whose norm comes through the rotation (norm_rtol). Appends of at
    most 8192 vectors per tensor take the warp-per-vector launch; unrotated roles and
    fp32 inputs compute the norm directly."""
    return dtype == torch.bfloat16 and role.rotate and vectors_per_tensor > 8192


def plane(cache, name, dtype, shape):
    return cache.plane(name).cpu().numpy().view(dtype).reshape(shape)


def gpu_encoded(cache, role, which, B, H, ntok):
    """Oracle Encoded records for tokens [0, ntok) of every (b, h), from a GPU cache."""
    cap = cache.struct.capacity
    d = 128
    cb = role.bits * d // 8
    codes = plane(cache, f"{which}_codes", np.uint8, (B, H, cap, cb))[:, :, :ntok].reshape(-1, cb)
    norm = plane(cache, f"{which}_norm", np.float32, (B, H, cap))[:, :, :ntok].reshape(-1)
    signs = rnorm = None
    if role.qjl:
        signs = plane(cache, f"{which}_signs", np.uint8, (B, H, cap, d // 8))[:, :, :ntok].reshape(-1, d // 8)
        rnorm = plane(cache, f"{which}_rnorm", np.float32, (B, H, cap))[:, :, :ntok].reshape(-1)
    return otq.encoded_from_storage(role, norm, codes, d, signs, rnorm), codes, signs


class BandReport:
    """Mismatch bookkeeping for one workload. Out-of-band mismatches are never
    allowed; the 1e-5 fraction is a property of the workload's whole code
    population, so a report should accumulate every comparison of one workload
    before `ok()` is asked (a single legitimate in-band flip in a 65536-code
    subset is already 1.5e-5 of that subset)."""

    def __init__(self):
        self.total = 0
        self.mismatch = 0
        self.out_of_band = 0
        self.in_band = 0
        self.worst = 0.0
        self.max_mismatch_distance = 0.0

    def add(self, mism_mask, dist):
        self.total += mism_mask.size
        self.mismatch += int(mism_mask.sum())
        ob = mism_mask & (dist >= BAND)
        self.out_of_band += int(ob.sum())
        self.in_band += int((dist < BAND).sum())
        if mism_mask.any():
            self.max_mismatch_distance = max(self.max_mismatch_distance, float(dist[mism_mask].max()))
        if ob.any():
            self.worst = max(self.worst, float(dist[ob].max()))

    def ok(self):
        return self.out_of_band == 0 and self.mismatch < MISMATCH_FRACTION * max(self.total, 1)

    def ok_out_of_band(self):
        return self.out_of_band == 0

    def __repr__(self):
        return (f"total={self.total} mismatch={self.mismatch} out_of_band={self.out_of_band} "
                f"in_band_population={self.in_band} max_mismatch_distance={self.max_mismatch_distance:.3g} "
                f"worst_out_of_band_distance={self.worst:.3g}")


def compare_codes(gpu_idx, ora, bounds32, report: BandReport):
    """gpu_idx, ora.idx: [N, d]; distance of the oracle's y to the nearest float32 boundary."""
    y = ora.y
    dist = np.min(np.abs(y[:, :, None] - bounds32.astype(np.float64)[None, None, :]), axis=2)
    report.add(gpu_idx != ora.idx, dist)
    return gpu_idx != ora.idx


def compare_signs(gpu_signs, ora, report: BandReport, skip_rows=None):
    """Signs of vectors whose codes matched (a legitimately flipped code changes the residual)."""
    mism = gpu_signs != ora.signs
    dist = np.abs(ora.z)
    if skip_rows is not None and skip_rows.any():
        keep = ~skip_rows
        mism, dist = mism[keep], dist[keep]
    report.add(mism, dist)


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def oracle_decode_from_cache(cache, params, q, lens, B, Hkv, Hq):
    """fp64 attention of the oracle over the GPU's own codes (so code mismatches cannot leak in)."""
    rk, rv = params.roles()
    N = int(max(lens))
    ek, _, _ = gpu_encoded(cache, rk, "k", B, Hkv, N)
    ev, _, _ = gpu_encoded(cache, rv, "v", B, Hkv, N)
    Kh = otq.decode(ek, params).reshape(B, Hkv, N, 128)
    Vh = otq.decode(ev, params).reshape(B, Hkv, N, 128)
    return oatt.attend_gqa(np.asarray(q, dtype=np.float64), Kh, Vh, lengths=lens)


def kivi_oracle_state(x, per_channel, window=128, group=32):
    return okivi.quantize_tensor(x, per_channel, window, group)


def kivi_gpu_codes(cache, which, B, H, ntok):
    cap = cache.struct.capacity
    c = plane(cache, f"{which}_codes", np.uint8, (B, H, cap, 32))[:, :, :ntok]
    return okivi.unpack2(c.reshape(-1, 32), 128).reshape(B, H, ntok, 128)


def kivi_gpu_stats(cache, which, B, H, per_channel):
    cap = cache.struct.capacity
    if per_channel:
        s = plane(cache, f"{which}_stats", np.float16, (B, H, cap // 32, 128, 2))
    else:
        s = plane(cache, f"{which}_stats", np.float16, (B, H, cap, 4, 2))
    return s[..., 0], s[..., 1]


def kivi_gpu_window(cache, which, B, H, window=128, group=32):
    R = window + group
    w = cache.plane(f"{which}_window").cpu().view(torch.bfloat16).float().numpy()
    return w.reshape(B, H, R, 128)


def kivi_dequant_gpu_state(cache, which, B, H, N, per_channel, window=128, group=32):
    """fp64 reconstruction of tokens [0, N) from the GPU's codes, stats and window."""
    nq = okivi.quantized_length(N, window, group)
    codes = kivi_gpu_codes(cache, which, B, H, N).astype(np.float64)
    z, s = kivi_gpu_stats(cache, which, B, H, per_channel)
    ring = kivi_gpu_window(cache, which, B, H, window, group)
    out = np.zeros((B, H, N, 128))
    for j in range(N):
        if j < nq:
            if per_channel:
                zz, ss = z[:, :, j // group].astype(np.float64), s[:, :, j // group].astype(np.float64)
            else:
                zz = np.repeat(z[:, :, j].astype(np.float64), group, axis=-1)
                ss = np.repeat(s[:, :, j].astype(np.float64), group, axis=-1)
            out[:, :, j] = zz + ss * codes[:, :, j]
        else:
            out[:, :, j] = ring[:, :, j % (window + group)]
    return out
