"""CPU check of the arithmetic rule the KIVI append kernels use for a code, against the oracle.

The oracle codes a value x of a group with stored statistics (z, s) (both float16) as
clamp(round_half_even((x - z) / s), 0, 3) with the quotient in fp64 (`oracle.kivi`). The kernels
take dx = fp32(x - z) and count the thresholds c_k = (k + 1/2) s, k = 0, 1, 2, that dx passes --
c_0 and c_2 strictly, c_1 from the threshold on -- reading the three tests off the sign bits of
A = c_0 - dx, B = dx - c_1, C = c_2 - dx: high bit = not sign(B), low bit = not sign(A ^ B ^ C).
A zero or infinite step makes every code 0, as the oracle's zero quotient does.

This restates that rule in numpy (float32 arithmetic, as on the device) and checks it against the
oracle's codes on bfloat16 and float32 groups, whose few significant bits make exact ties
(quotients of exactly 1/2, 3/2, 5/2) frequent; it also checks that the thresholds are exact in
float32. The kernels themselves are compared with the oracle by the GPU tests."""

import numpy as np
import pytest

from oracle import kivi as okivi


def rule_codes(x, z16, s16):
    """The kernels' code rule; x [groups, 32] float32, z16 / s16 [groups] float16."""
    x = np.asarray(x, dtype=np.float32)
    s = s16.astype(np.float32)
    ok = (s > 0) & np.isfinite(s)
    nz = np.where(ok, -z16.astype(np.float32), np.float32(0))[:, None]
    inf = np.float32(np.inf)
    c0 = np.where(ok, np.float32(0.5) * s, inf)[:, None]
    c1 = np.where(ok, np.float32(1.5) * s, inf)[:, None]
    c2 = np.where(ok, np.float32(2.5) * s, inf)[:, None]
    with np.errstate(over="ignore", invalid="ignore"):
        dx = (x + nz).astype(np.float32)
        a = (c0 - dx).astype(np.float32).view(np.uint32)
        b = (dx - c1).astype(np.float32).view(np.uint32)
        c = (c2 - dx).astype(np.float32).view(np.uint32)
    hi = 1 - (b >> 31)
    lo = 1 - ((a ^ b ^ c) >> 31)
    return (2 * hi + lo).astype(np.uint8), dx


def groups(rng, n, kind):
    """n groups of 32: bfloat16 values, or float32 ones; some groups with a zero range."""
    scale = np.exp(rng.normal(0, 2, size=(n, 1))).astype(np.float32)
    x = (rng.standard_normal((n, 32)).astype(np.float32) * scale + rng.normal(0, 3, size=(n, 1))).astype(np.float32)
    x[::17] = x[::17, :1]  # constant groups: step 0
    if kind == "bf16":
        x = okivi.to_bf16(x)
    return x


@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_threshold_rule_matches_the_oracle(kind):
    rng = np.random.default_rng(11 if kind == "bf16" else 12)
    x = groups(rng, 40_000, kind)
    z16, s16, codes, t = okivi.quantize_groups(x)
    got, dx = rule_codes(x, z16, s16)
    # groups with a zero step (code 0 either way), and elsewhere the values whose x - z is exact
    # in float32: there the rule is the oracle's rounding, ties included
    step_ok = ((s16 > 0) & np.isfinite(s16))[:, None]
    exact = ~step_ok | (dx.astype(np.float64) == x.astype(np.float64) - z16.astype(np.float64)[:, None])
    assert step_ok.mean() > 0.5
    np.testing.assert_array_equal(got[exact], codes[exact])
    if kind == "bf16":
        # bf16 values and their fp16 zero point differ exactly, and ties are frequent
        assert exact.mean() > 0.999
        assert np.isin(t[exact], (0.5, 1.5, 2.5)).sum() > 1000
    # where x - z rounds in float32 (a value far from a zero point of larger magnitude, so
    # |x - z| ~ |z| <~ 3 s), the rounding moves the quotient by at most ~3 2^-24 and the rule
    # may only differ next to a rounding boundary
    off = ~exact & (got != codes)
    if off.any():
        assert np.all(np.abs(np.abs(t[off] - np.floor(t[off])) - 0.5) < 1e-6)


def test_thresholds_are_exact_in_float32():
    s16 = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16)  # every finite positive fp16
    s = s16.astype(np.float32)
    for k in (0.5, 1.5, 2.5):
        np.testing.assert_array_equal((np.float32(k) * s).astype(np.float64), k * s16.astype(np.float64))


def test_degenerate_steps_code_zero():
    x = np.array([[5.0] * 32, [-7.0] * 32, [1e30] * 32], dtype=np.float32)
    z16 = np.array([1.0, -np.inf, 2.0], dtype=np.float16)
    for s in (0.0, np.inf):
        got, _ = rule_codes(x, z16, np.full(3, s, dtype=np.float16))
        assert not got.any()
