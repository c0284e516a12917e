"""Pins for the oracle's rotation, quantiser, QJL sketch, attention and KIVI path (CPU only)."""

import itertools
import math

import numpy as np
import pytest

from conftest import read_golden
from oracle import attention as att
from oracle import codebook as cb
from oracle import kivi
from oracle import metrics
from oracle import rng
from oracle import turboquant as tq


# ---------------------------------------------------------------- Walsh-Hadamard

@pytest.mark.parametrize("d", [2, 8, 64, 128])
def test_hadamard_matches_definition_and_is_orthonormal(d):
    H = tq.hadamard(d)
    brute = np.array([[(-1) ** bin(i & j).count("1") for j in range(d)] for i in range(d)]) / math.sqrt(d)
    np.testing.assert_array_equal(H, brute)
    np.testing.assert_allclose(H @ H, np.eye(d), atol=1e-14)


def test_rotation_preserves_norms_and_inverts():
    g = np.random.default_rng(2)
    p = tq.make_params(128, 4, "KQV", 42)
    x = g.standard_normal((64, 128))
    y = (x * p.D[None, :]) @ tq.hadamard(128).T
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)
    back = (y @ tq.hadamard(128).T) * p.D[None, :]
    np.testing.assert_allclose(back, x, atol=1e-13)


# ---------------------------------------------------------------- storage format

@pytest.mark.parametrize("row", [" ".join(r) for r in read_golden("pack_example.txt")])
def test_packing_matches_hand_worked_examples(row):
    left, right = row.split("|")
    vals = [int(x) for x in left.split()]
    bits, d, codes = vals[0], vals[1], np.array([vals[2:]])
    want = np.array([[int(x) for x in right.split()]], dtype=np.uint8)
    if bits == 1:
        got = tq.pack_signs(codes.astype(bool))
        np.testing.assert_array_equal(tq.unpack_signs(got, d), codes.astype(bool))
    else:
        got = tq.pack_codes(codes, bits)
        np.testing.assert_array_equal(tq.unpack_codes(got, bits, d), codes)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_pack_matches_brute_force_bit_setting(bits):
    """Slot order written out per coordinate: i = 8n + 2t + e -> code offset 32t + 2n + e."""
    g = np.random.default_rng(bits)
    d = 128
    idx = g.integers(0, 1 << bits, size=(5, d))
    got = tq.pack_codes(idx, bits)
    for n in range(5):
        stream = bytearray(bits * d // 8)
        for i in range(d):
            nn, t, e = i // 8, (i // 2) % 4, i % 2
            off = 32 * t + 2 * nn + e
            for k in range(bits):
                if (idx[n, i] >> k) & 1:
                    pos = bits * off + k
                    stream[pos // 8] |= 1 << (pos % 8)
        assert bytes(got[n]) == bytes(stream)
    # a tensor-core thread's 16 pairs (fixed t) are contiguous: 32*bits bits from 32*bits*t
    t = 2
    want = [(i, c) for i in range(d) if (i // 2) % 4 == t for c in [idx[0, i]]]
    seg = tq.unpack_codes(got[:1], bits, d)[0]
    assert [seg[i] for i, _ in want] == [c for _, c in want]


# ---------------------------------------------------------------- quantiser

def test_bucketize_equals_nearest_centroid():
    """Counting boundaries at or below y picks the nearest centroid (midpoint boundaries)."""
    p = tq.make_params(128, 4, "KQV", 3)
    g = np.random.default_rng(4)
    x = g.standard_normal((256, 128))
    enc = tq.encode(x, tq.Role(4, True, False), p)
    c = cb.lloyd_max(128, 4).centroids32.astype(np.float64)
    nearest = np.argmin(np.abs(enc.y[:, :, None] - c[None, None, :]), axis=2)
    np.testing.assert_array_equal(enc.idx, nearest)


@pytest.mark.parametrize("scheme", tq.SCHEMES)
@pytest.mark.parametrize("n", [2, 3, 4])
def test_scheme_roles_spend_the_equal_budget(scheme, n):
    rk, rv = tq.scheme_roles(scheme, n)
    # n bits per coordinate for each of K and V, sketch bit included
    assert rk.bits + rk.qjl == n and rv.bits + rv.qjl == n
    if scheme == "KV":
        assert not (rk.rotate or rv.rotate or rk.qjl or rv.qjl)
    if scheme == "KQV":
        assert rk.rotate and rv.rotate and not rk.qjl and rv.qjl
    if scheme == "QKQV":
        assert rk.qjl and rv.qjl


def test_zero_vector_and_scale_equivariance():
    p = tq.make_params(128, 4, "KQV", 9)
    role = tq.Role(3, True, True)
    g = np.random.default_rng(0)
    x = np.vstack([np.zeros(128), g.standard_normal(128)])
    e = tq.encode(x, role, p)
    assert e.norm[0] == 0 and e.rnorm[0] == 0 and e.signs[0].all()
    assert np.all(e.idx[0] == cb.lloyd_max(128, 3).levels // 2)
    np.testing.assert_array_equal(tq.decode(e, p)[0], 0.0)
    # codes and signs depend only on the direction (powers of two keep it exact)
    e2 = tq.encode(x * 8.0, role, p)
    np.testing.assert_array_equal(e2.idx, e.idx)
    np.testing.assert_array_equal(e2.signs, e.signs)


def test_rotated_mse_matches_codebook_distortion():
    """Rotating arbitrary vectors then bucketizing gives the sphere-marginal MSE."""
    p = tq.make_params(128, 4, "KQV", 21)
    g = np.random.default_rng(8)
    x = g.standard_normal((4000, 128)) * np.exp(g.standard_normal(128))[None, :]
    for bits in (2, 3, 4):
        e = tq.encode(x, tq.Role(bits, True, False), p)
        u = x / np.linalg.norm(x, axis=1, keepdims=True)
        xh = tq.decode(e, p) / e.norm.astype(np.float64)[:, None]
        err = np.sum((u - xh) ** 2, axis=1)
        want = cb.lloyd_max(128, bits).mse_per_vector()
        assert abs(err.mean() - want) < 0.1 * want


def test_qjl_inner_product_is_unbiased_with_the_pages_variance():
    """Over many S draws: E[sqrt(pi/2)/m ||r|| <S y, sign(S r)>] = <y, r>, and its variance is
    ((pi/2)||y||^2||r||^2 - <y,r>^2)/m, at least pi/2 times a scalar residual's share."""
    d = m = 32
    g = np.random.default_rng(12)
    y = g.standard_normal(d)
    r = 0.3 * g.standard_normal(d) + 0.2 * y
    ests = []
    for seed in range(3000):
        S = rng.gaussian_sketch(seed, d).astype(np.float64)
        sig = np.where(S @ r >= 0, 1.0, -1.0)
        ests.append(tq.SQRT_HALF_PI / m * np.linalg.norm(r) * (S @ y) @ sig)
    ests = np.array(ests)
    yr = y @ r
    se = ests.std() / math.sqrt(len(ests))
    assert abs(ests.mean() - yr) < 4 * se
    var_want = ((math.pi / 2) * (y @ y) * (r @ r) - yr ** 2) / m
    assert abs(ests.var() - var_want) < 0.1 * var_want
    claims = {row[0]: float(row[1]) for row in read_golden("page_claims.txt")}
    # the page's (pi/2)||r||^2/d per unit-norm query direction is the leading term
    assert (math.pi / 2) * (y @ y) * (r @ r) / m >= claims["qjl_inflation_min"] * ((y @ y) * (r @ r) - yr ** 2) / m


def test_sketched_reconstruction_is_unbiased_per_vector():
    """Averaged over S draws, the QJL-augmented reconstruction tends to the vector itself."""
    d = 16
    g = np.random.default_rng(1)
    x = g.standard_normal((1, d))
    acc = np.zeros(d)
    n = 2500
    for seed in range(n):
        p = tq.Params(d=d, n=3, scheme="KQV", seed=seed, D=rng.rademacher_diagonal(seed, d),
                      S=rng.gaussian_sketch(seed, d))
        acc += tq.decode(tq.encode(x, tq.Role(2, True, True), p), p)[0]
    assert np.linalg.norm(acc / n - x[0]) < 0.08 * np.linalg.norm(x[0])


# ---------------------------------------------------------------- attention

def test_softmax_invariant_to_a_shared_key_shift():
    """[HeadQ] 2.1: adding one vector to every key shifts all scores equally."""
    g = np.random.default_rng(3)
    q, K, V = g.standard_normal(128), g.standard_normal((300, 128)), g.standard_normal((300, 128))
    mu = 5.0 * g.standard_normal(128)
    o1, p1 = att.attend(q, K, V)
    o2, p2 = att.attend(q, K + mu[None, :], V)
    np.testing.assert_allclose(p1, p2, atol=1e-12)
    np.testing.assert_allclose(o1, o2, atol=1e-12)


@pytest.mark.parametrize("N", [1, 2, 5, 8])
def test_attention_against_brute_force_loops(N):
    g = np.random.default_rng(N)
    d = 8
    q, K, V = g.standard_normal(d), g.standard_normal((N, d)), g.standard_normal((N, d))
    s = [sum(q[i] * K[j][i] for i in range(d)) / math.sqrt(d) for j in range(N)]
    e = [math.exp(x) for x in s]
    Z = sum(e)
    o = [sum(e[j] / Z * V[j][i] for j in range(N)) for i in range(d)]
    got, _ = att.attend(q, K, V)
    np.testing.assert_allclose(got, o, atol=1e-13)
    if N == 1:
        np.testing.assert_array_equal(got, V[0])


def test_qkqv_score_forms_agree():
    p = tq.make_params(128, 4, "QKQV", 77)
    rk, _ = p.roles()
    g = np.random.default_rng(5)
    K, q = g.standard_normal((200, 128)), g.standard_normal(128)
    e = tq.encode(K, rk, p)
    direct = tq.decode(e, p) @ q / math.sqrt(128)
    np.testing.assert_allclose(att.qkqv_scores(q, e, p), direct, atol=1e-12, rtol=1e-12)


def test_gqa_maps_query_heads_to_their_kv_head():
    g = np.random.default_rng(6)
    Q = g.standard_normal((2, 8, 16))
    K, V = g.standard_normal((2, 2, 10, 16)), g.standard_normal((2, 2, 10, 16))
    out = att.attend_gqa(Q, K, V, lengths=[10, 7])
    for b, h in itertools.product(range(2), range(8)):
        n = 10 if b == 0 else 7
        o, _ = att.attend(Q[b, h], K[b, h // 4, :n], V[b, h // 4, :n])
        np.testing.assert_allclose(out[b, h], o, atol=1e-14)


@pytest.mark.slow
def test_kqv_beats_qkqv_in_kl_at_four_bits():
    """[TQ-stats] "Main contribution 2": at n = 4, KQV has lower KL than QKQV (2.25x on the page)."""
    g = np.random.default_rng(31)
    d, N, H = 128, 2048, 6
    kls = {}
    for scheme in ("KQV", "QKQV"):
        p = tq.make_params(d, 4, scheme, 42)
        rk, rv = p.roles()
        vals = []
        for h in range(H):
            gh = np.random.default_rng(100 + h)
            K, V, q = gh.standard_normal((N, d)), gh.standard_normal((N, d)), gh.standard_normal(d)
            _, pf = att.attend(q, K, V)
            kh = tq.decode(tq.encode(K, rk, p), p)
            _, pq = att.attend(q, kh, V)
            vals.append(metrics.kl(pf, pq))
        kls[scheme] = np.mean(vals)
    assert kls["QKQV"] > 1.3 * kls["KQV"], kls


# ---------------------------------------------------------------- KIVI

def test_kivi_quantised_length_follows_the_window_rule():
    W, G = 128, 32
    w, nq = 0, 0
    for N in range(1, 700):
        w += 1
        if w == W + G:
            nq += G
            w -= G
        assert kivi.quantized_length(N, W, G) == nq
    assert kivi.quantized_length(4096) == 3968


def test_kivi_group_error_within_half_a_step():
    """[KIVI-geometry]: zero = group min, step = range/(2^B - 1), error <= step/2."""
    g = np.random.default_rng(9)
    x = kivi.to_bf16(g.standard_normal((500, 32)).astype(np.float32) * np.exp(g.standard_normal((500, 1))))
    z, s, codes, t = kivi.quantize_groups(x)
    xh = kivi.dequantize_groups(z, s, codes)
    zerr = np.abs(z.astype(np.float64) - x.min(axis=1))
    bound = s.astype(np.float64) / 2 * (1 + 1e-3) + zerr + 1e-12
    assert np.all(np.abs(xh - x) <= bound[:, None])
    assert np.all(codes[np.arange(500), np.argmax(x, axis=1)] == 3)
    assert np.all(codes[np.arange(500), np.argmin(x, axis=1)] == 0)
    # a constant group stores step 0 and codes 0, reconstructing exactly
    z0, s0, c0, _ = kivi.quantize_groups(np.full((1, 32), 1.5))
    assert s0[0] == 0 and np.all(c0 == 0) and np.all(kivi.dequantize_groups(z0, s0, c0) == 1.5)


@pytest.mark.parametrize("per_channel", [True, False])
def test_kivi_tensor_groups_along_the_right_axis(per_channel):
    g = np.random.default_rng(10)
    x = kivi.to_bf16(g.standard_normal((300, 128)).astype(np.float32))
    T = kivi.quantize_tensor(x, per_channel)
    assert T.nq == 160 and T.window.shape == (140, 128)
    xh = T.dequantize()
    np.testing.assert_array_equal(xh[160:], x[160:])
    if per_channel:
        assert T.z16.shape == (5, 128)
        blk = x[32:64, 7].astype(np.float64)
    else:
        assert T.z16.shape == (160, 4)
        blk = x[7, 32:64].astype(np.float64)
    zz = T.z16[1, 7] if per_channel else T.z16[7, 1]
    assert zz == np.float16(blk.min())


def test_kivi_two_bit_packing_roundtrip():
    g = np.random.default_rng(3)
    c = g.integers(0, 4, size=(7, 128)).astype(np.uint8)
    np.testing.assert_array_equal(kivi.unpack2(kivi.pack2(c), 128), c)
    # plain channel order: channel i at bits [2i, 2i+2)
    for n in range(7):
        want = bytearray(32)
        for i in range(128):
            want[(2 * i) // 8] |= int(c[n, i]) << ((2 * i) % 8)
        assert bytes(kivi.pack2(c)[n]) == bytes(want)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], dtype=np.float32)
    want = np.array([1.0, 1.0, 1.0 + 4 * 2 ** -8, -2.5, 1.0], dtype=np.float32)
    np.testing.assert_array_equal(kivi.to_bf16(x), want)


# ---------------------------------------------------------------- metrics

def test_metrics_closed_forms():
    p = np.array([0.5, 0.25, 0.125, 0.125])
    assert metrics.kl(p, p) == 0.0
    u = np.full(4, 0.25)
    assert abs(metrics.kl(p, u) - (2.0 - 1.75) * math.log(2)) < 1e-15
    assert metrics.topk_recall(np.arange(10.0), np.arange(10.0)) == 1.0
    assert metrics.topk_recall(np.arange(10.0), -np.arange(10.0)) == 0.0
    x = np.array([[3.0, 4.0]])
    m = metrics.six_d(x, 2.0 * x)
    assert abs(m["scale_err"][0] - 1.0) < 1e-15 and abs(m["dir_err"][0]) < 1e-15
    m = metrics.six_d(x, np.array([[4.0, -3.0]]))
    assert abs(m["phi"][0] - math.pi / 2) < 1e-15 and abs(m["snr_db"][0] - 10 * math.log10(0.5)) < 1e-12
