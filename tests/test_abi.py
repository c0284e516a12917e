"""CPU checks of the C ABI: the library loads, exports every declared symbol,
and its host-side method constants (codebook, D, S) agree with the oracle.
No GPU call is made here."""

import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT
from oracle import codebook as cb
from oracle import rng


@pytest.fixture(scope="module")
def tqmod():
    from quantised_kv_cache_gb300 import build, tq
    build.build()  # no-op when up to date
    return tq


def declared_functions():
    text = open(os.path.join(ROOT, "include", "tq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("tq_init", "tq_append_quantize", "tq_decode_attention", "tq_dequantize", "tq_destroy"):
        assert must in names


def test_library_exports_every_declared_symbol(tqmod):
    L = tqmod.lib()
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    # and the binding wraps each of them under the same name
    assert all(hasattr(tqmod, n) for n in declared_functions())


def test_abi_version_and_status_strings(tqmod):
    assert tqmod.tq_abi_version() == 3
    assert tqmod.tq_status_str(0) == "ok"
    assert "capacity" in tqmod.tq_status_str(3)
    assert tqmod.tq_status_str(12345) == "unknown status"


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_library_codebook_matches_oracle(tqmod, d, bits):
    """Two independent fits (Gauss-Legendre quadrature in C++, incomplete beta in
    the oracle) of the same Lloyd-Max fixed point."""
    c, b = tqmod.tq_codebook_f64(d, bits)
    C = cb.lloyd_max(d, bits)
    assert np.max(np.abs(c - C.centroids)) < 1e-12
    assert np.max(np.abs(b - C.bounds)) < 1e-12
    np.testing.assert_array_equal(c.astype(np.float32), C.centroids32)
    np.testing.assert_array_equal(b.astype(np.float32), C.bounds32)


@pytest.mark.parametrize("seed", [0, 42, 2 ** 63 + 12345])
def test_library_method_randomness_is_bit_exact(tqmod, seed):
    D, S = tqmod.tq_draw_params(seed, 128)
    np.testing.assert_array_equal(D, rng.rademacher_diagonal(seed, 128))
    np.testing.assert_array_equal(S.view(np.uint32), rng.gaussian_sketch(seed, 128).view(np.uint32))


def test_host_argument_errors(tqmod):
    L = tqmod.lib()
    h = ctypes.c_void_p()
    # bad scheme / bits / dimension are rejected before any device work
    assert L.tq_init(128, 4, 9, ctypes.c_uint64(1), ctypes.byref(h)) == tqmod.TQ_ERR_ARG
    assert L.tq_init(128, 5, 1, ctypes.c_uint64(1), ctypes.byref(h)) == tqmod.TQ_ERR_ARG
    assert L.tq_init(100, 4, 1, ctypes.c_uint64(1), ctypes.byref(h)) == tqmod.TQ_ERR_ARG
    assert L.tq_init(64, 4, 1, ctypes.c_uint64(1), ctypes.byref(h)) == tqmod.TQ_ERR_UNSUPPORTED
    assert L.tq_init(128, 3, 3, ctypes.c_uint64(1), ctypes.byref(h)) == tqmod.TQ_ERR_UNSUPPORTED
    assert L.tq_codebook_f64(100, 2, None, None) == tqmod.TQ_ERR_ARG
    assert L.tq_draw_params(ctypes.c_uint64(1), 3, None, None) == tqmod.TQ_ERR_ARG
    assert L.tq_cache_sizes_get(None, 1, 1, 1, None) == tqmod.TQ_ERR_ARG
    assert L.tq_append_quantize(None, None, None, None, 0, 1, 1, 1, None, None) == tqmod.TQ_ERR_ARG
    assert L.tq_decode_attention(None, None, None, 0, 1, 1, 1, None, 1, 0, None, 0, None, None) == tqmod.TQ_ERR_ARG
    assert L.tq_decode_step(None, None, None, 0, None, None, 0, 1, 1, 1, None, 1, None, 0, None,
                            None) == tqmod.TQ_ERR_ARG
    L.tq_destroy(None)  # no-op


@pytest.mark.parametrize("seed", [0, 42, 300])
def test_library_dense_rotation_matches_oracle(tqmod, seed):
    """The library's Gram-Schmidt of the stream-3 Gaussian and the oracle's LAPACK QR,
    both sign-fixed to SO(d), round to the same float32 matrix (a last-place difference is
    allowed where the two fp64 values straddle a rounding point)."""
    from oracle import rotation as orot
    M = tqmod.tq_draw_rotation(seed, 128)
    want = orot.dense_rotation(seed, 128)
    assert np.max(np.abs(M.astype(np.float64) - want)) < 1e-7
    assert np.mean(M == want.astype(np.float32)) > 0.999
    assert abs(np.linalg.det(M.astype(np.float64)) - 1.0) < 1e-5


def test_library_principal_basis_matches_oracle(tqmod):
    """Jacobi rotations in C++ against LAPACK's symmetric eigensolver in the oracle, with the
    same sign convention."""
    from oracle import sidecode as sc
    g = np.random.default_rng(0)
    X = (g.standard_normal((300, 128)) @ np.diag(np.linspace(3, 0.1, 128))).astype(np.float32)
    for r in (1, 4, 8):
        U = tqmod.tq_principal_basis(X, r)
        np.testing.assert_allclose(U, sc.principal_basis(X.astype(np.float64), r), atol=1e-6)
