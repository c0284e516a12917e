"""CPU check of the launch-constant 32-bit division that the append kernels use for their index
arithmetic (warp index -> sequence-head and position, sequence-head -> batch).

The host constructor `make_fastdiv` is compiled from the library's internal header as it stands;
its constants are then run through the device formula (multiply-high, subtract, shift, add,
shift: Granlund and Montgomery, "Division by Invariant Integers using Multiplication", 1994,
section 4) and compared with true integer division over edge and random numerators. No GPU is
used."""

import os
import shutil
import subprocess

import numpy as np
import pytest

from conftest import ROOT

DIVISORS = [1, 2, 3, 5, 7, 8, 31, 32, 33, 40, 63, 64, 65, 127, 128, 129, 160, 255, 256, 257, 1000,
            1025, 4097, 8193, 65535, 65536, 65537, 999_983, 1 << 20, (1 << 20) + 1, (1 << 31) - 1,
            1 << 31, (1 << 31) + 1, 0xFFFFFFFE, 0xFFFFFFFF]


@pytest.fixture(scope="module")
def constants(tmp_path_factory):
    cxx = shutil.which("g++")
    cuda_inc = "/usr/local/cuda/include"
    if cxx is None or not os.path.isdir(cuda_inc):
        pytest.skip("needs g++ and the CUDA headers")
    d = tmp_path_factory.mktemp("fastdiv")
    src = d / "fd.cpp"
    src.write_text(
        '#include <cstdio>\n#include "tq_internal.h"\n'
        "int main() {\n  unsigned v;\n  while (std::scanf(\"%u\", &v) == 1) {\n"
        "    const tq::FastDiv f = tq::make_fastdiv(v);\n"
        "    std::printf(\"%u %u %u %u\\n\", f.d, f.m, f.s1, f.s2);\n  }\n  return 0;\n}\n")
    exe = d / "fd"
    csrc = os.path.join(ROOT, "quantised_kv_cache_gb300", "csrc")
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", csrc, "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                    str(src), "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], input=" ".join(str(v) for v in DIVISORS), capture_output=True, text=True,
                         check=True).stdout
    return {int(r.split()[0]): tuple(int(x) for x in r.split()[1:]) for r in out.strip().splitlines()}


def device_quotient(n, m, s1, s2):
    """The kernels' fast_div on uint64 arrays holding 32-bit values."""
    t = (m * n) >> np.uint64(32)
    return (t + ((n - t) >> np.uint64(s1))) >> np.uint64(s2)


@pytest.mark.parametrize("d", DIVISORS)
def test_fast_division_equals_integer_division(constants, d):
    m, s1, s2 = constants[d]
    rng = np.random.default_rng(d)
    edge = [0, 1, 2, d - 1, d, d + 1, 2 * d - 1, 2 * d, 0x7FFFFFFF, 0x80000000, 0xFFFFFFFE, 0xFFFFFFFF]
    near = [k * d + e for k in (1, 2, 3, 1000, 0xFFFFFFFF // d) for e in (-1, 0, 1)]
    n = np.array([v for v in edge + near if 0 <= v <= 0xFFFFFFFF], dtype=np.uint64)
    n = np.concatenate([n, rng.integers(0, 1 << 32, size=200_000, dtype=np.uint64)])
    got = device_quotient(n, np.uint64(m), s1, s2)
    np.testing.assert_array_equal(got, n // np.uint64(d))
