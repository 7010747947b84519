"""The decode kernel's division by P (reciprocal + Markstein correction; for P a power of two,
one multiply by the exact reciprocal) against CUDA's correctly rounded division, bit for bit,
for every divisor 1..256.

Coverage: every significand in one binade (scaling by powers of two leaves the rounding of a
normal quotient unchanged), every dividend below 2^-111 (quotients near and below the bottom
of the normal range, where the helper changes method), and zeros, infinities and NaN.
"""
import ctypes
import os
import subprocess

import pytest

from compressed_pseudo_gradient_gb300 import build as lib_build

HERE = os.path.dirname(os.path.abspath(__file__))


def test_power_of_two_division_is_one_rounded_multiply():
    """CPU, numpy fp32 (IEEE, round to nearest): x / 2^k == x * 2^-k for normal, subnormal and
    special x, the fact the decode relies on for power-of-two P."""
    import numpy as np
    rng = np.random.default_rng(0)
    bits = np.concatenate([rng.integers(0, 2**32, 200000, dtype=np.uint64),
                           np.arange(0, 1 << 16, dtype=np.uint64),            # subnormals
                           np.array([0x7F800000, 0xFF800000, 0x7F7FFFFF, 0x00800000,
                                     0x80000000, 0x00000001], dtype=np.uint64)])
    x = bits.astype(np.uint32).view(np.float32)
    with np.errstate(all="ignore"):
        for k in range(9):
            P = np.float32(2 ** k)
            q = x / P
            m = x * np.float32(1.0 / (2 ** k))
            same = (q.view(np.uint32) == m.view(np.uint32)) | (np.isnan(q) & np.isnan(m))
            assert same.all(), k


@pytest.fixture(scope="module")
def checker():
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libdivcheck.so")
    src = os.path.join(HERE, "cuda", "div_check.cu")
    subprocess.run([lib_build.nvcc(), *lib_build.NVCC_FLAGS, "-shared", "-o", so, src],
                   check=True)
    lib = ctypes.CDLL(so)
    lib.div_check.argtypes = [ctypes.c_int, ctypes.c_uint32, ctypes.c_uint32,
                              ctypes.POINTER(ctypes.c_ulonglong), ctypes.POINTER(ctypes.c_uint32)]
    return lib


def run(lib, lo, count, pmax=256):
    bad = ctypes.c_ulonglong(0)
    first = ctypes.c_uint32(0)
    assert lib.div_check(pmax, lo, count, ctypes.byref(bad), ctypes.byref(first)) == 0
    return bad.value, first.value


@pytest.mark.parametrize("sign", [0, 0x80000000])
@pytest.mark.gpu
def test_every_significand_one_binade(checker, sign):
    bad, first = run(checker, sign | 0x3f800000, 1 << 23)
    assert bad == 0, f"{bad} mismatches, first dividend bits {first:#x}"


@pytest.mark.gpu
def test_every_dividend_with_tiny_quotient(checker):
    # x < 2^-111: quotients below, at and just above the bottom of the normal range for
    # every P <= 256 (the helper switches method at 2^-125)
    bad, first = run(checker, 0, 0x08000000)
    assert bad == 0, f"{bad} mismatches, first dividend bits {first:#x}"


@pytest.mark.gpu
def test_special_values(checker):
    for lo, count in [(0x7f7fff00, 0x200), (0xff7fff00, 0x200), (0x7fc00000, 4), (0, 1),
                      (0x80000000, 1)]:
        bad, first = run(checker, lo, count)
        assert bad == 0, f"{bad} mismatches near {lo:#x}, first {first:#x}"
