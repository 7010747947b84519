"""The bounded wait behind every asynchronous-copy wait in the codec's kernels gives up after
its time limit and reports it (no fault, no trap, no hang), and returns at once when the
phase has completed."""
import ctypes
import os
import subprocess

import pytest

from compressed_pseudo_gradient_gb300 import build as lib_build

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib():
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libwaitcheck.so")
    subprocess.run([lib_build.nvcc(), *lib_build.NVCC_FLAGS, "-shared", "-o", so,
                    os.path.join(HERE, "cuda", "wait_check.cu")], check=True)
    lib = ctypes.CDLL(so)
    lib.wait_check.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_uint32),
                               ctypes.POINTER(ctypes.c_ulonglong)]
    return lib


def run(lib, complete):
    ok = ctypes.c_uint32(7)
    ns = ctypes.c_ulonglong(0)
    assert lib.wait_check(complete, ctypes.byref(ok), ctypes.byref(ns)) == 0
    return ok.value, ns.value


def test_wait_on_a_phase_that_never_completes_times_out(lib):
    ok, ns = run(lib, 0)
    assert ok == 0
    assert 0.9e9 <= ns <= 5e9          # about the one-second limit


def test_wait_on_a_completed_phase_returns_at_once(lib):
    ok, ns = run(lib, 1)
    assert ok == 1 and ns < 1e7
