"""The C ABI on the host (CPU only): the library builds, loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

import compressed_pseudo_gradient_gb300 as spl
from compressed_pseudo_gradient_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spl.h")

OK, INVALID, ALIGN = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    return spl.library()


def declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spl_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("spl_ef_compress", "spl_ef_compress_multi", "spl_decode_aggregate",
               "spl_decode_aggregate_stats", "spl_ef_compress_codec",
               "spl_decode_aggregate_codec", "spl_codec_record_bytes", "spl_codec_num_chunks",
               "spl_pack", "spl_unpack", "spl_num_chunks", "spl_flags_status",
               "spl_status_string", "spl_last_cuda_error"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    for fn in declared_functions():
        assert hasattr(lib, fn), f"{fn} declared in spl.h but not exported"
    assert os.path.exists(lib_build.LIB_PATH)


def test_library_exports_the_calibration_call(lib):
    """spl_calib.h declares the data-movement reference kernels' one call; both builds export
    it."""
    names = declared_functions(os.path.join(ROOT, "include", "spl_calib.h"))
    assert names == ["spl_calib_moves"]
    for path in (lib_build.LIB_PATH, lib_build.CHECKED_LIB_PATH):
        assert hasattr(ctypes.CDLL(path), "spl_calib_moves")


def test_checked_library_exports_the_same_calls_and_its_reader():
    """The checked build (same sources, -DSPL_CHECKED=1) exports every call of spl.h and the
    one call of spl_checked.h; the normal build does not export the reader."""
    chk = ctypes.CDLL(lib_build.CHECKED_LIB_PATH)
    for fn in declared_functions():
        assert hasattr(chk, fn), f"{fn} missing from the checked build"
    text = open(os.path.join(ROOT, "include", "spl_checked.h")).read()
    assert "spl_debug_read" in re.findall(r"\b(spl_[a-z_]+)\s*\(", re.sub(r"/\*.*?\*/", "", text, flags=re.S))
    assert hasattr(chk, "spl_debug_read")
    assert not hasattr(ctypes.CDLL(lib_build.LIB_PATH), "spl_debug_read")
    chk.spl_debug_read.argtypes, chk.spl_debug_read.restype = [ctypes.c_void_p, ctypes.c_int], ctypes.c_int
    assert chk.spl_debug_read(None, 0) == INVALID


def test_library_is_built_for_sm103a_only():
    assert any("arch=compute_103a,code=sm_103a" in f for f in lib_build.ARCH)


def test_num_chunks_and_status_strings(lib):
    for n, c in [(0, 0), (1, 1), (4095, 1), (4096, 1), (4097, 2), (1 << 30, 262144)]:
        assert lib.spl_num_chunks(n) == c
        assert spl.num_chunks(n) == c
    for s in range(7):
        assert lib.spl_status_string(s) and lib.spl_status_string(s) != b"unknown status"
    assert lib.spl_status_string(99) == b"unknown status"
    assert lib.spl_last_cuda_error() == 0


def test_flags_status(lib):
    """A flags word read back from the device maps to one status, most severe first."""
    NONFINITE, BAD, TIMEOUT, PENDING = 1, 2, 4, 8
    expect = {0: 0, NONFINITE: 4, BAD: 5, BAD | NONFINITE: 5, TIMEOUT: 6, TIMEOUT | BAD: 6,
              TIMEOUT | PENDING: 6, PENDING: 6, 0x10: 0}
    for flags, status in expect.items():
        assert lib.spl_flags_status(flags) == status
        assert spl.flags_status(flags) == status


# Fake device addresses: the checks below fail on the host before any CUDA call is made.
A = 0x10000000
B = 0x20000000
Cp = 0x30000000
D = 0x40000000


def test_compress_argument_errors(lib):
    f = lib.spl_ef_compress
    n = 8192
    assert f(None, 0, None, 0, 1.0, None, None, None, None) == OK            # empty: no-op
    assert f(None, 0, B, n, 1.0, Cp, D, None, None) == INVALID                # NULL delta
    assert f(A, 0, None, n, 1.0, Cp, D, None, None) == INVALID                # NULL ef
    assert f(A, 0, B, n, 1.0, None, D, None, None) == INVALID                 # NULL payload
    assert f(A, 7, B, n, 1.0, Cp, D, None, None) == INVALID                   # bad dtype
    assert f(A, 0, B, n, float("nan"), Cp, D, None, None) == INVALID          # beta NaN
    assert f(A, 0, B, n, float("inf"), Cp, D, None, None) == INVALID          # beta inf
    assert f(A + 4, 0, B, n, 1.0, Cp, D, None, None) == ALIGN                 # delta 4-B
    assert f(A, 0, B + 8, n, 1.0, Cp, D, None, None) == ALIGN                 # ef 8-B
    assert f(A, 0, B, n, 1.0, Cp + 4, D, None, None) == ALIGN                 # payload
    assert f(A, 0, B, n, 1.0, Cp, D + 2, None, None) == ALIGN                 # scales
    assert f(A, 0, B, n, 1.0, Cp, D, D + 0x100002, None) == ALIGN             # flags
    assert f(A, 0, A + 16, n, 1.0, Cp, D, None, None) == INVALID              # ef overlaps delta
    assert f(A, 0, B, n, 1.0, B + 64, D, None, None) == INVALID               # payload in ef
    assert f(A, 0, B, n, 1.0, Cp, Cp + 16, None, None) == INVALID             # scales in payload
    assert f(A, 0, B, 1 << 44, 1.0, Cp, D, None, None) == INVALID             # too many chunks


def test_compress_multi_argument_errors(lib):
    T = spl._binding._Tensor
    f = lib.spl_ef_compress_multi
    tab = (T * 2)()
    tab[0].delta, tab[0].ef, tab[0].n = A, B, 4096
    tab[1].delta, tab[1].ef, tab[1].n = A + 0x100000, B + 0x100000, 100
    assert f(None, 1, 0, 1.0, Cp, D, None, None) == INVALID
    assert f(tab, 0, 0, 1.0, Cp, D, None, None) == INVALID
    tab[1].ef = B + 0x800        # overlaps tensor 0's error buffer
    assert f(tab, 2, 0, 1.0, Cp, D, None, None) == INVALID
    tab[1].ef = B + 0x100004     # misaligned
    assert f(tab, 2, 0, 1.0, Cp, D, None, None) == ALIGN
    tab[0].n = tab[1].n = 0      # all empty: nothing to do
    assert f(tab, 2, 0, 1.0, None, None, None, None) == OK


def test_decode_argument_errors(lib):
    def f(pl, sc, P, n, mean, theta, lr, flags, stream):   # validation on
        return lib.spl_decode_aggregate(pl, sc, P, n, mean, theta, lr, 1, flags, stream)
    P = 2
    pl = (ctypes.c_void_p * P)(A, A + 0x100000)
    sc = (ctypes.c_void_p * P)(B, B + 0x100000)
    n = 8192
    assert f(pl, sc, 0, n, Cp, None, 0.0, None, None) == INVALID             # P = 0
    assert f(pl, sc, 257, n, Cp, None, 0.0, None, None) == INVALID           # P > max
    assert f(pl, sc, P, 0, Cp, None, 0.0, None, None) == OK                  # empty
    assert f(None, sc, P, n, Cp, None, 0.0, None, None) == INVALID
    assert f(pl, sc, P, n, None, None, 0.0, None, None) == INVALID           # NULL mean
    assert f(pl, sc, P, n, Cp, D, float("nan"), None, None) == INVALID       # lr NaN w/ theta
    assert f(pl, sc, P, n, Cp + 8, None, 0.0, None, None) == ALIGN
    assert f(pl, sc, P, n, Cp, D + 4, 0.7, None, None) == ALIGN
    assert f(pl, sc, P, n, Cp, Cp + 4096, 0.7, None, None) == INVALID        # theta in mean
    pl_bad = (ctypes.c_void_p * P)(A, A + 8)
    assert f(pl_bad, sc, P, n, Cp, None, 0.0, None, None) == ALIGN
    pl_null = (ctypes.c_void_p * P)(A, None)
    assert f(pl_null, sc, P, n, Cp, None, 0.0, None, None) == INVALID
    pl_alias = (ctypes.c_void_p * P)(A, Cp + 4096)                          # record in mean
    assert f(pl_alias, sc, P, n, Cp, None, 0.0, None, None) == INVALID
    assert f(pl, sc, P, n, Cp, None, 0.0, A + 0x100000 + 64, None) == INVALID   # flags in a record
    assert f(pl, sc, P, n, Cp, None, 0.0, B + 4, None) == INVALID           # flags in scales
    # validation off takes the same argument checks
    g = lib.spl_decode_aggregate
    assert g(pl, sc, 0, n, Cp, None, 0.0, 0, None, None) == INVALID
    assert g(pl, sc, P, n, Cp + 8, None, 0.0, 0, None, None) == ALIGN
    assert g(pl, sc, P, 0, Cp, None, 0.0, 0, None, None) == OK


def test_compress_flags_alias_outputs(lib):
    f = lib.spl_ef_compress
    n = 8192
    assert f(A, 0, B, n, 1.0, Cp, D, Cp + 32, None) == INVALID              # flags in payload
    assert f(A, 0, B, n, 1.0, Cp, D, D + 4, None) == INVALID                # flags in scales


def test_decode_stats_alias_records(lib):
    f = lib.spl_decode_aggregate_stats
    P = 2
    pl = (ctypes.c_void_p * P)(A, A + 0x100000)
    sc = (ctypes.c_void_p * P)(B, B + 0x100000)
    n = 8192
    assert f(pl, sc, P, n, Cp, None, 0.0, A + 0x100000 + 16, None, None) == INVALID  # in a record
    assert f(pl, sc, P, n, Cp, None, 0.0, B + 0x100000, None, None) == INVALID       # in scales
    assert f(pl, sc, P, n, Cp, None, 0.0, D, D + 8, None) == INVALID          # flags in stats
    Codec = spl._binding._Codec
    g = lib.spl_decode_aggregate_codec
    c = Codec(2048, 32, 0)
    assert g(ctypes.byref(c), pl, sc, P, n, Cp, None, 0.0, A + 32, None, None) == INVALID


def test_decode_stats_argument_errors(lib):
    f = lib.spl_decode_aggregate_stats
    P = 2
    pl = (ctypes.c_void_p * P)(A, A + 0x100000)
    sc = (ctypes.c_void_p * P)(B, B + 0x100000)
    n = 8192
    assert f(pl, sc, P, n, Cp, None, 0.0, None, None, None) == INVALID      # NULL stats
    assert f(pl, sc, P, n, Cp, None, 0.0, D + 4, None, None) == ALIGN       # stats 4-B
    assert f(pl, sc, P, n, Cp, None, 0.0, Cp + 64, None, None) == INVALID   # stats in mean
    assert f(pl, sc, 0, n, Cp, None, 0.0, D, None, None) == INVALID         # P = 0


def test_codec_sizes_and_argument_errors(lib):
    Codec = spl._binding._Codec
    sizes = {(2048, 32): 52, (4096, 32): 56, (4096, 64): 112, (4096, 128): 224, (8192, 128): 240}
    for (L, k), rb in sizes.items():
        for rule in (0, 1):
            c = Codec(L, k, rule)
            assert lib.spl_codec_record_bytes(ctypes.byref(c)) == rb
            assert lib.spl_codec_num_chunks(ctypes.byref(c), 3 * L + 1) == 4
    assert lib.spl_codec_record_bytes(None) == 112
    assert lib.spl_codec_num_chunks(None, 4097) == 2
    for bad in [(1024, 16, 0), (4096, 64, 2), (4096, 48, 0), (0, 0, 0), (2048, 64, 0)]:
        c = Codec(*bad)
        assert lib.spl_codec_record_bytes(ctypes.byref(c)) == -1
        assert lib.spl_codec_num_chunks(ctypes.byref(c), 100) == 0
    T = spl._binding._Tensor
    tab = (T * 1)()
    tab[0].delta, tab[0].ef, tab[0].n = A, B, 8192
    f = lib.spl_ef_compress_codec
    bad = Codec(1024, 16, 0)
    good = Codec(2048, 32, 1)
    assert f(ctypes.byref(bad), tab, 1, 0, 1.0, Cp, D, None, None) == INVALID
    assert f(ctypes.byref(good), tab, 1, 0, float("nan"), Cp, D, None, None) == INVALID
    assert f(ctypes.byref(good), tab, 1, 0, 1.0, Cp + 4, D, None, None) == ALIGN
    # 4 chunks of 52 bytes: scales placed inside the payload overlap it
    assert f(ctypes.byref(good), tab, 1, 0, 1.0, Cp, Cp + 200, None, None) == INVALID
    g = lib.spl_decode_aggregate_codec
    P = 2
    pl = (ctypes.c_void_p * P)(A, A + 0x100000)
    sc = (ctypes.c_void_p * P)(B, B + 0x100000)
    assert g(ctypes.byref(bad), pl, sc, P, 8192, Cp, None, 0.0, None, None, None) == INVALID
    assert g(ctypes.byref(good), pl, sc, 0, 8192, Cp, None, 0.0, None, None, None) == INVALID
    assert g(ctypes.byref(good), pl, sc, P, 8192, Cp, None, 0.0, D + 4, None, None) == ALIGN
    assert g(ctypes.byref(good), pl, sc, P, 0, Cp, None, 0.0, None, None, None) == OK
    pl_alias = (ctypes.c_void_p * P)(A, Cp + 4096)                           # record in mean
    assert g(ctypes.byref(good), pl_alias, sc, P, 8192, Cp, None, 0.0, None, None, None) == INVALID


def test_pack_unpack_argument_errors(lib):
    assert lib.spl_pack(None, None, 0, None, None) == OK
    assert lib.spl_pack(None, B, 4, Cp, None) == INVALID
    assert lib.spl_pack(A + 1, B, 4, Cp, None) == ALIGN
    assert lib.spl_pack(A, B, 4, Cp + 8, None) == ALIGN
    assert lib.spl_unpack(Cp, 4, None, B, None) == INVALID
    assert lib.spl_unpack(Cp, 4, A, A + 8, None) == INVALID                  # codes in idx


def test_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(4096)
    with pytest.raises(ValueError):
        spl.ef_compress(x, x.clone(), 1.0)


def test_header_is_plain_c_and_links(tmp_path, lib):
    """A C11 program includes spl.h, links libspl.so and calls the host-side entry points."""
    import subprocess
    exe = tmp_path / "abi_consumer"
    src = os.path.join(os.path.dirname(HEADER), "..", "tests", "c", "abi_consumer.c")
    libdir = os.path.dirname(lib_build.LIB_PATH)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.dirname(HEADER), src, "-o", str(exe), "-L", libdir, "-lspl",
                    f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout


def test_calib_argument_errors(lib):
    f = lib.spl_calib_moves
    f.argtypes = [ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 4 + [ctypes.c_size_t] + \
        [ctypes.c_void_p] * 2
    n = 8192
    for persistent in (0, 1):
        g = lambda *a: f(a[0], persistent, *a[1:])   # noqa: E731
        assert g(0, None, None, None, None, 0, None, None) == OK             # empty: no-op
        assert g(2, A, B, Cp, None, n, None, None) == INVALID                # unknown pattern
        assert g(0, A, B, Cp, None, n + 1, None, None) == INVALID            # not whole chunks
        assert g(0, A, None, Cp, None, n, None, None) == INVALID             # sender without in1
        assert g(1, A, B, Cp, None, n, None, None) == INVALID                # receiver, no out1
        assert g(0, A + 4, B, Cp, None, n, None, None) == ALIGN
        assert g(1, A, None, Cp, D + 8, n, None, None) == ALIGN
        assert g(0, A, B, A + 1024, None, n, None, None) == INVALID          # out0 overlaps in0
        assert g(1, A, None, Cp, A + 64, n, None, None) == INVALID           # out1 overlaps in0
        assert g(0, A, B, Cp, None, n, Cp + 16, None) == INVALID             # flags in out0
