"""CPU oracle for the SparseLoCo pseudo-gradient codec.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package.  The product path (the CUDA library and its
binding in ``compressed_pseudo_gradient_gb300``) never imports, links or calls it, and this
package never imports the product: the two share nothing but the seeded input generators.

The arithmetic lives in ``spl_oracle.c`` (plain single-threaded C, built with
``-O2 -ffp-contract=off``); this module only compiles it with gcc, loads it with ctypes and
marshals numpy arrays.  Each wrapper names the page section the C function restates; see the
header of ``spl_oracle.c`` for the readings taken where the pages leave a step open.

bf16 arrays are passed as their uint16 bit patterns (numpy has no bfloat16).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spl_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libspl_oracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None

CHUNK = 4096
TOPK = 64
RECORD_BYTES = 112
FLAG_NONFINITE = 1
FLAG_BAD_RECORD = 2
SCALE_MAX = 0        # s = max |a| / 1.5 (the default)
SCALE_MEAN_ABS = 1   # s = pairwise sum of the chosen |a| / k (variant)
DEFAULT_CODEC = (CHUNK, TOPK, SCALE_MAX)


def build(force: bool = False) -> str:
    """Compile spl_oracle.c into a shared library next to it (if stale) and return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # SPL_ORACLE_LIB: load another build of this oracle instead (the mutation test runs the
        # pins against deliberately broken copies of spl_oracle.c this way)
        lib = ctypes.CDLL(os.environ.get("SPL_ORACLE_LIB") or build())
        vp, i64, f32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_uint32
        lib.orc_num_chunks.argtypes, lib.orc_num_chunks.restype = [i64], i64
        lib.orc_topk_select.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp]
        lib.orc_topk_select.restype = ctypes.c_int
        lib.orc_scale.argtypes, lib.orc_scale.restype = [f32], f32
        lib.orc_code.argtypes, lib.orc_code.restype = [f32, f32], ctypes.c_int
        lib.orc_level.argtypes, lib.orc_level.restype = [ctypes.c_int, f32], f32
        lib.orc_pack.argtypes, lib.orc_pack.restype = [vp, vp, i64, vp], None
        lib.orc_unpack.argtypes, lib.orc_unpack.restype = [vp, i64, vp, vp], None
        lib.orc_ef_compress.argtypes = [vp, ctypes.c_int, vp, i64, f32, vp, vp]
        lib.orc_ef_compress.restype = u32
        lib.orc_decode_aggregate.argtypes = [vp, vp, ctypes.c_int, i64, vp, vp, f32]
        lib.orc_decode_aggregate.restype = u32
        lib.orc_peer_stats.argtypes = [vp, vp, ctypes.c_int, i64, vp, vp, vp, vp, vp]
        lib.orc_peer_stats.restype = None
        ci = ctypes.c_int
        lib.orc_codec_record_bytes.argtypes, lib.orc_codec_record_bytes.restype = [ci, ci], ci
        lib.orc_num_chunks_codec.argtypes, lib.orc_num_chunks_codec.restype = [ci, i64], i64
        lib.orc_pairwise_sum.argtypes, lib.orc_pairwise_sum.restype = [vp, ci], f32
        lib.orc_pack_codec.argtypes, lib.orc_pack_codec.restype = [ci, ci, vp, vp, i64, vp], ci
        lib.orc_unpack_codec.argtypes, lib.orc_unpack_codec.restype = [ci, ci, vp, i64, vp, vp], ci
        lib.orc_ef_compress_codec.argtypes = [ci, ci, ci, vp, ci, vp, i64, f32, vp, vp]
        lib.orc_ef_compress_codec.restype = u32
        lib.orc_decode_aggregate_codec.argtypes = [ci, ci, vp, vp, ci, i64, vp, vp, f32]
        lib.orc_decode_aggregate_codec.restype = u32
        lib.orc_peer_stats_codec.argtypes = [ci, ci, vp, vp, ci, i64, vp, vp, vp, vp, vp]
        lib.orc_peer_stats_codec.restype = ci
        for name in ("orc_chunk", "orc_topk", "orc_record_bytes"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def constants() -> dict:
    """Chunk length, k and record size as the C oracle states them."""
    lib = _load()
    return {"chunk": lib.orc_chunk(), "topk": lib.orc_topk(),
            "record_bytes": lib.orc_record_bytes()}


def _codec(codec) -> tuple[int, int, int]:
    """(L, k, rule) of a codec argument (None = the default 4096 / 64 / max-abs codec)."""
    if codec is None:
        return DEFAULT_CODEC
    L, k, rule = (int(x) for x in codec)
    if _load().orc_codec_record_bytes(L, k) < 0 or rule not in (SCALE_MAX, SCALE_MEAN_ABS):
        raise ValueError(f"not a codec: {codec}")
    return L, k, rule


def record_bytes(codec=None) -> int:
    """Bytes of one record: ceil(k * (2 + ceil(log2 L)) / 8)."""
    L, k, _ = _codec(codec)
    return int(_load().orc_codec_record_bytes(L, k))


def num_chunks(n: int, codec=None) -> int:
    L, _, _ = _codec(codec)
    return int(_load().orc_num_chunks_codec(L, n))


def pairwise_sum(x: np.ndarray) -> np.float32:
    """Pairwise (recursive halving) fp32 sum, the mean-abs scale rule's summation."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.size >= 1
    return np.float32(_load().orc_pairwise_sum(_ptr(x), x.size))


def topk_select(a: np.ndarray, k: int) -> tuple[np.ndarray, int]:
    """Chunk top-k by |a| (ties to the lower index), ascending; also the first-ranked index.

    The Sparse Frontier, "SparseLoCo: Three Compression Levers in One Pass", item 1.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.zeros(k, dtype=np.int32)
    top = _load().orc_topk_select(_ptr(a), a.size, k, _ptr(out))
    return out, int(top)


def scale(m: float) -> np.float32:
    return np.float32(_load().orc_scale(m))


def code(v: float, s: float) -> int:
    return int(_load().orc_code(v, s))


def level(c: int, s: float) -> np.float32:
    return np.float32(_load().orc_level(c, s))


def pack(idx: np.ndarray, codes: np.ndarray, codec=None) -> np.ndarray:
    """(idx[C,k] u16, codes[C,k] u8) -> payload[C,record_bytes] u8 (bit-at-a-time writer)."""
    L, k, _ = _codec(codec)
    idx = np.ascontiguousarray(idx, dtype=np.uint16).reshape(-1, k)
    codes = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1, k)
    C = idx.shape[0]
    out = np.zeros((C, record_bytes(codec)), dtype=np.uint8)
    assert _load().orc_pack_codec(L, k, _ptr(idx), _ptr(codes), C, _ptr(out))
    return out


def unpack(payload: np.ndarray, codec=None) -> tuple[np.ndarray, np.ndarray]:
    L, k, _ = _codec(codec)
    payload = np.ascontiguousarray(payload, dtype=np.uint8).reshape(-1, record_bytes(codec))
    C = payload.shape[0]
    idx = np.zeros((C, k), dtype=np.uint16)
    codes = np.zeros((C, k), dtype=np.uint8)
    assert _load().orc_unpack_codec(L, k, _ptr(payload), C, _ptr(idx), _ptr(codes))
    return idx, codes


def ef_compress(delta: np.ndarray, ef: np.ndarray, beta: float, *, bf16: bool = False,
                codec=None):
    """One sender round; ``ef`` (fp32) is updated in place.

    ``delta`` is fp32, or with ``bf16=True`` a uint16 array of bf16 bit patterns.  ``codec``
    is (L, k, rule) or None for the default codec.
    Returns (payload[C,record_bytes] u8, scales[C] f32, flags).
    """
    L, k, rule = _codec(codec)
    if bf16:
        delta = np.ascontiguousarray(delta, dtype=np.uint16)
    else:
        delta = np.ascontiguousarray(delta, dtype=np.float32)
    assert ef.dtype == np.float32 and ef.flags["C_CONTIGUOUS"] and ef.size == delta.size
    n = delta.size
    C = num_chunks(n, codec)
    payload = np.zeros((C, record_bytes(codec)), dtype=np.uint8)
    scales = np.zeros(C, dtype=np.float32)
    flags = _load().orc_ef_compress_codec(L, k, rule, _ptr(delta), 1 if bf16 else 0, _ptr(ef),
                                          n, np.float32(beta), _ptr(payload), _ptr(scales))
    return payload, scales, int(flags)


def _peer_arrays(payloads, scales, n, codec):
    P = len(payloads)
    assert P == len(scales) and P >= 1
    C = num_chunks(n, codec)
    rb = record_bytes(codec)
    pl = [np.ascontiguousarray(p, dtype=np.uint8).reshape(C, rb) for p in payloads]
    sc = [np.ascontiguousarray(s, dtype=np.float32).reshape(C) for s in scales]
    parr = (ctypes.c_void_p * P)(*[_ptr(p) for p in pl])
    sarr = (ctypes.c_void_p * P)(*[_ptr(s) for s in sc])
    return P, pl, sc, parr, sarr


def decode_aggregate(payloads, scales, n: int, theta: np.ndarray | None = None,
                     lr: float = 0.0, codec=None):
    """Mean of P peers' decoded records; with ``theta`` also theta -= lr * mean (in place).

    Returns (mean[n] f32, flags).
    """
    L, k, _ = _codec(codec)
    P, pl, sc, parr, sarr = _peer_arrays(payloads, scales, n, codec)
    mean = np.zeros(n, dtype=np.float32)
    tptr = None
    if theta is not None:
        assert theta.dtype == np.float32 and theta.flags["C_CONTIGUOUS"] and theta.size == n
        tptr = _ptr(theta)
    flags = _load().orc_decode_aggregate_codec(L, k, parr, sarr, P, n, _ptr(mean), tptr,
                                               np.float32(lr))
    return mean, int(flags)


def peer_stats(payloads, scales, n: int, codec=None) -> dict:
    """Per-peer statistics of the accepted records (rejected, big, negative, max_scale, sumsq).

    The Sparse Frontier, "What the Blockchain Does (and Doesn't Do)": crafted sparse updates
    look different from naturally concentrated ones.
    """
    L, k, _ = _codec(codec)
    P, pl, sc, parr, sarr = _peer_arrays(payloads, scales, n, codec)
    out = {"rejected": np.zeros(P, np.uint32), "big": np.zeros(P, np.uint32),
           "negative": np.zeros(P, np.uint32), "max_scale": np.zeros(P, np.float32),
           "sumsq": np.zeros(P, np.float64)}
    assert _load().orc_peer_stats_codec(L, k, parr, sarr, P, n, _ptr(out["rejected"]),
                                        _ptr(out["big"]), _ptr(out["negative"]),
                                        _ptr(out["max_scale"]), _ptr(out["sumsq"]))
    return out
