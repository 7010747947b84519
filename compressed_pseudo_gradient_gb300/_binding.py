"""ctypes binding of libspl.so: argument marshalling only (torch tensors -> device pointers).

Function names follow the C ABI in include/spl.h without the ``spl_`` prefix.  Outputs that
the caller does not pass are allocated with torch on the input's device; the library itself
allocates nothing.  All work is enqueued on ``torch.cuda.current_stream()`` of the inputs'
device and is not waited for.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

CHUNK = 4096
TOPK = 64
RECORD_BYTES = 112
MAX_PEERS = 256
FLAG_NONFINITE = 1
FLAG_BAD_RECORD = 2
FLAG_TIMEOUT = 4
FLAG_COPY_PENDING = 8
SCALE_MAX_ABS = 0     # s = max |a| / 1.5 (the default)
SCALE_MEAN_ABS = 1    # s = pairwise sum of the chosen |a| / k (codec variant)

_F32, _BF16 = 0, 1
_lock = threading.Lock()
_lib = None
_lib_path = None   # None: the library this package builds (libspl.so)


class SplError(RuntimeError):
    """A non-OK status from libspl (argument error, alignment error or CUDA failure)."""

    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        lib = _lib
        text = lib.spl_status_string(status).decode() if lib is not None else str(status)
        msg = f"{fn}: {text} (status {status})"
        if status == 3:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)
        self.status = status
        self.cuda_error = cuda_error


class _Tensor(ctypes.Structure):
    _fields_ = [("delta", ctypes.c_void_p), ("ef", ctypes.c_void_p), ("n", ctypes.c_size_t)]


class _Codec(ctypes.Structure):
    _fields_ = [("chunk", ctypes.c_uint32), ("topk", ctypes.c_uint32),
                ("scale_rule", ctypes.c_uint32)]


def library_path() -> str:
    return _lib_path or _build.LIB_PATH


def checked_library_path() -> str:
    """Path of the checked build (libspl_checked.so): the same calls, with every kernel memory
    index tested before the access (include/spl_checked.h)."""
    return _build.CHECKED_LIB_PATH


def use_library(path=None):
    """Makes later calls go through another build of the library, e.g. checked_library_path();
    None returns to libspl.so.  Returns the previous selection.  Both builds are built together
    by build.build(); work already enqueued is not affected."""
    global _lib, _lib_path
    with _lock:
        prev = _lib_path
        _lib_path = path
        _lib = None
        return prev


def library():
    """The loaded libspl.so, or the build chosen with use_library (built first if missing or
    older than its sources)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _lib_path or _build.LIB_PATH
        if _build.is_stale():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"{os.path.basename(path)} is missing at {path}; the CUDA "
                               f"library must be built")
        lib = ctypes.CDLL(path)
        vp, sz, ci, cf = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
        lib.spl_num_chunks.argtypes, lib.spl_num_chunks.restype = [sz], sz
        lib.spl_status_string.argtypes, lib.spl_status_string.restype = [ci], ctypes.c_char_p
        lib.spl_last_cuda_error.argtypes, lib.spl_last_cuda_error.restype = [], ci
        lib.spl_ef_compress.argtypes = [vp, ci, vp, sz, cf, vp, vp, vp, vp]
        lib.spl_ef_compress.restype = ci
        lib.spl_ef_compress_multi.argtypes = [ctypes.POINTER(_Tensor), ci, ci, cf, vp, vp, vp, vp]
        lib.spl_ef_compress_multi.restype = ci
        lib.spl_flags_status.argtypes, lib.spl_flags_status.restype = [ctypes.c_uint32], ci
        lib.spl_decode_aggregate.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), ci, sz, vp,
                                             vp, cf, ci, vp, vp]
        lib.spl_decode_aggregate.restype = ci
        lib.spl_decode_aggregate_stats.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), ci,
                                                   sz, vp, vp, cf, vp, vp, vp]
        lib.spl_decode_aggregate_stats.restype = ci
        cp = ctypes.POINTER(_Codec)
        lib.spl_codec_record_bytes.argtypes = [cp]
        lib.spl_codec_record_bytes.restype = ctypes.c_int64
        lib.spl_codec_num_chunks.argtypes, lib.spl_codec_num_chunks.restype = [cp, sz], sz
        lib.spl_ef_compress_codec.argtypes = [cp, ctypes.POINTER(_Tensor), ci, ci, cf, vp, vp,
                                              vp, vp]
        lib.spl_ef_compress_codec.restype = ci
        lib.spl_decode_aggregate_codec.argtypes = [cp, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                                   ci, sz, vp, vp, cf, vp, vp, vp]
        lib.spl_decode_aggregate_codec.restype = ci
        lib.spl_pack.argtypes, lib.spl_pack.restype = [vp, vp, sz, vp, vp], ci
        lib.spl_unpack.argtypes, lib.spl_unpack.restype = [vp, sz, vp, vp, vp], ci
        lib.spl_calib_moves.argtypes = [ci, ci, vp, vp, vp, vp, sz, vp, vp]
        lib.spl_calib_moves.restype = ci
        if hasattr(lib, "spl_debug_read"):   # the checked build
            lib.spl_debug_read.argtypes, lib.spl_debug_read.restype = [vp, ci], ci
        _lib = lib
        return lib


DEBUG_WORDS = 16
DEBUG_NAMES = {0: "sites", 1: "first_site", 2: "first_index", 3: "failures", 8: "chunks",
               9: "whole", 10: "rank32", 11: "rank64", 12: "full_scan", 13: "generic"}


def debug_words(reset: bool = False) -> dict:
    """Checked build only (use_library(checked_library_path())): the debug words of every kernel
    since the last reset, by name (spl_debug_read); waits for the device."""
    lib = library()
    if not hasattr(lib, "spl_debug_read"):
        raise RuntimeError("debug_words needs the checked build of the library")
    out = (ctypes.c_uint32 * DEBUG_WORDS)()
    _check("spl_debug_read", lib.spl_debug_read(out, 1 if reset else 0))
    return {name: int(out[i]) for i, name in DEBUG_NAMES.items()}


def flags_status(flags) -> int:
    """The status a device flags word stands for (spl_flags_status): 0 (ok), 4 (non-finite
    accumulated value), 5 (rejected record) or 6 (a kernel stopped on a bounded wait).
    ``flags`` is the 1-element int32 tensor the calls OR into, or its value; reading a tensor
    synchronises with its device."""
    if isinstance(flags, torch.Tensor):
        flags = int(flags.item())
    return int(library().spl_flags_status(int(flags) & 0xffffffff))


def _check(fn: str, status: int):
    if status != 0:
        lib = library()
        raise SplError(fn, status, lib.spl_last_cuda_error() if status == 3 else 0)


def _cuda(t: torch.Tensor, name: str, dtypes) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}; expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _stream(dev: torch.device) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def _flags_ptr(flags, dev):
    if flags is None:
        return None
    _cuda(flags, "flags", (torch.int32,))
    if flags.numel() < 1 or flags.device != dev:
        raise ValueError("flags must be a 1-element int32 tensor on the inputs' device")
    return flags.data_ptr()


def _codec(codec):
    """ctypes codec of a (L, k, rule) tuple, or None for the default codec."""
    if codec is None:
        return None
    L, k, rule = (int(x) for x in codec)
    c = _Codec(L, k, rule)
    if library().spl_codec_record_bytes(ctypes.byref(c)) < 0:
        raise ValueError(f"codec {tuple(codec)} is not implemented by libspl")
    return c


def record_bytes(codec=None) -> int:
    """Bytes of one record: 112 for the default codec, k * (2 + log2 L) / 8 for a variant."""
    c = _codec(codec)
    return RECORD_BYTES if c is None else int(library().spl_codec_record_bytes(ctypes.byref(c)))


def num_chunks(n: int, codec=None) -> int:
    L = CHUNK if codec is None else int(codec[0])
    return (int(n) + L - 1) // L


def _ef_tensor(ef: torch.Tensor, dev: torch.device) -> torch.Tensor:
    """The error buffer: an fp32 CUDA tensor on dev, or a pinned CPU tensor (host-resident)."""
    if isinstance(ef, torch.Tensor) and not ef.is_cuda:
        if not ef.is_pinned():
            raise ValueError("a CPU error buffer must be in pinned memory")
        if ef.dtype != torch.float32 or not ef.is_contiguous():
            raise ValueError("the error buffer must be contiguous fp32")
        return ef
    _cuda(ef, "ef", (torch.float32,))
    if ef.device != dev:
        raise ValueError("delta and ef must be on the same device")
    return ef


def ef_compress(delta: torch.Tensor, ef: torch.Tensor, beta: float, *, payload=None,
                scales=None, flags=None, codec=None):
    """One sender round (spl_ef_compress); ``ef`` is updated in place.

    delta: fp32 or bf16 CUDA tensor of n values; ef: fp32 tensor of n values, on the same
    GPU or in pinned host memory (then read and written over the host link).  ``codec``:
    (L, k, rule) of a codec variant (spl_ef_compress_codec), or None for the default codec.
    Returns (payload uint8 [C, record_bytes], scales fp32 [C]).
    """
    if codec is not None:
        return ef_compress_multi([delta], [ef], beta, payload=payload, scales=scales,
                                 flags=flags, codec=codec)
    lib = library()
    _cuda(delta, "delta", (torch.float32, torch.bfloat16))
    _ef_tensor(ef, delta.device)
    if ef.numel() != delta.numel():
        raise ValueError("delta and ef must have the same size")
    dev = delta.device
    n = delta.numel()
    C = num_chunks(n)
    if payload is None:
        payload = torch.empty((C, RECORD_BYTES), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(C, dtype=torch.float32, device=dev)
    _cuda(payload, "payload", (torch.uint8,))
    _cuda(scales, "scales", (torch.float32,))
    if payload.numel() < C * RECORD_BYTES or scales.numel() < C:
        raise ValueError("payload/scales too small")
    with torch.cuda.device(dev):
        st = lib.spl_ef_compress(delta.data_ptr(), _BF16 if delta.dtype == torch.bfloat16 else _F32,
                                 ef.data_ptr(), n, float(beta), payload.data_ptr(),
                                 scales.data_ptr(), _flags_ptr(flags, dev), _stream(dev))
    _check("spl_ef_compress", st)
    return payload, scales


def ef_compress_multi(deltas, efs, beta: float, *, payload=None, scales=None, flags=None,
                      codec=None):
    """One sender round over a list of tensors, each chunked on its own (spl_ef_compress_multi,
    or spl_ef_compress_codec for a codec variant (L, k, rule)).

    Returns (payload uint8 [sum C_i, record_bytes], scales fp32 [sum C_i]) in tensor order.
    """
    lib = library()
    cd = _codec(codec)
    rb = record_bytes(codec)
    if len(deltas) != len(efs) or not deltas:
        raise ValueError("deltas and efs must be non-empty lists of equal length")
    dtype = deltas[0].dtype
    dev = deltas[0].device
    table = (_Tensor * len(deltas))()
    C = 0
    for i, (d, e) in enumerate(zip(deltas, efs)):
        _cuda(d, f"deltas[{i}]", (torch.float32, torch.bfloat16))
        _ef_tensor(e, dev)
        if d.dtype != dtype or d.device != dev or e.numel() != d.numel():
            raise ValueError(f"tensor {i}: dtype/device/size mismatch")
        table[i].delta = d.data_ptr() if d.numel() else None
        table[i].ef = e.data_ptr() if e.numel() else None
        table[i].n = d.numel()
        C += num_chunks(d.numel(), codec)
    if payload is None:
        payload = torch.empty((C, rb), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(C, dtype=torch.float32, device=dev)
    _cuda(payload, "payload", (torch.uint8,))
    _cuda(scales, "scales", (torch.float32,))
    if payload.numel() < C * rb or scales.numel() < C:
        raise ValueError("payload/scales too small")
    args = (table, len(deltas), _BF16 if dtype == torch.bfloat16 else _F32, float(beta),
            payload.data_ptr() if C else None, scales.data_ptr() if C else None,
            _flags_ptr(flags, dev), _stream(dev))
    with torch.cuda.device(dev):
        if cd is None:
            st = lib.spl_ef_compress_multi(*args)
        else:
            st = lib.spl_ef_compress_codec(ctypes.byref(cd), *args)
    _check("spl_ef_compress_multi" if cd is None else "spl_ef_compress_codec", st)
    return payload, scales


PEER_STATS_BYTES = 24


def new_peer_stats(P: int, device) -> torch.Tensor:
    """A zeroed device buffer for P spl_peer_stats entries (uint8 [P, 24])."""
    return torch.zeros((P, PEER_STATS_BYTES), dtype=torch.uint8, device=device)


def read_peer_stats(stats: torch.Tensor) -> dict:
    """Host copy of a peer-statistics buffer as numpy arrays: rejected, big, negative (uint32),
    max_scale (float32), sumsq (float64)."""
    import numpy as np
    raw = stats.detach().cpu().numpy().reshape(-1, PEER_STATS_BYTES)
    u = raw[:, :12].copy().view(np.uint32)
    return {"rejected": u[:, 0].copy(), "big": u[:, 1].copy(), "negative": u[:, 2].copy(),
            "max_scale": raw[:, 12:16].copy().view(np.float32)[:, 0].copy(),
            "sumsq": raw[:, 16:24].copy().view(np.float64)[:, 0].copy()}


def decode_aggregate(payloads, scales, n: int, *, mean=None, theta=None, lr: float = 0.0,
                     flags=None, stats=None, codec=None, validate: bool = True):
    """Mean of P peers' decoded records, optionally fused with theta -= lr * mean in place
    (spl_decode_aggregate).  With ``stats`` (from new_peer_stats, accumulated into), also the
    per-peer statistics (spl_decode_aggregate_stats).  ``codec``: (L, k, rule) of a codec
    variant (spl_decode_aggregate_codec), or None.  ``validate=False`` skips the record checks
    (default codec without statistics only; the statistics and the variants always check).
    Returns mean (fp32 [n])."""
    lib = library()
    cd = _codec(codec)
    rb = record_bytes(codec)
    if not validate and (cd is not None or stats is not None):
        raise ValueError("validate=False is only offered by the default codec without stats")
    P = len(payloads)
    if P != len(scales) or P < 1:
        raise ValueError("payloads and scales must be non-empty lists of equal length")
    dev = payloads[0].device
    C = num_chunks(n, codec)
    for i, (p, s) in enumerate(zip(payloads, scales)):
        _cuda(p, f"payloads[{i}]", (torch.uint8,))
        _cuda(s, f"scales[{i}]", (torch.float32,))
        if p.device != dev or s.device != dev or p.numel() < C * rb or s.numel() < C:
            raise ValueError(f"peer {i}: device mismatch or arrays too small")
    if mean is None:
        mean = torch.empty(n, dtype=torch.float32, device=dev)
    _cuda(mean, "mean", (torch.float32,))
    if mean.numel() < n or mean.device != dev:
        raise ValueError("mean too small or on another device")
    tptr = None
    if theta is not None:
        _cuda(theta, "theta", (torch.float32,))
        if theta.numel() < n or theta.device != dev:
            raise ValueError("theta too small or on another device")
        tptr = theta.data_ptr()
    parr = (ctypes.c_void_p * P)(*[p.data_ptr() for p in payloads])
    sarr = (ctypes.c_void_p * P)(*[s.data_ptr() for s in scales])
    sptr = None
    if stats is not None:
        _cuda(stats, "stats", (torch.uint8,))
        if stats.numel() < P * PEER_STATS_BYTES or stats.device != dev:
            raise ValueError("stats must hold P x 24 bytes on the inputs' device")
        sptr = stats.data_ptr()
    with torch.cuda.device(dev):
        if cd is not None:
            fn = "spl_decode_aggregate_codec"
            st = lib.spl_decode_aggregate_codec(ctypes.byref(cd), parr, sarr, P, int(n),
                                                mean.data_ptr(), tptr, float(lr), sptr,
                                                _flags_ptr(flags, dev), _stream(dev))
        elif stats is None:
            fn = "spl_decode_aggregate"
            st = lib.spl_decode_aggregate(parr, sarr, P, int(n), mean.data_ptr(), tptr, float(lr),
                                          1 if validate else 0, _flags_ptr(flags, dev),
                                          _stream(dev))
        else:
            fn = "spl_decode_aggregate_stats"
            st = lib.spl_decode_aggregate_stats(parr, sarr, P, int(n), mean.data_ptr(), tptr,
                                                float(lr), sptr, _flags_ptr(flags, dev),
                                                _stream(dev))
    _check(fn, st)
    return mean


def pack(idx: torch.Tensor, codes: torch.Tensor, *, payload=None):
    """(idx int16/uint16-as-int16 [C, 64], codes uint8 [C, 64]) -> payload uint8 [C, 112]."""
    lib = library()
    _cuda(idx, "idx", (torch.int16,))
    _cuda(codes, "codes", (torch.uint8,))
    C = idx.numel() // TOPK
    if idx.numel() != C * TOPK or codes.numel() != C * TOPK:
        raise ValueError("idx and codes must hold C x 64 entries")
    dev = idx.device
    if payload is None:
        payload = torch.empty((C, RECORD_BYTES), dtype=torch.uint8, device=dev)
    _cuda(payload, "payload", (torch.uint8,))
    with torch.cuda.device(dev):
        st = lib.spl_pack(idx.data_ptr(), codes.data_ptr(), C, payload.data_ptr(), _stream(dev))
    _check("spl_pack", st)
    return payload


def unpack(payload: torch.Tensor, *, idx=None, codes=None):
    """payload uint8 [C, 112] -> (idx int16 [C, 64] holding 0..4095, codes uint8 [C, 64])."""
    lib = library()
    _cuda(payload, "payload", (torch.uint8,))
    C = payload.numel() // RECORD_BYTES
    if payload.numel() != C * RECORD_BYTES:
        raise ValueError("payload must hold C x 112 bytes")
    dev = payload.device
    if idx is None:
        idx = torch.empty((C, TOPK), dtype=torch.int16, device=dev)
    if codes is None:
        codes = torch.empty((C, TOPK), dtype=torch.uint8, device=dev)
    _cuda(idx, "idx", (torch.int16,))
    _cuda(codes, "codes", (torch.uint8,))
    with torch.cuda.device(dev):
        st = lib.spl_unpack(payload.data_ptr(), C, idx.data_ptr(), codes.data_ptr(), _stream(dev))
    _check("spl_unpack", st)
    return idx, codes


CALIB_SENDER_MOVES = 0
CALIB_RECEIVER_MOVES = 1


def calib_moves(pattern: int, in0: torch.Tensor, in1=None, *, out0=None, out1=None, flags=None,
                persistent: bool = False):
    """Data-movement reference kernels (include/spl_calib.h), for roofline calibration, not the
    codec: CALIB_SENDER_MOVES moves the sender's bytes (out0 = in0 + in1, in0 and in1 staged
    by bulk copies, plain stores); CALIB_RECEIVER_MOVES the receiver's (out0 = -in0,
    out1 = in0, in0 staged, plain stores).  Chunks in the codec kernels' order, or with
    persistent=True in one persistent wave.  fp32 CUDA tensors, numel a multiple of 4096.
    Returns out0 (sender) or (out0, out1) (receiver)."""
    lib = library()
    sender = pattern == CALIB_SENDER_MOVES
    if not sender and pattern != CALIB_RECEIVER_MOVES:
        raise ValueError(f"unknown calibration pattern {pattern}")
    _cuda(in0, "in0", (torch.float32,))
    dev, n = in0.device, in0.numel()
    if sender:
        if in1 is None:
            raise ValueError("the sender pattern takes in1")
        _cuda(in1, "in1", (torch.float32,))
        if in1.numel() != n or in1.device != dev:
            raise ValueError("in1 must match in0")
    if out0 is None:
        out0 = torch.empty_like(in0)
    if not sender and out1 is None:
        out1 = torch.empty_like(in0)
    for t, name in ((out0, "out0"), (out1, "out1")):
        if t is not None:
            _cuda(t, name, (torch.float32,))
            if t.numel() != n or t.device != dev:
                raise ValueError(f"{name} must match in0")
    with torch.cuda.device(dev):
        st = lib.spl_calib_moves(pattern, int(bool(persistent)), in0.data_ptr(),
                                 in1.data_ptr() if sender else None,
                                 out0.data_ptr(), None if sender else out1.data_ptr(), n,
                                 _flags_ptr(flags, dev), _stream(dev))
    _check("spl_calib_moves", st)
    return out0 if sender else (out0, out1)
