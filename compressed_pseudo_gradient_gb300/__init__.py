"""SparseLoCo pseudo-gradient codec on one GB300 (sm_103a).

A thin binding over the C ABI of ``libspl.so`` (declared in ``include/spl.h``): each function
checks the torch tensors it is given, passes their device pointers and the current CUDA
stream to the library, and raises on a non-OK status.  Every step of the codec runs in the
library's CUDA kernels; there is no CPU path.  The library is loaded on first use, and a
missing or unloadable library raises instead of falling back.

The codec: "The Sparse Frontier: SparseLoCo and the Compression Math Behind Permissionless
Pre-Training", "SparseLoCo: Three Compression Levers in One Pass" and "Why Extreme Sparsity
Doesn't Break Convergence".
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    CALIB_RECEIVER_MOVES,
    CALIB_SENDER_MOVES,
    CHUNK,
    FLAG_BAD_RECORD,
    FLAG_COPY_PENDING,
    FLAG_NONFINITE,
    FLAG_TIMEOUT,
    MAX_PEERS,
    RECORD_BYTES,
    SCALE_MAX_ABS,
    SCALE_MEAN_ABS,
    TOPK,
    SplError,
    calib_moves,
    checked_library_path,
    debug_words,
    decode_aggregate,
    ef_compress,
    ef_compress_multi,
    flags_status,
    library,
    library_path,
    new_peer_stats,
    num_chunks,
    pack,
    read_peer_stats,
    record_bytes,
    unpack,
    use_library,
)
