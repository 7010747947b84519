"""One pseudo-gradient spread over the GPUs of a node: chunk-sharded sender and receiver.

The codec works chunk by chunk ("The Sparse Frontier: SparseLoCo and the Compression Math
Behind Permissionless Pre-Training", "SparseLoCo: Three Compression Levers in One Pass", item
1: non-overlapping chunks of 4096 values, each compressed on its own), so a tensor split on
chunk boundaries compresses with no communication at all:

- rank g of G owns chunks [g C / G, (g + 1) C / G) of the tensor's C chunks, and the matching
  slice of the pseudo-gradient and of the error-feedback buffer (only the last rank's slice
  can end inside a chunk: the tensor's own tail chunk);
- each rank compresses its slice with the single-GPU sender (``spl_ef_compress`` on the
  slice's pointers); its records are exactly the whole tensor's records of those chunks;
- one exchange step, an all-gather of the fixed-size records (112 B + a 4 B scale per chunk),
  gives every rank the peer's whole payload: what the pages' peers send over the internet and
  aggregate ("AllReduce aggregation" across the active peers, same section, and "Why Extreme
  Sparsity Doesn't Break Convergence", "Sparse aggregation can improve model quality");
- on the receiving side each rank decodes and averages all peers' records of its own chunk
  range into its slice of the mean (and applies the outer step to its slice of theta), with no
  dense reduction between ranks.

The functions here are host logic over torch tensors: slicing on chunk boundaries, the record
all-gather (``torch.distributed``: NCCL between GPUs, gloo on CPU) and the choice of record
rows.  The codec's arithmetic runs in the CUDA library (``ef_compress`` and
``decode_aggregate`` of this package, the defaults of the ``compress`` and ``decode``
arguments); those arguments exist so that the partitioning and the exchange can be checked on
CPU ranks with another implementation of the same two calls.
"""
from __future__ import annotations

import torch

from . import _binding

CHUNK = _binding.CHUNK
RECORD_BYTES = _binding.RECORD_BYTES


def _world(group=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        return dist.get_rank(group), dist.get_world_size(group)
    return 0, 1


def shard_chunks(C: int, world: int, rank: int) -> tuple[int, int]:
    """Chunk range [c0, c1) of `rank` among `world` ranks: [rank C / world, (rank + 1) C / world)
    (contiguous, in rank order, sizes differing by at most one)."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    return rank * C // world, (rank + 1) * C // world


def shard_range(n: int, world: int, rank: int) -> tuple[int, int]:
    """Element range [lo, hi) of `rank`'s slice of an n-value tensor: its chunk range in values,
    cut at n.  lo is a multiple of 4096 (or n, for a rank left without chunks when there are
    fewer chunks than ranks), so the slice's own chunks are the tensor's chunks [c0, c1)."""
    C = (n + CHUNK - 1) // CHUNK
    c0, c1 = shard_chunks(C, world, rank)
    return min(n, c0 * CHUNK), min(n, c1 * CHUNK)


def compress_shard(delta: torch.Tensor, ef: torch.Tensor, beta: float, *, compress=None,
                   flags=None):
    """This rank's sender round on its slice of the tensor.

    delta, ef: this rank's slices (``shard_range`` of the whole tensor), the error buffer
    updated in place.  Returns (payload [c1 - c0, 112] uint8, scales [c1 - c0] fp32): the
    whole tensor's records of chunks [c0, c1).  ``compress(delta, ef, beta, flags=...)``
    defaults to the CUDA library's ``ef_compress``."""
    if delta.numel() != ef.numel():
        raise ValueError("delta and ef slices differ in size")
    fn = compress if compress is not None else _binding.ef_compress
    return fn(delta, ef, beta, flags=flags)


def gather_records(payload: torch.Tensor, scales: torch.Tensor, C: int, *, group=None):
    """All-gather of every rank's records: returns (payload [C, 112], scales [C]) of the whole
    tensor, chunks in order, on every rank.

    Each rank contributes its chunk range's records, packed with their scales as 116-byte
    rows and padded to ceil(C / world) rows, so every rank sends the same number of bytes; the
    padding rows are dropped after the gather.  Without a process group (one rank) the records
    are returned as they are."""
    rank, world = _world(group)
    c0, c1 = shard_chunks(C, world, rank)
    if payload.shape != (c1 - c0, RECORD_BYTES) or scales.numel() != c1 - c0:
        raise ValueError(f"rank {rank}: expected records of chunks [{c0}, {c1})")
    if world == 1:
        return payload, scales
    import torch.distributed as dist
    m = (C + world - 1) // world
    row = RECORD_BYTES + 4
    mine = torch.zeros((m, row), dtype=torch.uint8, device=payload.device)
    if c1 > c0:
        mine[: c1 - c0, :RECORD_BYTES] = payload
        mine[: c1 - c0, RECORD_BYTES:] = scales.contiguous().view(torch.uint8).view(-1, 4)
    parts = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(parts, mine, group=group)
    rows = []
    for r in range(world):
        a, b = shard_chunks(C, world, r)
        rows.append(parts[r][: b - a])
    full = torch.cat(rows)
    out_payload = full[:, :RECORD_BYTES].contiguous()
    out_scales = full[:, RECORD_BYTES:].contiguous().view(torch.float32).view(-1)
    return out_payload, out_scales


def decode_shard(payloads, scales, n: int, *, mean=None, theta=None, lr: float = 0.0,
                 group=None, decode=None, flags=None, validate: bool = True):
    """This rank's slice of the P-peer mean (and of the outer step on theta).

    payloads, scales: the P peers' records of the WHOLE tensor ([C, 112] and [C] each, e.g.
    from ``gather_records``) or of this rank's chunk range only ([c1 - c0, 112] and
    [c1 - c0]); theta, if given, is this rank's slice, updated in place.  Returns the mean's
    slice [hi - lo] fp32.  ``decode(payloads, scales, n, mean=, theta=, lr=, flags=,
    validate=)`` defaults to the CUDA library's ``decode_aggregate``."""
    rank, world = _world(group)
    C = (n + CHUNK - 1) // CHUNK
    c0, c1 = shard_chunks(C, world, rank)
    lo, hi = shard_range(n, world, rank)
    pls, scs = [], []
    for p, (pl, sc) in enumerate(zip(payloads, scales)):
        if pl.shape[0] == C and sc.numel() == C:
            pl, sc = pl[c0:c1], sc[c0:c1]   # rows of this range: still 16-byte aligned
        elif pl.shape[0] != c1 - c0 or sc.numel() != c1 - c0:
            raise ValueError(f"peer {p}: records of neither the tensor nor chunks [{c0}, {c1})")
        pls.append(pl)
        scs.append(sc)
    if theta is not None and theta.numel() != hi - lo:
        raise ValueError(f"theta slice has {theta.numel()} values, expected {hi - lo}")
    fn = decode if decode is not None else _binding.decode_aggregate
    return fn(pls, scs, hi - lo, mean=mean, theta=theta, lr=lr, flags=flags, validate=validate)
