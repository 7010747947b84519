"""Chunk-sharded sender and receiver (compressed_pseudo_gradient_gb300.sharded) on CPU ranks.

Two and three gloo ranks each take their slice of one tensor, compress it, all-gather the
records and decode their own chunk range of several peers' records.  The two compute calls
are the oracle's here (the partitioning and the exchange are what is under test; the CUDA
library's calls on slices are checked against whole-tensor calls on the GPU in
test_gpu_sharded.py).  Every rank must end with the oracle's whole-tensor records byte for
byte, and its slices of the error buffer, the mean and theta must be the whole-tensor results'
slices, bit for bit.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

CHUNK = 4096


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _orc_compress(delta, ef, beta, flags=None):
    """The oracle behind the sender call's signature (torch CPU tensors in and out)."""
    import oracle
    bf16 = delta.dtype == torch.bfloat16
    d = delta.view(torch.int16).numpy().view(np.uint16) if bf16 else delta.numpy()
    e = ef.numpy().copy()
    pl, sc, _ = oracle.ef_compress(d, e, beta, bf16=bf16)
    ef.copy_(torch.from_numpy(e))
    return torch.from_numpy(pl), torch.from_numpy(sc)


def _orc_decode(pls, scs, n, mean=None, theta=None, lr=0.0, flags=None, validate=True):
    """The oracle behind the receiver call's signature."""
    import oracle
    th = theta.numpy().copy() if theta is not None else None
    m, _ = oracle.decode_aggregate([p.contiguous().numpy() for p in pls],
                                   [s.contiguous().numpy() for s in scs], n, theta=th, lr=lr)
    if theta is not None:
        theta.copy_(torch.from_numpy(th))
    return torch.from_numpy(m)


def _inputs(n, P, bf16):
    """The whole tensor's inputs, drawn identically on every rank from fixed seeds."""
    from compressed_pseudo_gradient_gb300 import synth
    cpu = torch.device("cpu")
    delta = synth.laplace(n, 1e-4, synth.generator(11, cpu), cpu)
    if bf16:
        delta = delta.to(torch.bfloat16)
    ef = synth.normal(n, 1e-4, synth.generator(12, cpu), cpu)
    peers = []
    for p in range(P):
        d = synth.laplace(n, 1e-4, synth.generator(100 + p, cpu), cpu)
        peers.append(_orc_compress(d, torch.zeros(n), 0.95))
    theta = synth.theta(n, synth.generator(13, cpu), cpu)
    return delta, ef, peers, theta


def _rank_main(rank, world, port, n, P, bf16, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    from compressed_pseudo_gradient_gb300 import sharded
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        delta, ef, peers, theta = _inputs(n, P, bf16)
        C = (n + CHUNK - 1) // CHUNK
        lo, hi = sharded.shard_range(n, world, rank)
        ef_mine = ef[lo:hi].clone()
        pl, sc = sharded.compress_shard(delta[lo:hi], ef_mine, 0.95, compress=_orc_compress)
        full_pl, full_sc = sharded.gather_records(pl, sc, C)
        th_mine = theta[lo:hi].clone()
        mean_mine = sharded.decode_shard([p for p, _ in peers] + [full_pl],
                                         [s for _, s in peers] + [full_sc], n, theta=th_mine,
                                         lr=0.7, decode=_orc_decode)
        # the mean slices gathered back (padded to equal length) for the whole-tensor check
        m = ((C + world - 1) // world) * CHUNK
        pad = torch.zeros(m)
        pad[: hi - lo] = mean_mine
        parts = [torch.empty(m) for _ in range(world)]
        dist.all_gather(parts, pad)
        mean_all = torch.cat([parts[r][: sharded.shard_range(n, world, r)[1] -
                                      sharded.shard_range(n, world, r)[0]] for r in range(world)])
        out.put((rank, lo, hi, full_pl.numpy(), full_sc.numpy(), ef_mine.numpy(),
                 mean_mine.numpy(), th_mine.numpy(), mean_all.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,n,bf16", [(2, 9 * CHUNK + 777, False), (3, 10 * CHUNK, True),
                                          (3, 2 * CHUNK + 5, False), (4, 2 * CHUNK + 5, False)])
def test_sharded_compress_gather_decode_match_whole_tensor(world, n, bf16):
    import oracle
    P = 3
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, n, P, bf16, out))
             for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((out.get(timeout=180) for _ in range(world)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0

    # the whole tensor on one oracle call
    delta, ef, peers, theta = _inputs(n, P, bf16)
    d = delta.view(torch.int16).numpy().view(np.uint16) if bf16 else delta.numpy()
    e = ef.numpy().copy()
    o_pl, o_sc, _ = oracle.ef_compress(d, e, 0.95, bf16=bf16)
    th = theta.numpy().copy()
    o_mean, _ = oracle.decode_aggregate([p.numpy() for p, _ in peers] + [o_pl],
                                        [s.numpy() for _, s in peers] + [o_sc], n, theta=th,
                                        lr=0.7)
    covered = 0
    for rank, lo, hi, pl, sc, ef_mine, mean_mine, th_mine, mean_all in res:
        assert lo == covered and (lo % CHUNK == 0 or lo == n)
        covered = hi
        assert np.array_equal(pl, o_pl), f"rank {rank}: gathered records differ"
        assert np.array_equal(sc.view(np.uint32), o_sc.view(np.uint32))
        assert np.array_equal(ef_mine.view(np.uint32), e[lo:hi].view(np.uint32))
        assert np.array_equal(mean_mine.view(np.uint32), o_mean[lo:hi].view(np.uint32))
        assert np.array_equal(th_mine.view(np.uint32), th[lo:hi].view(np.uint32))
        assert np.array_equal(mean_all.view(np.uint32), o_mean.view(np.uint32))
    assert covered == n


def test_shard_ranges_tile_the_tensor():
    from compressed_pseudo_gradient_gb300 import sharded
    for n in (1, 4095, 4096, 4097, 5 * CHUNK + 1, 1 << 20):
        C = (n + CHUNK - 1) // CHUNK
        for world in (1, 2, 3, 4, 8):
            prev = 0
            for r in range(world):
                c0, c1 = sharded.shard_chunks(C, world, r)
                lo, hi = sharded.shard_range(n, world, r)
                assert lo == prev and lo <= hi               # contiguous, in rank order
                assert lo % CHUNK == 0 or lo == n            # slices start on a chunk
                assert c1 - c0 in (C // world, C // world + 1)
                assert hi - lo == min(n, c1 * CHUNK) - min(n, c0 * CHUNK)
                prev = hi
            assert prev == n
    with pytest.raises(ValueError):
        sharded.shard_chunks(10, 2, 2)


def test_decode_shard_rejects_records_of_another_range():
    from compressed_pseudo_gradient_gb300 import sharded
    pl = torch.zeros((3, 112), dtype=torch.uint8)
    sc = torch.zeros(3)
    with pytest.raises(ValueError):
        sharded.decode_shard([pl], [sc], 10 * CHUNK, decode=_orc_decode)
    with pytest.raises(ValueError):
        sharded.gather_records(pl, sc, 10)
