"""Multi-rank host logic of bench.py on CPU: two gloo ranks (world size 2).

The codec's multi-GPU mode runs one independent peer per GPU with no collective on the data
path; what needs testing is the host side: rank/seed mapping, the barrier, the max-over-ranks
time and the whole-job aggregate.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world) and dist.is_initialized()
    bench.barrier()
    t = 1.5 if rank == 0 else 2.5          # per-rank "elapsed seconds"
    tmax = bench.max_over_ranks(t)
    value = bench.aggregate_value(1_000_000_000, w, tmax)
    out.put((rank, tmax, value, bench.rank_seed_base(rank)))
    bench.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_share_max_time_and_aggregate():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        assert p.exitcode == 0
    res = sorted(out.get(timeout=10) for _ in range(2))
    for rank, tmax, value, seed in res:
        assert tmax == 2.5                     # the slowest rank's time on every rank
        assert value == pytest.approx(2 * 1e9 / 2.5 / 1e9)
    seeds = [r[3] for r in res]
    import bench
    blocks = [set(range(s, s + 25)) | {s + 5000} | set(bench.round_seeds(s)) for s in seeds]
    assert all(len(b) == 25 + 1 + bench.ROUNDS - 1 for b in blocks)   # no clash inside a block
    assert not (blocks[0] & blocks[1])        # each rank draws its own peer's data


def test_single_process_helpers_without_a_group():
    import bench
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.aggregate_value(2_000_000_000, 1, 2.0) == pytest.approx(1.0)
    assert bench.dist_env() == (0, 1, 0) or "RANK" in os.environ
