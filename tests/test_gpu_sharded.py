"""The chunk-sharded path's CUDA calls on one GPU: G slices of one tensor compressed by
separate library calls (as G ranks would, each on its own slice) give the whole-tensor call's
records and error buffer bit for bit, and decoding each slice's chunk range gives the slices of
the whole-tensor mean and theta.  The record exchange itself (an all-gather) is tested on CPU
ranks in test_sharded_gloo.py; here the slices' records are concatenated in rank order, which
is what the all-gather returns."""
import numpy as np
import pytest
import torch

import compressed_pseudo_gradient_gb300 as spl
from compressed_pseudo_gradient_gb300 import sharded, synth
import oracle
from parity_util import assert_bit_equal, host

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.mark.parametrize("G,n,dtype", [(2, 9 * 4096 + 777, torch.float32),
                                       (3, 37 * 4096, torch.bfloat16),
                                       (4, 2 * 4096 + 5, torch.float32),
                                       (8, 1000 * 4096 + 4095, torch.float32)])
def test_slices_compress_and_decode_like_the_whole_tensor(G, n, dtype):
    delta = synth.laplace(n, 1e-4, synth.generator(71, DEV), DEV).to(dtype)
    ef0 = synth.normal(n, 1e-4, synth.generator(72, DEV), DEV)
    C = spl.num_chunks(n)

    ef_whole = ef0.clone()
    pl_whole, sc_whole = spl.ef_compress(delta, ef_whole, 0.95)
    ef_sh = ef0.clone()
    parts = []
    for r in range(G):
        lo, hi = sharded.shard_range(n, G, r)
        parts.append(sharded.compress_shard(delta[lo:hi], ef_sh[lo:hi], 0.95))
    pl_cat = torch.cat([p for p, _ in parts])
    sc_cat = torch.cat([s for _, s in parts])
    torch.cuda.synchronize()
    assert pl_cat.shape == (C, 112)
    assert_bit_equal(host(pl_cat), host(pl_whole), "records of the slices")
    assert_bit_equal(host(sc_cat), host(sc_whole), "scales of the slices")
    assert_bit_equal(host(ef_sh), host(ef_whole), "error buffer of the slices")
    o_pl, o_sc, _ = oracle.ef_compress(host(delta), host(ef0).copy(), 0.95,
                                       bf16=dtype == torch.bfloat16)
    assert_bit_equal(host(pl_cat), o_pl, "records vs oracle")

    peers_pl, peers_sc = [pl_cat], [sc_cat]
    for p in range(3):
        d = synth.laplace(n, 1e-4, synth.generator(80 + p, DEV), DEV)
        a, b = spl.ef_compress(d, torch.zeros(n, device=DEV), 0.95)
        peers_pl.append(a), peers_sc.append(b)
    theta = synth.theta(n, synth.generator(73, DEV), DEV)
    th_whole = theta.clone()
    m_whole = spl.decode_aggregate(peers_pl, peers_sc, n, theta=th_whole, lr=0.7)
    for r in range(G):
        lo, hi = sharded.shard_range(n, G, r)
        c0, c1 = sharded.shard_chunks(C, G, r)
        th = theta[lo:hi].clone()
        # the whole tensor's records, and only this range's rows, give the same slice
        m_full = _decode_range(peers_pl, peers_sc, n, G, r, th)
        th2 = theta[lo:hi].clone()
        m_rows = _decode_range([p[c0:c1] for p in peers_pl], [s[c0:c1] for s in peers_sc], n,
                               G, r, th2)
        torch.cuda.synchronize()
        assert_bit_equal(host(m_full), host(m_whole[lo:hi]), f"mean slice {r}")
        assert_bit_equal(host(m_rows), host(m_whole[lo:hi]), f"mean slice {r} from its rows")
        assert_bit_equal(host(th), host(th_whole[lo:hi]), f"theta slice {r}")
        assert_bit_equal(host(th2), host(th_whole[lo:hi]), f"theta slice {r} from its rows")


def _decode_range(pls, scs, n, G, r, theta):
    """decode_shard as rank r of G would call it (no process group: the rank is passed via a
    stand-in world)."""
    orig = sharded._world
    sharded._world = lambda group=None: (r, G)
    try:
        return sharded.decode_shard(pls, scs, n, theta=theta, lr=0.7)
    finally:
        sharded._world = orig


def test_gather_without_a_group_returns_the_records():
    n = 5 * 4096 + 3
    d = synth.laplace(n, 1e-4, synth.generator(74, DEV), DEV)
    pl, sc = sharded.compress_shard(d, torch.zeros(n, device=DEV), 1.0)
    a, b = sharded.gather_records(pl, sc, spl.num_chunks(n))
    assert a.data_ptr() == pl.data_ptr() and b.data_ptr() == sc.data_ptr()
    np.testing.assert_array_equal(host(a), host(pl))
