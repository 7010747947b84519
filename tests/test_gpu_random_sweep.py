"""A seeded randomized sweep over the library's parameters against the oracle (GPU): codec
(the default and every variant), tensor size (1 value to a few chunks, ragged), delta type,
beta (including negative and zero), peer count, the outer step on or off, statistics on or
off, and malformed records.  Every output is compared bit for bit (statistics' sum of squares
within 1e-6 relative).  SPL_SWEEP_CASES sets the number of cases (80 by default)."""
import os

import numpy as np
import pytest
import torch

import compressed_pseudo_gradient_gb300 as spl
import oracle
from compressed_pseudo_gradient_gb300 import synth
from parity_util import assert_bit_equal, host

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
CODECS = [None, (4096, 64, 1), (4096, 32, 0), (4096, 32, 1), (4096, 128, 0), (4096, 128, 1),
          (2048, 32, 0), (2048, 32, 1), (8192, 128, 0), (8192, 128, 1)]


@pytest.mark.parametrize("case", range(int(os.environ.get("SPL_SWEEP_CASES", "80"))))
def test_random_case_matches_oracle(case):
    rng = np.random.default_rng(1000 + case)
    codec = CODECS[case % len(CODECS)]
    L = 4096 if codec is None else codec[0]
    n = int(rng.integers(1, 4 * L + 2))
    bf16 = bool(rng.integers(0, 2))
    beta = float(rng.choice([1.0, 0.95, 0.5, 0.0, -0.3]))
    P = int(rng.integers(1, 31))
    with_theta = bool(rng.integers(0, 2))
    with_stats = bool(rng.integers(0, 2))
    scale = float(10.0 ** rng.uniform(-6, 2))

    gen = synth.generator(5000 + case, DEV)
    delta = (synth.laplace(n, scale, gen, DEV) if not bf16
             else synth.laplace(n, scale, gen, DEV).to(torch.bfloat16))
    ef = synth.laplace(n, scale / 4, gen, DEV)
    d_h, e_h = host(delta), host(ef).copy()
    payload, scales = spl.ef_compress(delta, ef, beta, codec=codec)
    torch.cuda.synchronize()
    o_pl, o_sc, _ = oracle.ef_compress(d_h, e_h, beta, bf16=bf16, codec=codec)
    what = f"case {case}: codec {codec}, n {n}, bf16 {bf16}, beta {beta}"
    assert_bit_equal(host(payload), o_pl, f"{what}: payload")
    assert_bit_equal(host(scales), o_sc, f"{what}: scales")
    assert_bit_equal(host(ef), e_h, f"{what}: error buffer")

    # P peers: this round's records and P - 1 others from fresh deltas; one may be malformed
    pls, scs = [o_pl], [o_sc]
    for p in range(P - 1):
        d = synth.laplace(n, scale, gen, DEV)
        pl, sc, _ = oracle.ef_compress(host(d), np.zeros(n, np.float32), 1.0, codec=codec)
        pls.append(pl)
        scs.append(sc)
    if P > 2 and rng.integers(0, 2):
        idx, codes = oracle.unpack(pls[1], codec)
        k = idx.shape[1]
        idx[0, [k - 2, k - 1]] = idx[0, [k - 1, k - 2]]
        pls[1] = oracle.pack(idx, codes, codec)
    theta = synth.theta(n, gen, DEV) if with_theta else None
    th_h = host(theta).copy() if with_theta else None
    stats = spl.new_peer_stats(P, DEV) if with_stats else None
    mean = spl.decode_aggregate([torch.from_numpy(p).to(DEV) for p in pls],
                                [torch.from_numpy(s).to(DEV) for s in scs], n, theta=theta,
                                lr=0.7, stats=stats, codec=codec)
    torch.cuda.synchronize()
    o_mean, _ = oracle.decode_aggregate(pls, scs, n, theta=th_h, lr=0.7, codec=codec)
    assert_bit_equal(host(mean), o_mean, f"{what}, P {P}: mean")
    if with_theta:
        assert_bit_equal(host(theta), th_h, f"{what}, P {P}: theta")
    if with_stats:
        got = spl.read_peer_stats(stats)
        ref = oracle.peer_stats(pls, scs, n, codec=codec)
        for key in ("rejected", "big", "negative"):
            assert np.array_equal(got[key], ref[key]), (what, key)
        assert_bit_equal(got["max_scale"], ref["max_scale"], f"{what}: max_scale")
        assert np.allclose(got["sumsq"], ref["sumsq"], rtol=1e-6, atol=0)
