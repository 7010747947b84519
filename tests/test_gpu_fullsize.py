"""Every chunk of the full-size workloads against the oracle, in the launch configuration the
benchmark times.

The oracle runs on host copies of exactly the bytes the GPU consumed, split into contiguous
chunk ranges over the host cores (chunks are independent, so the pieces' outputs are the whole
tensor's; the oracle's C calls release the GIL).  Bar: payload bytes, scales and the error
buffer bit-exact for every chunk of every round; the mean and theta within 1e-6 of max |ref|
(and bit-exact, with the fixed peer order).  The sender's rounds are also run through the
checked build of the library on the same inputs, whose outputs must be the same bytes and whose
select-path counters show which paths the workload's data took (printed with -s).
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import compressed_pseudo_gradient_gb300 as spl
import oracle
from compressed_pseudo_gradient_gb300 import synth
from parity_util import assert_bit_equal, assert_close, host

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
CHUNK = 4096
THREADS = os.cpu_count() or 1


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _ranges(C: int):
    parts = min(C, 8 * THREADS)
    bounds = np.linspace(0, C, parts + 1).astype(np.int64)
    return [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]


def oracle_compress(d_h: np.ndarray, e_h: np.ndarray, beta: float, bf16: bool):
    """oracle.ef_compress over chunk ranges on the host cores; e_h is updated in place."""
    n = d_h.size
    C = (n + CHUNK - 1) // CHUNK
    rs = _ranges(C)

    def work(r):
        a, b = r
        lo, hi = a * CHUNK, min(n, b * CHUNK)
        pl, sc, fl = oracle.ef_compress(d_h[lo:hi], e_h[lo:hi], beta, bf16=bf16)
        return pl, sc, fl
    oracle.build()
    with ThreadPoolExecutor(max_workers=THREADS) as ex:
        out = list(ex.map(work, rs))
    return (np.concatenate([o[0] for o in out]), np.concatenate([o[1] for o in out]),
            int(np.bitwise_or.reduce([o[2] for o in out])))


def oracle_decode(pls, scs, n: int, theta_h=None, lr: float = 0.0):
    """oracle.decode_aggregate over chunk ranges on the host cores; theta_h in place."""
    C = (n + CHUNK - 1) // CHUNK
    rs = _ranges(C)

    def work(r):
        a, b = r
        lo, hi = a * CHUNK, min(n, b * CHUNK)
        th = theta_h[lo:hi] if theta_h is not None else None
        m, fl = oracle.decode_aggregate([p[a:b] for p in pls], [s[a:b] for s in scs], hi - lo,
                                        theta=th, lr=lr)
        return m, fl
    oracle.build()
    with ThreadPoolExecutor(max_workers=THREADS) as ex:
        out = list(ex.map(work, rs))
    return np.concatenate([o[0] for o in out]), int(np.bitwise_or.reduce([o[1] for o in out]))


def checked_paths(run):
    """Runs run() through the checked build; returns its debug words (after checking that no
    memory check failed)."""
    torch.cuda.synchronize()
    prev = spl.use_library(spl.checked_library_path())
    try:
        spl.debug_words(reset=True)
        out = run()
        torch.cuda.synchronize()
        d = spl.debug_words(reset=True)
    finally:
        spl.use_library(prev)
    assert d["failures"] == 0, f"checked build: failed memory checks {d}"
    assert d["whole"] + d["rank32"] + d["rank64"] + d["generic"] == d["chunks"], d
    return out, d


def compress_round_every_chunk(deltas, efs, beta, what):
    """One round of the default sender over a table of tensors (one call, as the benchmark
    launches it), every chunk compared with the oracle; the same round through the checked
    build must give the same bytes.  Returns the path counters."""
    bf16 = deltas[0].dtype == torch.bfloat16
    d_h = [host(d) for d in deltas]
    e_h = [host(e) for e in efs]
    efs_chk = [e.clone() for e in efs]
    if len(deltas) == 1:
        payload, scales = spl.ef_compress(deltas[0], efs[0], beta)
    else:
        payload, scales = spl.ef_compress_multi(deltas, efs, beta)
    torch.cuda.synchronize()
    o = [oracle_compress(d, e, beta, bf16) for d, e in zip(d_h, e_h)]
    assert_bit_equal(host(payload), np.concatenate([x[0] for x in o]), f"{what}: payload")
    assert_bit_equal(host(scales), np.concatenate([x[1] for x in o]), f"{what}: scales")
    for i, (e, oe) in enumerate(zip(efs, e_h)):
        assert_bit_equal(host(e), oe, f"{what}: error buffer {i}")
    (pc, sc2), d = checked_paths(lambda: spl.ef_compress_multi(deltas, efs_chk, beta))
    assert torch.equal(pc, payload) and torch.equal(sc2.view(torch.int32), scales.view(torch.int32))
    for e, e2 in zip(efs, efs_chk):
        assert torch.equal(e.view(torch.int32), e2.view(torch.int32))
    print(f"\n{what}: {d['chunks']} chunks: whole bin {d['whole']}, ranked <= 32 {d['rank32']}, "
          f"ranked 33-64 {d['rank64']}, search past the top 512 bins {d['full_scan']}, "
          f"generic select {d['generic']}")
    return d


def test_large_flat_every_chunk():
    """2^30 fp32 Laplace(0, 1e-4), beta 0.95, three rounds of fresh pseudo-gradients."""
    wl = synth.WORKLOADS["large_flat"]
    gen = synth.generator(0, DEV)
    ef = torch.zeros(wl.n, device=DEV)
    for r in range(3):
        delta = synth.delta_round(wl, gen, DEV)
        compress_round_every_chunk([delta], [ef], wl.beta, f"large flat round {r}")
        del delta


def test_heavy_tail_bf16_every_chunk():
    """2^27 bf16 heavy-tailed, beta 0.95, all five rounds, then the 8-peer mean (also through
    the checked build)."""
    wl = synth.WORKLOADS["heavy_tail_bf16"]
    gen = synth.generator(0, DEV)
    ef = torch.zeros(wl.n, device=DEV)
    for r in range(wl.rounds):
        delta = synth.delta_round(wl, gen, DEV)
        compress_round_every_chunk([delta], [ef], wl.beta, f"heavy tail round {r}")
    pls, scs = [], []
    for p in range(wl.peers):
        d = synth.delta_round(wl, synth.generator(1 + p, DEV), DEV)
        a, b = spl.ef_compress(d, torch.zeros(wl.n, device=DEV), wl.beta)
        pls.append(a), scs.append(b)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    mean = spl.decode_aggregate(pls, scs, wl.n, flags=flags)
    torch.cuda.synchronize()
    mean_chk, _ = checked_paths(lambda: spl.decode_aggregate(pls, scs, wl.n))
    assert torch.equal(mean_chk.view(torch.int32), mean.view(torch.int32))
    o_mean, o_flags = oracle_decode([host(p) for p in pls], [host(s) for s in scs], wl.n)
    assert int(flags.item()) == o_flags == 0
    assert_close(host(mean), o_mean, "heavy tail mean of 8")
    assert_bit_equal(host(mean), o_mean, "heavy tail mean of 8 (fixed peer order)")


def test_decoder_layer_every_chunk():
    """The nine tensors of a 72B-class decoder layer, one multi-tensor call per round, three
    rounds."""
    wl = synth.WORKLOADS["decoder_layer"]
    gen = synth.generator(0, DEV)
    deltas = synth.decoder_layer_round(gen, DEV)
    efs = [torch.zeros_like(d) for d in deltas]
    for r in range(wl.rounds if wl.rounds else 3):
        compress_round_every_chunk(deltas, efs, wl.beta, f"decoder layer round {r}")
        deltas = synth.decoder_layer_round(gen, DEV)


def test_receive_24_peers_every_value():
    """24 peers' records of 2^30 values into the mean, fused with the outer step; the same
    decode through the checked build gives the same bytes with no failed memory check."""
    wl = synth.WORKLOADS["receive"]
    n = wl.n
    pls, scs = [], []
    e = torch.empty(n, device=DEV)
    for p in range(wl.peers):
        d = synth.delta_round(wl, synth.generator(1 + p, DEV), DEV)
        e.zero_()
        a, b = spl.ef_compress(d, e, wl.beta)
        pls.append(a), scs.append(b)
        del d
    del e
    theta = synth.theta(n, synth.generator(0, DEV), DEV)
    th_h = host(theta)
    theta_chk = theta.clone()
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    mean = spl.decode_aggregate(pls, scs, n, theta=theta, lr=wl.lr, flags=flags)
    torch.cuda.synchronize()
    mean_chk, d = checked_paths(lambda: spl.decode_aggregate(pls, scs, n, theta=theta_chk,
                                                             lr=wl.lr))
    assert torch.equal(mean_chk.view(torch.int32), mean.view(torch.int32))
    assert torch.equal(theta_chk.view(torch.int32), theta.view(torch.int32))
    del mean_chk, theta_chk
    o_mean, o_flags = oracle_decode([host(p) for p in pls], [host(s) for s in scs], n,
                                    theta_h=th_h, lr=wl.lr)
    assert int(flags.item()) == o_flags == 0
    assert_close(host(mean), o_mean, "mean of 24")
    assert_close(host(theta), th_h, "theta")
    assert_bit_equal(host(mean), o_mean, "mean of 24 (fixed peer order)")
    assert_bit_equal(host(theta), th_h, "theta (one fma)")


def test_several_waves_with_a_ragged_tail():
    """A tensor of 40,000 chunks whose last chunk is partial: the sender and both receiver
    shapes take several waves of CTAs (16 or 32 chunks per CTA, the last wave partial), and
    every chunk, the tail included, matches the oracle; also through the checked build."""
    n = 40000 * CHUNK - 1234
    P = 3
    gen = synth.generator(77, DEV)
    pls, scs = [], []
    for p in range(P):
        d = synth.laplace(n, 1e-4, synth.generator(80 + p, DEV), DEV)
        e = synth.normal(n, 1e-4, synth.generator(90 + p, DEV), DEV)
        compress_round_every_chunk([d], [e], 0.95, f"ragged waves, peer {p}")
        a, b = spl.ef_compress(d, e, 0.95)     # a second round, kept for the decode
        pls.append(a), scs.append(b)
        del d, e
    pls_h, scs_h = [host(p) for p in pls], [host(s) for s in scs]
    theta = synth.theta(n, gen, DEV)
    th_h = host(theta)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    mean = spl.decode_aggregate(pls, scs, n, theta=theta, lr=0.7, flags=flags)   # wide shape
    lean = spl.decode_aggregate(pls, scs, n, flags=flags)                         # lean shape
    torch.cuda.synchronize()
    (lean_chk, _) = checked_paths(lambda: spl.decode_aggregate(pls, scs, n))
    assert torch.equal(lean_chk.view(torch.int32), lean.view(torch.int32))
    o_mean, o_flags = oracle_decode(pls_h, scs_h, n, theta_h=th_h, lr=0.7)
    assert int(flags.item()) == o_flags == 0
    assert_bit_equal(host(mean), o_mean, "ragged waves: mean with theta")
    assert_bit_equal(host(theta), th_h, "ragged waves: theta")
    assert_bit_equal(host(lean), o_mean, "ragged waves: mean, lean shape")
