"""GPU parity: the CUDA library against the CPU oracle on the same seeded inputs.

Bar: payload bytes, indices, codes, scales and the error buffer bit-exact; the mean and theta
within 1e-6 of max |reference| (and, with the fixed peer summation order, bit-exact where
checked).  Small and medium cases compare every chunk here; the full workload sizes are in
test_gpu_fullsize.py (every chunk as well).
"""
import numpy as np
import pytest
import torch

import compressed_pseudo_gradient_gb300 as spl
import oracle
from compressed_pseudo_gradient_gb300 import synth
from parity_util import assert_bit_equal, assert_close, host

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def gpu_round(delta, ef, beta, flags=None):
    return spl.ef_compress(delta, ef, beta, flags=flags)


def compare_full_round(delta, ef, beta, what):
    d_h, e_h = host(delta), host(ef)
    payload, scales = gpu_round(delta, ef, beta)
    torch.cuda.synchronize()
    o_pl, o_sc, _ = oracle.ef_compress(d_h, e_h, beta, bf16=delta.dtype == torch.bfloat16)
    assert_bit_equal(host(payload), o_pl, f"{what}: payload")
    assert_bit_equal(host(scales), o_sc, f"{what}: scales")
    assert_bit_equal(host(ef), e_h, f"{what}: error buffer")
    return payload, scales, o_pl, o_sc


# ---------------------------------------------------------------------------------------------
# Tiny workload, every chunk: 2^20 fp32 N(0, 1e-3), beta 1, 3 rounds; mean of 4 peers
# ---------------------------------------------------------------------------------------------
def test_tiny_workload_all_chunks():
    wl = synth.WORKLOADS["tiny"]
    gen = synth.generator(0, DEV)
    ef = torch.zeros(wl.n, device=DEV)
    for r in range(wl.rounds):
        delta = synth.delta_round(wl, gen, DEV)
        compare_full_round(delta, ef, wl.beta, f"round {r}")
    payloads, scales, o_pl, o_sc = [], [], [], []
    for p in range(wl.peers):
        g = synth.generator(1 + p, DEV)
        d = synth.delta_round(wl, g, DEV)
        e = torch.zeros(wl.n, device=DEV)
        pl, sc, opl, osc = compare_full_round(d, e, wl.beta, f"peer {p}")
        payloads.append(pl), scales.append(sc), o_pl.append(opl), o_sc.append(osc)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    mean = spl.decode_aggregate(payloads, scales, wl.n, flags=flags)
    torch.cuda.synchronize()
    o_mean, o_flags = oracle.decode_aggregate(o_pl, o_sc, wl.n)
    assert int(flags.item()) == o_flags == 0
    assert_close(host(mean), o_mean, "mean")
    assert_bit_equal(host(mean), o_mean, "mean (fixed peer order)")
    theta = synth.theta(wl.n, synth.generator(0, DEV), DEV)
    th_h = host(theta)
    spl.decode_aggregate(payloads, scales, wl.n, theta=theta, lr=0.7)
    torch.cuda.synchronize()
    oracle.decode_aggregate(o_pl, o_sc, wl.n, theta=th_h, lr=0.7)
    assert_close(host(theta), th_h, "theta")
    assert_bit_equal(host(theta), th_h, "theta (one fma)")


# ---------------------------------------------------------------------------------------------
# Sizes and edge cases
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("n", [1, 63, 64, 65, 4095, 4096, 4097, 8191, 3 * 4096 + 1, 40 * 4096 + 123])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_edge_sizes(n, dtype):
    gen = synth.generator(n, DEV)
    delta = synth.laplace(n, 1e-4, gen, DEV).to(dtype)
    ef = synth.normal(n, 1e-4, gen, DEV)
    pl, sc, o_pl, o_sc = compare_full_round(delta, ef, 0.95, f"n={n}")
    pl2, sc2, o_pl2, o_sc2 = compare_full_round(delta, ef, 0.95, f"n={n} round 2")
    theta = synth.theta(n, gen, DEV)
    th_h = host(theta)
    mean = spl.decode_aggregate([pl, pl2, pl], [sc, sc2, sc], n, theta=theta, lr=0.7)
    torch.cuda.synchronize()
    o_mean, _ = oracle.decode_aggregate([o_pl, o_pl2, o_pl], [o_sc, o_sc2, o_sc], n, theta=th_h, lr=0.7)
    assert_bit_equal(host(mean), o_mean, f"n={n}: mean")
    assert_bit_equal(host(theta), th_h, f"n={n}: theta")


def _chunks(*blocks):
    return torch.cat([torch.as_tensor(b, dtype=torch.float32).reshape(-1) for b in blocks]).to(DEV)


def test_degenerate_chunks():
    rng = np.random.default_rng(0)
    L = 4096
    spikes = np.zeros(L, np.float32)
    spikes[rng.choice(L, 64, replace=False)] = rng.choice([-1, 1], 64) * (1 + rng.random(64))
    few = np.zeros(L, np.float32)
    few[[5, 900, 4000]] = [0.5, -2.0, 1.0]
    ties = np.round(rng.standard_normal(L) * 2).astype(np.float32)          # many equal |a|
    coarse = (rng.integers(-3, 4, L) * 0.25).astype(np.float32)
    sub = (rng.standard_normal(L) * 1e-39).astype(np.float32)               # subnormal values
    tiny = np.full(L, np.float32(1.4e-45))                                  # smallest subnormal
    big = rng.standard_normal(L).astype(np.float32)
    big[77] = 3e38
    delta = _chunks(np.zeros(L), np.full(L, -0.0), np.full(L, -2.5), np.arange(L) * -1.0,
                    np.arange(L)[::-1].copy(), spikes, few, ties, coarse, sub, tiny, big)
    ef = torch.zeros_like(delta)
    compare_full_round(delta, ef, 1.0, "degenerate round 1")
    compare_full_round(torch.zeros_like(delta), ef, 1.0, "degenerate round 2 (zero delta)")
    compare_full_round(delta, ef, -0.5, "degenerate round 3 (negative beta)")


def test_select_window_edges():
    """Chunks built around the compress kernel's fast path: its histogram spans the 16 octaves
    below the chunk max and ranks a boundary bin of at most 64 keys directly (one per lane up to
    32, two per lane beyond); everything else takes the generic radix select.  Both must agree
    with the oracle."""
    rng = np.random.default_rng(17)
    L = 4096
    base = (rng.random(L).astype(np.float32) * 0.5 + 0.25)               # ~[0.25, 0.75)

    def chunk(f):
        c = base.copy() * rng.choice([-1.0, 1.0], L).astype(np.float32)
        f(c)
        return c

    def spikes_far_above(c):       # 63 values 2^40 above: 64th key 40 octaves below the max
        c[rng.choice(L, 63, replace=False)] = 2.0 ** 40
    def spikes_just_inside(c):     # 63 values 2^14 above: the 64th key inside the window
        c[rng.choice(L, 63, replace=False)] = 2.0 ** 14
    def ties(count):
        def f(c):                  # `count` keys equal at the threshold, 40 above it
            pos = rng.choice(L, 40 + count, replace=False)
            c[pos[:40]] = 2.0
            c[pos[40:]] = -1.0     # the rest of the chunk stays below 0.75
        return f
    def dense(count):
        def f(c):                  # `count` distinct keys inside one bin, 40 above them
            pos = rng.choice(L, 40 + count, replace=False)
            c[pos[:40]] = 2.0
            # 1 + (i + 1) 2^-20: keys 0x3F800008 + 8 i, inside one bin of the window whose
            # top bin starts at the key of 2.0 (bin edges at keys ending in 0x0001)
            vals = (1.0 + (1 + np.arange(count)) * 2.0 ** -20).astype(np.float32)
            c[pos[40:]] = rng.permutation(vals) * rng.choice([-1.0, 1.0], count)
        return f
    def one_per_bin(c):            # distinct powers of two: each key alone in its bin
        c[:] = 0.0
        c[rng.choice(L, 80, replace=False)] = 2.0 ** -np.arange(80, dtype=np.float32) * 8
    def exact_bin(c):              # exactly 64 keys at or above one value
        c[rng.choice(L, 64, replace=False)] = 3.0
    blocks = [chunk(spikes_far_above), chunk(spikes_just_inside), chunk(ties(20)),
              chunk(ties(24)), chunk(ties(25)), chunk(ties(33)), chunk(ties(48)),
              chunk(ties(64)), chunk(ties(65)), chunk(ties(200)), chunk(dense(25)),
              chunk(dense(32)), chunk(dense(33)), chunk(dense(47)), chunk(dense(63)),
              chunk(dense(64)), chunk(dense(65)), chunk(one_per_bin), chunk(exact_bin)]
    delta = _chunks(*blocks)
    ef = torch.zeros_like(delta)
    compare_full_round(delta, ef, 1.0, "window edges round 1")
    compare_full_round(delta, ef, 0.5, "window edges round 2")


def test_bf16_ties_stress():
    """bf16 values have 8 significant bits: many exact ties at the threshold."""
    gen = synth.generator(5, DEV)
    n = 64 * 4096
    x = (synth.normal(n, 1.0, gen, DEV) * 4).round() / 4
    delta = x.to(torch.bfloat16)
    ef = torch.zeros(n, device=DEV)
    compare_full_round(delta, ef, 1.0, "bf16 ties")
    compare_full_round(delta, ef, 1.0, "bf16 ties round 2")


def test_exact_ties_in_the_boundary_bin_and_sparse_chunks():
    """Chunks whose boundary bin holds up to 64 keys that are all equal (chosen by index
    alone), the same next to a bin of different keys, and chunks with fewer than 64 nonzero
    magnitudes (every nonzero plus the lowest-index zeros), in fp32 and bf16, over rounds that
    turn selected zeros into tied residuals."""
    rng = np.random.default_rng(11)
    L = 4096

    def tied(n_top, n_tie, top=2.0, tie=1.0):
        x = np.zeros(L, np.float32)
        pos = rng.choice(L, n_top + n_tie, replace=False)
        x[pos[:n_top]] = top * rng.choice([-1, 1], n_top)
        x[pos[n_top:]] = tie * rng.choice([-1, 1], n_tie)
        return x

    mixed = tied(40, 30)
    mixed[rng.choice(np.flatnonzero(mixed == 0), 3, replace=False)] = 1.0 + 2.0 ** -20
    sparse = np.zeros(L, np.float32)
    sparse[rng.choice(L, 10, replace=False)] = rng.standard_normal(10).astype(np.float32)
    one = np.zeros(L, np.float32)
    one[4095] = -3.0
    chunks = (tied(40, 40), tied(0, 64 + 1), tied(63, 2), tied(10, 60), mixed, sparse, one,
              tied(60, 4, 1.0, 1.0))
    for dtype in (torch.float32, torch.bfloat16):
        delta = _chunks(*chunks).to(dtype)
        ef = torch.zeros(delta.numel(), device=DEV)
        compare_full_round(delta, ef, 1.0, f"{dtype} ties round 1")
        compare_full_round(delta, ef, 0.95, f"{dtype} ties round 2")
        compare_full_round(torch.zeros_like(delta), ef, 0.95, f"{dtype} ties round 3 (zero delta)")


def test_nonfinite_inputs_flagged_and_deterministic():
    n = 4 * 4096
    gen = synth.generator(9, DEV)
    delta = synth.laplace(n, 1e-4, gen, DEV)
    delta[100] = float("inf")
    delta[5000] = float("nan")
    delta[9000] = -float("inf")
    delta[9001] = float("nan")
    ef = torch.zeros(n, device=DEV)
    d_h, e_h = host(delta), host(ef)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    payload, scales = spl.ef_compress(delta, ef, 1.0, flags=flags)
    torch.cuda.synchronize()
    o_pl, o_sc, o_flags = oracle.ef_compress(d_h, e_h, 1.0)
    assert int(flags.item()) & spl.FLAG_NONFINITE and o_flags & oracle.FLAG_NONFINITE
    assert_bit_equal(host(payload), o_pl, "payload with non-finite values")
    g_sc = host(scales)
    assert np.array_equal(np.isnan(g_sc), np.isnan(o_sc))
    fin = np.isfinite(o_sc)
    assert_bit_equal(g_sc[fin], o_sc[fin], "finite scales")
    g_e = host(ef)
    same = (g_e == e_h) | (np.isnan(g_e) & np.isnan(e_h))
    assert same.all()
    assert int(flags.item()) & spl.FLAG_BAD_RECORD == 0


# ---------------------------------------------------------------------------------------------
# Heavy-tailed bf16 workload
# ---------------------------------------------------------------------------------------------
def test_heavy_tail_bf16_medium_all_chunks():
    wl = synth.WORKLOADS["heavy_tail_bf16"]
    n = 1 << 22
    gen = synth.generator(0, DEV)
    ef = torch.zeros(n, device=DEV)
    for r in range(wl.rounds):
        delta = synth.delta_round(wl, gen, DEV, n=n)
        compare_full_round(delta, ef, wl.beta, f"heavy tail medium round {r}")


# ---------------------------------------------------------------------------------------------
# 72B-class decoder layer, chunked per tensor (multi-tensor launch)
# ---------------------------------------------------------------------------------------------
SMALL_LAYER = tuple((name, (max(1, s[0] // 64),) + tuple(s[1:])) for name, s in synth.DECODER_LAYER_SHAPES)


def test_decoder_layer_multi_tensor_small_all_chunks():
    shapes = SMALL_LAYER + (("odd", (3, 1000)), ("empty", (0,)), ("one", (1,)))
    gen = synth.generator(3, DEV)
    deltas = [synth.row_scaled_normal(s, 2e-4, gen, DEV) if np.prod(s) else
              torch.zeros(0, device=DEV) for _, s in shapes]
    efs = [torch.zeros_like(d) for d in deltas]
    for r in range(3):
        d_h = [host(d) for d in deltas]
        e_h = [host(e) for e in efs]
        payload, scales = spl.ef_compress_multi(deltas, efs, 1.0)
        torch.cuda.synchronize()
        o_pl, o_sc = [], []
        for d, e in zip(d_h, e_h):
            if d.size:
                p, s, _ = oracle.ef_compress(d, e, 1.0)
                o_pl.append(p), o_sc.append(s)
        assert_bit_equal(host(payload), np.concatenate(o_pl), f"layer round {r}: payload")
        assert_bit_equal(host(scales), np.concatenate(o_sc), f"layer round {r}: scales")
        for i, (e, oe) in enumerate(zip(efs, e_h)):
            assert_bit_equal(host(e), oe, f"layer round {r}: error buffer {i}")
        deltas = [synth.row_scaled_normal(s, 2e-4, gen, DEV) if np.prod(s) else
                  torch.zeros(0, device=DEV) for _, s in shapes]


def test_multi_tensor_matches_single_calls_and_splits_long_tables():
    gen = synth.generator(4, DEV)
    sizes = [int(x) for x in np.random.default_rng(4).integers(1, 3 * 4096, size=150)]
    deltas = [synth.laplace(k, 1e-4, gen, DEV) for k in sizes]        # 150 tensors: 3 launches
    efs = [synth.normal(k, 1e-4, gen, DEV) for k in sizes]
    efs2 = [e.clone() for e in efs]
    payload, scales = spl.ef_compress_multi(deltas, efs, 0.9)
    singles = [spl.ef_compress(d, e, 0.9) for d, e in zip(deltas, efs2)]
    torch.cuda.synchronize()
    assert_bit_equal(host(payload), np.concatenate([host(p) for p, _ in singles]), "payload")
    assert_bit_equal(host(scales), np.concatenate([host(s) for _, s in singles]), "scales")
    for e, e2 in zip(efs, efs2):
        assert_bit_equal(host(e), host(e2), "error buffer")


# ---------------------------------------------------------------------------------------------
# Record layout helpers and malformed records
# ---------------------------------------------------------------------------------------------
def test_pack_unpack_match_oracle():
    rng = np.random.default_rng(21)
    C = 1000
    idx = np.sort(np.stack([rng.choice(4096, 64, replace=False) for _ in range(C)]), 1)
    idx = idx.astype(np.uint16)
    codes = rng.integers(0, 4, (C, 64)).astype(np.uint8)
    o_pl = oracle.pack(idx, codes)
    g_pl = spl.pack(torch.from_numpy(idx.view(np.int16)).to(DEV), torch.from_numpy(codes).to(DEV))
    g_idx, g_codes = spl.unpack(torch.from_numpy(o_pl).to(DEV))
    torch.cuda.synchronize()
    assert_bit_equal(host(g_pl), o_pl, "pack")
    assert np.array_equal(host(g_idx).view(np.uint16), idx)
    assert np.array_equal(host(g_codes), codes)


@pytest.mark.parametrize("with_theta", [False, True])
def test_malformed_records_rejected_like_oracle(with_theta):
    n = 6 * 4096
    gen = synth.generator(31, DEV)
    pls, scs = [], []
    for _ in range(3):
        d = synth.laplace(n, 1e-4, gen, DEV)
        pl, sc = gpu_round(d, torch.zeros(n, device=DEV), 1.0)
        pls.append(host(pl)), scs.append(host(sc))
    idx, codes = oracle.unpack(pls[1])
    idx[0, [3, 4]] = idx[0, [4, 3]]           # chunk 0: not ascending
    idx[2, 40] = idx[2, 39]                   # chunk 2: duplicate
    idx[5, 63] = idx[5, 0]                    # chunk 5: wraps
    idx[3, 33] = idx[3, 1]                    # chunk 3: entries one adding lane holds both
    pls[1] = oracle.pack(idx, codes)
    scs[2][1] = np.nan                        # chunk 1 of peer 2
    scs[2][3] = np.inf
    scs[2][4] = -1.0
    scs[0][5] = -0.0                          # -0.0 is a valid (zero) scale
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    theta = synth.theta(n, synth.generator(32, DEV), DEV) if with_theta else None
    th_h = host(theta) if with_theta else None
    mean = spl.decode_aggregate([torch.from_numpy(p).to(DEV) for p in pls],
                                [torch.from_numpy(s).to(DEV) for s in scs], n, flags=flags,
                                theta=theta, lr=0.7)
    torch.cuda.synchronize()
    o_mean, o_flags = oracle.decode_aggregate(pls, scs, n, theta=th_h, lr=0.7)
    assert int(flags.item()) == o_flags == oracle.FLAG_BAD_RECORD
    assert_bit_equal(host(mean), o_mean, "mean with rejected records")
    if with_theta:
        assert_bit_equal(host(theta), th_h, "theta with rejected records")


@pytest.mark.parametrize("P", [1, 5, 8, 24])
def test_decode_without_validation_matches_oracle(P):
    """validate = 0 skips the record checks: on well-formed records the mean and theta are
    the validated call's, bit for bit (and the oracle's)."""
    n = 37 * 4096 + 1001
    pls, scs = [], []
    for p in range(P):
        d = synth.laplace(n, 1e-4, synth.generator(400 + p, DEV), DEV)
        pl, sc = gpu_round(d, synth.normal(n, 1e-4, synth.generator(500 + p, DEV), DEV), 0.95)
        pls.append(pl), scs.append(sc)
    theta = synth.theta(n, synth.generator(600, DEV), DEV)
    th_h = host(theta)
    theta2 = theta.clone()
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    m_on = spl.decode_aggregate(pls, scs, n, theta=theta, lr=0.7, flags=flags)
    m_off = spl.decode_aggregate(pls, scs, n, theta=theta2, lr=0.7, flags=flags, validate=False)
    m_plain = spl.decode_aggregate(pls, scs, n, flags=flags, validate=False)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    o_mean, o_flags = oracle.decode_aggregate([host(p) for p in pls], [host(s) for s in scs], n,
                                              theta=th_h, lr=0.7)
    assert o_flags == 0
    assert_bit_equal(host(m_off), host(m_on), "mean, validation off vs on")
    assert_bit_equal(host(m_plain), host(m_on), "mean without theta, validation off")
    assert_bit_equal(host(theta2), host(theta), "theta, validation off vs on")
    assert_bit_equal(host(m_off), o_mean, "mean, validation off vs oracle")
    assert_bit_equal(host(theta2), th_h, "theta, validation off vs oracle")


# ---------------------------------------------------------------------------------------------
# Checkpoint/resume of the only codec state, and streams
# ---------------------------------------------------------------------------------------------
def test_resume_from_host_copy_of_error_buffer():
    n = 50 * 4096 + 17
    gen = synth.generator(41, DEV)
    deltas = [synth.laplace(n, 1e-4, gen, DEV) for _ in range(3)]
    ef_a = torch.zeros(n, device=DEV)
    outs_a = [gpu_round(d, ef_a, 0.95) for d in deltas]
    ef_b = torch.zeros(n, device=DEV)
    for d in deltas[:2]:
        gpu_round(d, ef_b, 0.95)
    saved = ef_b.cpu()
    del ef_b
    ef_c = saved.to(DEV)
    pl, sc = gpu_round(deltas[2], ef_c, 0.95)
    torch.cuda.synchronize()
    assert_bit_equal(host(pl), host(outs_a[2][0]), "resumed payload")
    assert_bit_equal(host(sc), host(outs_a[2][1]), "resumed scales")
    assert_bit_equal(host(ef_c), host(ef_a), "resumed error buffer")


def test_side_stream_and_stream_order():
    n = 20 * 4096
    gen = synth.generator(51, DEV)
    delta = synth.laplace(n, 1e-4, gen, DEV)
    ef1 = torch.zeros(n, device=DEV)
    ef2 = torch.zeros(n, device=DEV)
    ref = gpu_round(delta, ef1, 0.95)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = gpu_round(delta, ef2, 0.95)
        mean = spl.decode_aggregate([out[0]], [out[1]], n)
    s.synchronize()
    torch.cuda.synchronize()
    assert_bit_equal(host(out[0]), host(ref[0]), "side-stream payload")
    assert_bit_equal(host(ef2), host(ef1), "side-stream error buffer")
    assert np.count_nonzero(host(mean)) == 64 * 20


# ---------------------------------------------------------------------------------------------
# Error buffer resident in pinned host memory (read and written over the host link)
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_error_buffer_in_pinned_host_memory(dtype):
    n = 37 * 4096 + 101
    gen = synth.generator(61, DEV)
    ef_dev = synth.normal(n, 1e-4, gen, DEV)
    ef_host = ef_dev.cpu().pin_memory()
    for r in range(3):
        delta = synth.laplace(n, 1e-4, gen, DEV).to(dtype)
        d_h, e_h = host(delta), host(ef_dev)
        pl_d, sc_d = spl.ef_compress(delta, ef_dev, 0.95)
        pl_h, sc_h = spl.ef_compress(delta, ef_host, 0.95)
        torch.cuda.synchronize()
        assert_bit_equal(host(pl_h), host(pl_d), f"round {r}: payload (host vs device buffer)")
        assert_bit_equal(host(sc_h), host(sc_d), f"round {r}: scales")
        assert_bit_equal(ef_host.numpy(), host(ef_dev), f"round {r}: error buffer")
        o_pl, o_sc, _ = oracle.ef_compress(d_h, e_h, 0.95, bf16=dtype == torch.bfloat16)
        assert_bit_equal(host(pl_h), o_pl, f"round {r}: payload vs oracle")
        assert_bit_equal(ef_host.numpy(), e_h, f"round {r}: error buffer vs oracle")


def test_multi_tensor_host_error_buffers():
    gen = synth.generator(62, DEV)
    sizes = [5000, 4096, 1, 9 * 4096 + 7]
    deltas = [synth.laplace(k, 1e-4, gen, DEV) for k in sizes]
    efs_dev = [synth.normal(k, 1e-4, gen, DEV) for k in sizes]
    efs_host = [e.cpu().pin_memory() for e in efs_dev]
    pl_d, sc_d = spl.ef_compress_multi(deltas, efs_dev, 1.0)
    pl_h, sc_h = spl.ef_compress_multi(deltas, efs_host, 1.0)
    torch.cuda.synchronize()
    assert_bit_equal(host(pl_h), host(pl_d), "payload")
    assert_bit_equal(host(sc_h), host(sc_d), "scales")
    for a, b in zip(efs_host, efs_dev):
        assert_bit_equal(a.numpy(), host(b), "error buffer")
    with pytest.raises(spl.SplError):            # one kind of memory per table
        spl.ef_compress_multi(deltas[:2], [efs_dev[0], efs_host[1]], 1.0)


def test_memory_kinds_that_bulk_copies_cannot_read_are_rejected():
    import ctypes
    lib = spl.library()
    n = 8192
    delta = torch.zeros(n, device=DEV)
    ef = torch.zeros(n, device=DEV)
    payload = torch.empty((2, 112), dtype=torch.uint8, device=DEV)
    scales = torch.empty(2, device=DEV)
    pageable = np.zeros(n + 8, np.float32)
    pp = pageable.ctypes.data + (-pageable.ctypes.data) % 16
    st = torch.cuda.current_stream().cuda_stream
    assert lib.spl_ef_compress(delta.data_ptr(), 0, pp, n, 1.0, payload.data_ptr(),
                               scales.data_ptr(), None, st) == 1      # pageable error buffer
    pinned = torch.zeros(n).pin_memory()
    assert lib.spl_ef_compress(pinned.data_ptr(), 0, ef.data_ptr(), n, 1.0, payload.data_ptr(),
                               scales.data_ptr(), None, st) == 1      # delta in host memory
    mean = torch.empty(n, device=DEV)
    parr = (ctypes.c_void_p * 1)(payload.data_ptr())
    sarr = (ctypes.c_void_p * 1)(scales.data_ptr())
    assert lib.spl_decode_aggregate(parr, sarr, 1, n, mean.data_ptr(), pinned.data_ptr(), 0.7,
                                    1, None, st) == 1                 # theta in host memory
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------------------------
# Per-peer statistics fused into the receive pass
# ---------------------------------------------------------------------------------------------
def test_peer_stats_match_oracle():
    n = 1024 * 4096 + 333
    P = 24
    gen = synth.generator(81, DEV)
    pls, scs = [], []
    for p in range(P):
        d = synth.laplace(n, 1e-4, synth.generator(100 + p, DEV), DEV)
        pl, sc = gpu_round(d, torch.zeros(n, device=DEV), 0.95)
        pls.append(pl)
        scs.append(sc)
    torch.cuda.synchronize()
    h_pl = [host(p).copy() for p in pls]
    h_sc = [host(s).copy() for s in scs]
    idx, codes = oracle.unpack(h_pl[3])
    idx[[5, 700], 9], idx[[5, 700], 10] = idx[[5, 700], 10], idx[[5, 700], 9]
    h_pl[3] = oracle.pack(idx, codes)                       # two malformed records of peer 3
    h_sc[7][11] = np.nan                                     # one bad scale of peer 7
    for q, c, z in ((5, 20, 0.0), (6, 30, -0.0)):            # zero scales, codes all 3: both
        idx, codes = oracle.unpack(h_pl[q])                  # levels decode to -0.0, yet the
        codes[c, :] = 3                                      # code bits still count
        h_pl[q] = oracle.pack(idx, codes)
        h_sc[q][c] = z
    pls = [torch.from_numpy(p).to(DEV) for p in h_pl]
    scs = [torch.from_numpy(s).to(DEV) for s in h_sc]
    theta = synth.theta(n, gen, DEV)
    theta2 = theta.clone()
    stats = spl.new_peer_stats(P, DEV)
    mean = spl.decode_aggregate(pls, scs, n, theta=theta, lr=0.7, stats=stats)
    mean_plain = spl.decode_aggregate(pls, scs, n, theta=theta2, lr=0.7)
    torch.cuda.synchronize()
    assert_bit_equal(host(mean), host(mean_plain), "mean with and without statistics")
    assert_bit_equal(host(theta), host(theta2), "theta with and without statistics")
    got = spl.read_peer_stats(stats)
    ref = oracle.peer_stats(h_pl, h_sc, n)
    for key in ("rejected", "big", "negative"):
        assert np.array_equal(got[key], ref[key]), key
    assert_bit_equal(got["max_scale"], ref["max_scale"], "max_scale")
    assert np.allclose(got["sumsq"], ref["sumsq"], rtol=1e-6, atol=0)   # fp32 per record
    assert ref["rejected"][3] == 2 and ref["rejected"][7] == 1
    assert ref["rejected"][5] == 0 and ref["rejected"][6] == 0
    # accumulated across calls
    spl.decode_aggregate(pls, scs, n, stats=stats)
    torch.cuda.synchronize()
    again = spl.read_peer_stats(stats)
    for key in ("rejected", "big", "negative"):
        assert np.array_equal(again[key], 2 * ref[key]), key
    assert_bit_equal(again["max_scale"], ref["max_scale"], "max_scale after two calls")
    assert np.allclose(again["sumsq"], 2 * ref["sumsq"], rtol=1e-6, atol=0)


# ---------------------------------------------------------------------------------------------
# Many peers: the decode unpacks peers in groups of 64, so these span several groups
# ---------------------------------------------------------------------------------------------
def random_records(rng, C: int, L: int = 4096, k: int = 64):
    """C records with random strictly ascending indices and random codes, as (idx, codes)."""
    idx = np.sort(np.stack([rng.choice(L, k, replace=False) for _ in range(C)]), axis=1)
    return idx.astype(np.uint16), rng.integers(0, 4, size=(C, k)).astype(np.uint8)


@pytest.mark.parametrize("P", [65, 130, 256])
def test_many_peers_span_several_groups(P):
    n = 9 * 4096 + 11
    C = 10
    rng = np.random.default_rng(P)
    pls, scs = [], []
    for p in range(P):
        idx, codes = random_records(rng, C)
        if p % 37 == 5:
            idx[p % C, [7, 8]] = idx[p % C, [8, 7]]          # a malformed record
        pls.append(oracle.pack(idx, codes))
        scs.append((rng.random(C) * 1e-3).astype(np.float32))
    theta = synth.theta(n, synth.generator(P, DEV), DEV)
    th_h = host(theta).copy()
    theta2 = theta.clone()
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    stats = spl.new_peer_stats(P, DEV)
    d_pls = [torch.from_numpy(p).to(DEV) for p in pls]
    d_scs = [torch.from_numpy(s).to(DEV) for s in scs]
    mean = spl.decode_aggregate(d_pls, d_scs, n, theta=theta, lr=0.7, flags=flags, stats=stats)
    # and without statistics (the shape whose records come as one bulk copy each)
    flags2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    mean2 = spl.decode_aggregate(d_pls, d_scs, n, theta=theta2, lr=0.7, flags=flags2)
    torch.cuda.synchronize()
    o_mean, o_flags = oracle.decode_aggregate(pls, scs, n, theta=th_h, lr=0.7)
    assert int(flags.item()) == int(flags2.item()) == o_flags == oracle.FLAG_BAD_RECORD
    assert_bit_equal(host(mean), o_mean, f"P={P}: mean")
    assert_bit_equal(host(theta), th_h, f"P={P}: theta")
    assert_bit_equal(host(mean2), o_mean, f"P={P}: mean without statistics")
    assert_bit_equal(host(theta2), th_h, f"P={P}: theta without statistics")
    got = spl.read_peer_stats(stats)
    ref = oracle.peer_stats(pls, scs, n)
    for key in ("rejected", "big", "negative"):
        assert np.array_equal(got[key], ref[key]), key
    assert_bit_equal(got["max_scale"], ref["max_scale"], "max_scale")
    assert np.allclose(got["sumsq"], ref["sumsq"], rtol=1e-6, atol=0)


# ---------------------------------------------------------------------------------------------
# CUDA graphs: the calls are stream-ordered, allocate nothing and never synchronise, so a
# round can be captured once and replayed
# ---------------------------------------------------------------------------------------------
def test_round_captures_into_a_cuda_graph_and_replays_like_eager_calls():
    n = 9 * 4096 + 5
    P = 3
    gen = synth.generator(77, DEV)
    deltas = [synth.laplace(n, 1e-4, gen, DEV) for _ in range(3)]
    peers = []
    for p in range(P):
        pl, sc = gpu_round(synth.laplace(n, 1e-4, gen, DEV), torch.zeros(n, device=DEV), 1.0)
        peers.append((pl, sc))
    theta0 = synth.theta(n, gen, DEV)
    C = spl.num_chunks(n)

    def make_state():
        return {"delta": torch.empty(n, device=DEV), "ef": torch.zeros(n, device=DEV),
                "payload": torch.empty((C, 112), dtype=torch.uint8, device=DEV),
                "scales": torch.empty(C, device=DEV), "mean": torch.empty(n, device=DEV),
                "theta": theta0.clone()}

    def step(st):
        spl.ef_compress(st["delta"], st["ef"], 0.9, payload=st["payload"], scales=st["scales"])
        spl.decode_aggregate([p[0] for p in peers] + [st["payload"]],
                             [p[1] for p in peers] + [st["scales"]], n, mean=st["mean"],
                             theta=st["theta"], lr=0.7)

    eager, graphed = make_state(), make_state()
    torch.cuda.synchronize()
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):        # warm-up on the capture stream
        graphed["delta"].copy_(deltas[0])
        step(graphed)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for k in ("ef", "theta"):             # restart both from the same state
        graphed[k].copy_(eager[k])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(graphed)
    for r in range(3):                    # three rounds, a fresh delta each
        eager["delta"].copy_(deltas[r])
        step(eager)
        graphed["delta"].copy_(deltas[r])
        g.replay()
    torch.cuda.synchronize()
    for k in ("payload", "scales", "ef", "mean", "theta"):
        assert_bit_equal(host(graphed[k]), host(eager[k]), f"graph replay: {k}")
