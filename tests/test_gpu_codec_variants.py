"""GPU parity of the codec variants (other chunk length L and k, the mean-abs scale rule)
against the oracle's variants, on the same seeded inputs.

Bar, as for the default codec: payload bytes, scales and the error buffer bit-exact; the mean
and theta bit-exact (fixed peer order, one rounding each); statistics counts exact.  Every
case spans several chunks and a ragged tail; the edge cases cover the generic select (ties,
zeros, few nonzeros) at each geometry, 4-byte-aligned records (52 and 56 bytes) and
malformed records whose fault lies past the 64th entry.
"""
import numpy as np
import pytest
import torch

import compressed_pseudo_gradient_gb300 as spl
import oracle
from compressed_pseudo_gradient_gb300 import synth
from parity_util import assert_bit_equal, host

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
MAX, MEAN = spl.SCALE_MAX_ABS, spl.SCALE_MEAN_ABS
GEOMETRIES = [(4096, 32), (4096, 128), (2048, 32), (8192, 128)]
CODECS = [(4096, 64, MEAN)] + [(L, k, r) for (L, k) in GEOMETRIES for r in (MAX, MEAN)]


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def compare_round(delta, ef, beta, codec, what):
    d_h, e_h = host(delta), host(ef)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    payload, scales = spl.ef_compress(delta, ef, beta, codec=codec, flags=flags)
    torch.cuda.synchronize()
    o_pl, o_sc, o_flags = oracle.ef_compress(d_h, e_h, beta, bf16=delta.dtype == torch.bfloat16,
                                             codec=codec)
    assert payload.shape == (oracle.num_chunks(delta.numel(), codec), oracle.record_bytes(codec))
    assert_bit_equal(host(payload), o_pl, f"{what}: payload")
    assert_bit_equal(host(scales), o_sc, f"{what}: scales")
    assert_bit_equal(host(ef), e_h, f"{what}: error buffer")
    assert int(flags.item()) == o_flags
    return payload, scales, o_pl, o_sc


@pytest.mark.parametrize("codec", CODECS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_variant_rounds_match_oracle(codec, dtype):
    L = codec[0]
    n = 37 * L + 123
    gen = synth.generator(7 + L + codec[1] + codec[2], DEV)
    ef = torch.zeros(n, device=DEV)
    for r in range(3):
        if dtype == torch.bfloat16:
            delta = synth.heavy_tail_bf16(n, gen, DEV)
        else:
            delta = synth.laplace(n, 1e-3, gen, DEV)
        compare_round(delta, ef, 0.95, codec, f"{codec} {dtype} round {r}")


@pytest.mark.parametrize("codec", CODECS)
def test_variant_edge_chunks(codec):
    """Chunks that take the generic select (zeros, constants, heavy ties, fewer nonzeros than
    k) and tiny tensors, at each geometry."""
    L, k, _ = codec
    rng = np.random.default_rng(L + k)
    few = np.zeros(L, np.float32)
    few[rng.choice(L, k // 2, replace=False)] = rng.standard_normal(k // 2)
    ties = np.round(rng.standard_normal(L) * 2).astype(np.float32)
    coarse = (rng.integers(-3, 4, L) * 0.25).astype(np.float32)
    spikes = (rng.standard_normal(L) * 1e-3).astype(np.float32)
    spikes[rng.choice(L, k, replace=False)] = rng.choice([-1.0, 1.0], k) * (1 + rng.random(k))
    blocks = [np.zeros(L), np.full(L, -2.5), np.arange(L) * -1.0, few, ties, coarse, spikes,
              np.full(L, 1.4e-45)]
    delta = torch.cat([torch.as_tensor(b, dtype=torch.float32) for b in blocks]).to(DEV)
    ef = torch.zeros_like(delta)
    compare_round(delta, ef, 1.0, codec, f"{codec} edge round 1")
    compare_round(torch.zeros_like(delta), ef, 1.0, codec, f"{codec} edge round 2")


@pytest.mark.parametrize("codec", CODECS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_variant_exact_ties_and_sparse_chunks(codec, dtype):
    """At each geometry: boundary bins of up to 64 exactly tied keys (ranked by index), the
    same beside keys of the same bin that differ, a bin of more than 64 tied keys, and chunks
    with fewer than k nonzeros; three rounds, the last with a zero delta, so selected zeros
    come back as tied residuals."""
    L, k, _ = codec
    rng = np.random.default_rng(3 * L + k)

    def tied(n_top, n_tie, top=2.0, tie=1.0):
        x = np.zeros(L, np.float32)
        pos = rng.choice(L, n_top + n_tie, replace=False)
        x[pos[:n_top]] = top * rng.choice([-1, 1], n_top)
        x[pos[n_top:]] = tie * rng.choice([-1, 1], n_tie)
        return x

    mixed = tied(k - 24, 30)
    mixed[rng.choice(np.flatnonzero(mixed == 0), 3, replace=False)] = 1.0 + 2.0 ** -20
    sparse = np.zeros(L, np.float32)
    sparse[rng.choice(L, k // 4, replace=False)] = rng.standard_normal(k // 4)
    blocks = [tied(k - 24, 40), tied(k - 1, 2), tied(0, 65), tied(0, k + 1), mixed, sparse,
              tied(k - 4, 4, 1.0, 1.0)]
    delta = torch.cat([torch.as_tensor(b, dtype=torch.float32) for b in blocks]).to(DEV)
    delta = delta.to(dtype)
    ef = torch.zeros(delta.numel(), device=DEV)
    compare_round(delta, ef, 1.0, codec, f"{codec} {dtype} ties round 1")
    compare_round(delta, ef, 0.95, codec, f"{codec} {dtype} ties round 2")
    compare_round(torch.zeros_like(delta), ef, 0.95, codec, f"{codec} {dtype} ties round 3")
    for n in (1, k - 1, k, k + 1, L - 1, L + 1):
        d = synth.laplace(n, 1.0, synth.generator(n, DEV), DEV)
        compare_round(d, torch.zeros(n, device=DEV), 0.5, codec, f"{codec} n={n}")


@pytest.mark.parametrize("codec", [(L, k, MAX) for (L, k) in GEOMETRIES])
def test_variant_decode_matches_oracle(codec):
    L, k, _ = codec
    n = 21 * L + 77
    P = 5
    pls, scs, o_pls, o_scs = [], [], [], []
    for p in range(P):
        d = synth.laplace(n, 1e-3, synth.generator(50 + p, DEV), DEV)
        pl, sc, opl, osc = compare_round(d, torch.zeros(n, device=DEV), 1.0, codec, f"peer {p}")
        pls.append(pl), scs.append(sc), o_pls.append(opl), o_scs.append(osc)
    theta = synth.theta(n, synth.generator(3, DEV), DEV)
    th_h = host(theta).copy()
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    stats = spl.new_peer_stats(P, DEV)
    mean = spl.decode_aggregate(pls, scs, n, theta=theta, lr=0.7, flags=flags, stats=stats,
                                codec=codec)
    mean_plain = spl.decode_aggregate(pls, scs, n, codec=codec)
    torch.cuda.synchronize()
    o_mean, o_flags = oracle.decode_aggregate(o_pls, o_scs, n, theta=th_h, lr=0.7, codec=codec)
    assert int(flags.item()) == o_flags == 0
    assert_bit_equal(host(mean), o_mean, f"{codec}: mean")
    assert_bit_equal(host(mean_plain), o_mean, f"{codec}: mean without theta or statistics")
    assert_bit_equal(host(theta), th_h, f"{codec}: theta")
    got = spl.read_peer_stats(stats)
    ref = oracle.peer_stats(o_pls, o_scs, n, codec=codec)
    for key in ("rejected", "big", "negative"):
        assert np.array_equal(got[key], ref[key]), key
    assert_bit_equal(got["max_scale"], ref["max_scale"], "max_scale")
    assert np.allclose(got["sumsq"], ref["sumsq"], rtol=1e-6, atol=0)


@pytest.mark.parametrize("codec", [(4096, 128, MAX), (2048, 32, MAX), (8192, 128, MAX)])
def test_variant_malformed_records_rejected_like_oracle(codec):
    L, k, _ = codec
    n = 6 * L
    pls, scs = [], []
    for p in range(3):
        d = synth.laplace(n, 1e-4, synth.generator(90 + p, DEV), DEV)
        pl, sc = spl.ef_compress(d, torch.zeros(n, device=DEV), 1.0, codec=codec)
        pls.append(host(pl).copy()), scs.append(host(sc).copy())
    idx, codes = oracle.unpack(pls[1], codec)
    idx[0, [k - 3, k - 2]] = idx[0, [k - 2, k - 3]]   # chunk 0: not ascending near the end
    idx[2, 20] = idx[2, 19]                            # chunk 2: duplicate
    # chunk 3: duplicate; for k > 32 the two entries one lane of the adding warp holds
    idx[3, k - 1] = idx[3, k - 33 if k > 32 else k - 2]
    pls[1] = oracle.pack(idx, codes, codec)
    scs[2][1] = np.nan
    scs[2][4] = -1.0
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    stats = spl.new_peer_stats(3, DEV)
    mean = spl.decode_aggregate([torch.from_numpy(p).to(DEV) for p in pls],
                                [torch.from_numpy(s).to(DEV) for s in scs], n, flags=flags,
                                stats=stats, codec=codec)
    torch.cuda.synchronize()
    o_mean, o_flags = oracle.decode_aggregate(pls, scs, n, codec=codec)
    assert int(flags.item()) == o_flags == oracle.FLAG_BAD_RECORD
    assert_bit_equal(host(mean), o_mean, f"{codec}: mean with rejected records")
    got = spl.read_peer_stats(stats)
    assert list(got["rejected"]) == list(oracle.peer_stats(pls, scs, n, codec=codec)["rejected"])
    assert list(got["rejected"]) == [0, 3, 2]


def test_variant_multi_tensor_matches_single_calls():
    codec = (2048, 32, MEAN)
    sizes = [2048 * 3, 100, 2048 * 5 + 7, 0, 1]
    gen = synth.generator(4, DEV)
    deltas = [synth.laplace(m, 1e-3, gen, DEV) for m in sizes]
    efs = [synth.laplace(m, 1e-4, gen, DEV) for m in sizes]
    efs2 = [e.clone() for e in efs]
    payload, scales = spl.ef_compress_multi(deltas, efs, 0.9, codec=codec)
    parts_p, parts_s = [], []
    for d, e in zip(deltas, efs2):
        if d.numel():
            p, s = spl.ef_compress(d, e, 0.9, codec=codec)
            parts_p.append(p), parts_s.append(s)
    torch.cuda.synchronize()
    assert_bit_equal(host(payload), host(torch.cat(parts_p)), "multi-tensor payload")
    assert_bit_equal(host(scales), host(torch.cat(parts_s)), "multi-tensor scales")
    for e, e2 in zip(efs, efs2):
        assert_bit_equal(host(e), host(e2), "multi-tensor error buffers")


def test_variant_host_error_buffer_rejected():
    n = 3 * 4096
    delta = torch.zeros(n, device=DEV)
    ef = torch.zeros(n).pin_memory()
    with pytest.raises(spl.SplError):
        spl.ef_compress(delta, ef, 1.0, codec=(4096, 32, MAX))
    spl.ef_compress(delta, ef, 1.0, codec=(4096, 64, MAX))   # the default codec takes it


@pytest.mark.parametrize("codec", [(L, k, MAX) for (L, k) in GEOMETRIES])
@pytest.mark.parametrize("P", [24, 70, 200])
def test_variant_many_peers_span_several_groups(codec, P):
    """Peers are unpacked in groups (32 for k = 128 at L = 8192, 64 otherwise); 24, 70 and 200
    peers span one to seven groups, and 200 peers need the second scale slot of a lane where a
    CTA has four warps (L = 2048)."""
    L, k, _ = codec
    n = 5 * L + 9
    C = 6
    rng = np.random.default_rng(P + L + k)
    pls, scs = [], []
    for p in range(P):
        idx = np.sort(np.stack([rng.choice(L, k, replace=False) for _ in range(C)]), axis=1)
        idx = idx.astype(np.uint16)
        codes = rng.integers(0, 4, size=(C, k)).astype(np.uint8)
        if p % 11 == 3:
            idx[p % C, [k - 2, k - 1]] = idx[p % C, [k - 1, k - 2]]   # a malformed record
        pls.append(oracle.pack(idx, codes, codec))
        scs.append((rng.random(C) * 1e-3).astype(np.float32))
    theta = synth.theta(n, synth.generator(P, DEV), DEV)
    th_h = host(theta).copy()
    theta2 = theta.clone()
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    stats = spl.new_peer_stats(P, DEV)
    d_pls = [torch.from_numpy(p).to(DEV) for p in pls]
    d_scs = [torch.from_numpy(s).to(DEV) for s in scs]
    mean = spl.decode_aggregate(d_pls, d_scs, n, theta=theta, lr=0.7, flags=flags, stats=stats,
                                codec=codec)
    # and without statistics (another receiver shape: bulk-copied records where they are
    # 16-byte multiples)
    flags2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    mean2 = spl.decode_aggregate(d_pls, d_scs, n, theta=theta2, lr=0.7, flags=flags2, codec=codec)
    torch.cuda.synchronize()
    o_mean, o_flags = oracle.decode_aggregate(pls, scs, n, theta=th_h, lr=0.7, codec=codec)
    assert int(flags.item()) == int(flags2.item()) == o_flags == oracle.FLAG_BAD_RECORD
    assert_bit_equal(host(mean), o_mean, f"{codec} P={P}: mean")
    assert_bit_equal(host(theta), th_h, f"{codec} P={P}: theta")
    assert_bit_equal(host(mean2), o_mean, f"{codec} P={P}: mean without statistics")
    assert_bit_equal(host(theta2), th_h, f"{codec} P={P}: theta without statistics")
    got = spl.read_peer_stats(stats)
    ref = oracle.peer_stats(pls, scs, n, codec=codec)
    for key in ("rejected", "big", "negative"):
        assert np.array_equal(got[key], ref[key]), key
    assert np.allclose(got["sumsq"], ref["sumsq"], rtol=1e-6, atol=0)


@pytest.mark.parametrize("codec", CODECS)
def test_variant_nonfinite_inputs_flagged_and_deterministic(codec):
    """Inf and NaN in a few chunks: the records are still the oracle's, bit for bit (a NaN ranks
    above every number and codes as +0.5 s); scales and the error buffer agree up to NaN bit
    patterns; the non-finite flag is set."""
    L, k, _ = codec
    n = 4 * L + 5
    delta = synth.laplace(n, 1e-4, synth.generator(9 + L + k, DEV), DEV)
    delta[100] = float("inf")
    delta[L + 7] = float("nan")
    delta[2 * L + 9] = -float("inf")
    delta[2 * L + 10] = float("nan")
    delta[3 * L + 1] = float("inf")
    delta[3 * L + 2] = -float("inf")
    ef = torch.zeros(n, device=DEV)
    d_h, e_h = host(delta), host(ef)
    flags = torch.zeros(1, dtype=torch.int32, device=DEV)
    payload, scales = spl.ef_compress(delta, ef, 1.0, codec=codec, flags=flags)
    torch.cuda.synchronize()
    o_pl, o_sc, o_flags = oracle.ef_compress(d_h, e_h, 1.0, codec=codec)
    assert int(flags.item()) & spl.FLAG_NONFINITE and o_flags & oracle.FLAG_NONFINITE
    assert_bit_equal(host(payload), o_pl, f"{codec}: payload with non-finite values")
    g_sc = host(scales)
    assert np.array_equal(np.isnan(g_sc), np.isnan(o_sc))
    fin = ~np.isnan(o_sc)
    assert_bit_equal(g_sc[fin], o_sc[fin], f"{codec}: scales that are not NaN")
    g_e = host(ef)
    assert ((g_e == e_h) | (np.isnan(g_e) & np.isnan(e_h))).all()
