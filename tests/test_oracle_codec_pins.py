"""Pins of the oracle's codec variants (other chunk length L, other k, the mean-abs scale rule)
to facts fixed outside the oracle (CPU only).

The pages fix L = 4096 and k = 64, give the index width as ceil(log2 L) and leave the scale
rule open ("The Sparse Frontier", "SparseLoCo: Three Compression Levers in One Pass").  The
checks: record sizes from the size equation and hand-derived bytes (tests/golden/
codec_variants.txt), the big-integer definition of the bit layout, exhaustive enumeration of
the chosen set on tiny chunks, and chunks whose scale, codes and residuals are exact by
construction, including one where the pairwise and the sequential sums differ.
"""
import itertools
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "codec_variants.txt")
F32 = np.float32
MAX, MEAN = oracle.SCALE_MAX, oracle.SCALE_MEAN_ABS
GEOMETRIES = [(2048, 32), (4096, 32), (4096, 64), (4096, 128), (8192, 128)]


def _golden():
    sizes, data = {}, {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split(";")[0].strip()
            if not line or line.startswith("#"):
                continue
            key, val = (t.strip() for t in line.split("="))
            if key.startswith("size_"):
                _, L, k = key.split("_")
                sizes[(int(L), int(k))] = int(val)
            else:
                data[key] = bytes(int(t, 16) for t in val.split())
    return sizes, data


def _fields(L):
    return 2 + (L - 1).bit_length()


def _big_int_record(idx, codes, L, k):
    """The record as the bit string definition gives it: field r at bits [r*b, r*b + b)."""
    b = _fields(L)
    v = sum((int(codes[r]) | int(idx[r]) << 2) << (b * r) for r in range(k))
    return v.to_bytes((k * b + 7) // 8, "little")


def _decode_dense(payload, scales, n, L, k):
    """Dense decoded vector of one peer, read from the bit string with Python integers."""
    b = _fields(L)
    C = payload.shape[0]
    out = np.zeros(C * L, dtype=np.float32)
    for c in range(C):
        v = int.from_bytes(bytes(payload[c]), "little")
        s = F32(scales[c])
        for r in range(k):
            f = (v >> (b * r)) & ((1 << b) - 1)
            q = F32(1.5) * s if f & 1 else F32(0.5) * s
            out[c * L + (f >> 2)] = -q if f & 2 else q
    return out[:n]


# ---------------------------------------------------------------------------------------------
# Sizes and layout
# ---------------------------------------------------------------------------------------------
def test_record_sizes_follow_the_size_equation():
    sizes, _ = _golden()
    assert sizes[(4096, 64)] == 112
    for (L, k), nbytes in sizes.items():
        assert oracle.record_bytes((L, k, MAX)) == nbytes
        assert oracle.record_bytes((L, k, MEAN)) == nbytes
    assert oracle.record_bytes(None) == 112
    for bad in [(3, 1, MAX), (1, 1, MAX), (4096, 0, MAX), (8, 9, MAX), (4096, 64, 2)]:
        with pytest.raises(ValueError):
            oracle.record_bytes(bad)
    assert oracle.num_chunks(2048 * 3 + 1, (2048, 32, MAX)) == 4
    assert oracle.num_chunks(8192, (8192, 128, MAX)) == 1


def test_variant_pack_known_answer_bytes():
    _, g = _golden()
    idx = np.arange(32, dtype=np.uint16)[None]
    codes = np.zeros((1, 32), np.uint8)
    codes[0, 0] = 3
    assert bytes(oracle.pack(idx, codes, (2048, 32, MAX))[0][:12]) == g["C_first12"]
    idx = np.zeros((1, 128), np.uint16)
    codes = np.zeros((1, 128), np.uint8)
    idx[0, 127], codes[0, 127] = 8191, 3
    rec = bytes(oracle.pack(idx, codes, (8192, 128, MAX))[0])
    assert len(rec) == 240 and rec[-2:] == g["D_last2"] and not any(rec[:-2])


@pytest.mark.parametrize("L,k", GEOMETRIES + [(8, 3), (16, 4)])
def test_variant_pack_matches_big_integer_definition(L, k):
    rng = np.random.default_rng(L + k)
    C = 12
    idx = np.sort(np.stack([rng.choice(L, k, replace=False) for _ in range(C)]), axis=1)
    idx = idx.astype(np.uint16)
    codes = rng.integers(0, 4, size=(C, k)).astype(np.uint8)
    payload = oracle.pack(idx, codes, (L, k, MAX))
    for c in range(C):
        assert bytes(payload[c]) == _big_int_record(idx[c], codes[c], L, k)
    i2, c2 = oracle.unpack(payload, (L, k, MAX))
    assert (i2 == idx).all() and (c2 == codes).all()


# ---------------------------------------------------------------------------------------------
# The mean-abs scale's pairwise sum
# ---------------------------------------------------------------------------------------------
def test_pairwise_sum_order():
    e = F32(2.0 ** -24)   # half an ulp of 1.0: 1 + e rounds back to 1 (tie to even)
    one = F32(1.0)
    assert oracle.pairwise_sum(np.array([one])) == one
    # ((1 + e) + (e + e)) = 1 + 2^-23, where a left-to-right sum gives 1
    assert oracle.pairwise_sum(np.array([one, e, e, e])) == F32(1.0 + 2.0 ** -23)
    # two such halves: 2 + 2^-22 (exact)
    assert oracle.pairwise_sum(np.array([one, e, e, e] * 2)) == F32(2.0 + 2.0 ** -22)
    # n = 3 splits after the first entry: e + (e + 1) = e + 1 = 1; a split after two would
    # give (e + e) + 1 = 1 + 2^-23
    assert oracle.pairwise_sum(np.array([e, e, one])) == one


# ---------------------------------------------------------------------------------------------
# The sender with a variant codec
# ---------------------------------------------------------------------------------------------
def _chosen_by_definition(a, k):
    """The unique k-subset S with every chosen entry ranked above every other entry."""
    L = len(a)
    mag = np.abs(a)
    found = []
    for S in itertools.combinations(range(L), k):
        rest = [j for j in range(L) if j not in S]
        if all(mag[i] > mag[j] or (mag[i] == mag[j] and i < j) for i in S for j in rest):
            found.append(S)
    assert len(found) == 1
    return list(found[0])


@pytest.mark.parametrize("L,k,rule", [(8, 3, MAX), (8, 3, MEAN), (16, 4, MAX), (16, 4, MEAN)])
def test_variant_sender_on_tiny_chunks(L, k, rule):
    rng = np.random.default_rng(31 * L + k + rule)
    for trial in range(20):
        # small integers and halves: many ties, every sum below exact
        delta = (rng.integers(-6, 7, size=2 * L) / 2).astype(np.float32)
        ef = np.zeros(2 * L, np.float32)
        payload, scales, flags = oracle.ef_compress(delta, ef, 1.0, codec=(L, k, rule))
        assert flags == 0 and payload.shape == (2, oracle.record_bytes((L, k, rule)))
        for c in range(2):
            a = delta[c * L:(c + 1) * L]
            S = _chosen_by_definition(a, k)
            m = np.abs(a[S])
            if rule == MAX:
                s = F32(np.abs(a).max()) / F32(1.5)
            elif k == 3:   # floor split: x0 + (x1 + x2)
                s = (m[0] + (m[1] + m[2])) / F32(3)
            else:          # (x0 + x1) + (x2 + x3)
                s = ((m[0] + m[1]) + (m[2] + m[3])) / F32(4)
            assert scales[c] == s
            codes = [(2 if a[j] < 0 else 0) | (1 if abs(a[j]) > s else 0) for j in S]
            assert bytes(payload[c]) == _big_int_record(S, codes, L, k)
            want = a.copy()
            for j, code in zip(S, codes):
                q = F32(1.5) * s if code & 1 else F32(0.5) * s
                want[j] = a[j] - (-q if code & 2 else q)
            assert np.array_equal(ef[c * L:(c + 1) * L], want)


@pytest.mark.parametrize("L,k", [(4096, 64), (2048, 32), (8192, 128)])
def test_mean_abs_planted_chunk_is_exact(L, k):
    """k spikes alternating +1 and -5 over small noise: mean |a| = 3 exactly, so s = 3 (the
    max-abs rule would give 5 / 1.5); +1 codes 0 (q = 1.5) and -5 codes 3 (q = -4.5), so
    every transmitted residual is -0.5 exactly."""
    rng = np.random.default_rng(k)
    delta = (rng.uniform(-0.5, 0.5, L) * 1e-3).astype(np.float32)
    pos = np.sort(rng.choice(L, k, replace=False))
    delta[pos] = np.where(np.arange(k) % 2 == 0, 1.0, -5.0).astype(np.float32)
    ef = np.zeros(L, np.float32)
    payload, scales, _ = oracle.ef_compress(delta, ef, 1.0, codec=(L, k, MEAN))
    assert scales[0] == F32(3.0)
    codes = [0 if r % 2 == 0 else 3 for r in range(k)]
    assert bytes(payload[0]) == _big_int_record(pos, codes, L, k)
    assert (ef[pos] == F32(-0.5)).all()
    rest = np.setdiff1d(np.arange(L), pos)
    assert np.array_equal(ef[rest], delta[rest])
    _, s_max, _ = oracle.ef_compress(delta, np.zeros(L, np.float32), 1.0, codec=(L, k, MAX))
    assert s_max[0] == F32(5.0) / F32(1.5)


def test_mean_abs_sums_pairwise_in_index_order():
    """32 spikes at positions 0..31 in the pattern 1, e, e, e (e = 2^-24): the pairwise sum
    is 8 + 2^-20, so s = 1/4 + 2^-25; a left-to-right sum would give exactly 8 (s = 1/4)."""
    L, k = 4096, 32
    e = 2.0 ** -24
    delta = np.zeros(L, np.float32)
    delta[:32] = np.array([1.0, e, e, e] * 8, np.float32)
    ef = np.zeros(L, np.float32)
    payload, scales, _ = oracle.ef_compress(delta, ef, 1.0, codec=(L, k, MEAN))
    assert scales[0] == F32(0.25 + 2.0 ** -25)
    idx, _ = oracle.unpack(payload, (L, k, MEAN))
    assert (idx[0] == np.arange(32)).all()


def test_mean_abs_sums_in_index_order_not_rank_order():
    """Chosen |a| in index order 1, 2^-24, 0.5, 2^-25: (1 + 2^-24) + (0.5 + 2^-25) = 1 + 0.5
    (both small terms are ties that round to even), so s = 1.5 / 4; in rank order the sum
    would be (1 + 0.5) + 3 * 2^-25 = 1.5 + 2^-23."""
    L, k = 16, 4
    delta = np.zeros(L, np.float32)
    delta[[0, 1, 2, 3]] = np.array([1.0, 2.0 ** -24, -0.5, 2.0 ** -25], np.float32)
    ef = np.zeros(L, np.float32)
    _, scales, _ = oracle.ef_compress(delta, ef, 1.0, codec=(L, k, MEAN))
    assert scales[0] == F32(0.375)


def test_mean_abs_pairs_neighbours_in_index_order():
    """Chosen |a| in index order 1, 2^-24, 2^-24, 1 + 2^-23.  Pairwise: 1 + 2^-24 rounds to 1
    (a tie, to even) and 2^-24 + (1 + 2^-23) to 1 + 2^-22 (a tie, to even), so the sum is
    2 + 2^-22 and s = 1/2 + 2^-24.  Any other order the summation might take (left to right,
    rank order, the pairs shifted by one place) rounds the small terms away: s = 1/2."""
    L, k = 16, 4
    delta = np.zeros(L, np.float32)
    delta[[0, 1, 2, 3]] = np.array([1.0, 2.0 ** -24, -(2.0 ** -24), 1.0 + 2.0 ** -23], np.float32)
    ef = np.zeros(L, np.float32)
    _, scales, _ = oracle.ef_compress(delta, ef, 1.0, codec=(L, k, MEAN))
    assert scales[0] == F32(0.5 + 2.0 ** -24)


def test_variant_tail_chunk_pads_lose_ties_and_are_not_stored():
    L, k = 2048, 32
    n = L + 5
    delta = np.full(n, 0.25, np.float32)
    delta[L:] = np.array([1, -2, 3, -4, 5], np.float32)
    ef = np.zeros(n, np.float32)
    payload, scales, _ = oracle.ef_compress(delta, ef, 1.0, codec=(L, k, MAX))
    assert payload.shape == (2, 52)
    idx, codes = oracle.unpack(payload, (L, k, MAX))
    assert (idx[1] == np.arange(32)).all()              # 5 real entries, then pads 5..31
    s = F32(5.0) / F32(1.5)
    assert scales[1] == s
    assert list(codes[1][:5]) == [0, 2, 0, 3, 1] and (codes[1][5:] == 0).all()
    mean, _ = oracle.decode_aggregate([payload], [scales], n, codec=(L, k, MAX))
    assert mean.shape == (n,)
    assert np.array_equal(mean, _decode_dense(payload, scales, n, L, k))


@pytest.mark.parametrize("L,k,rule", [(2048, 32, MEAN), (4096, 128, MAX), (8192, 128, MEAN)])
def test_variant_residual_conserves_the_accumulator(L, k, rule):
    """ef_new = a off the chosen set; on it ef_new = RN(a - q), so ef_new + q - a is at most
    half an ulp of ef_new (checked in fp64, where the sum of the three is exact)."""
    rng = np.random.default_rng(L + k)
    n = 3 * L + 77
    delta = rng.laplace(0, 1e-3, n).astype(np.float32)
    ef0 = rng.laplace(0, 1e-3, n).astype(np.float32)
    ef = ef0.copy()
    beta = 0.5
    payload, scales, _ = oracle.ef_compress(delta, ef, beta, codec=(L, k, rule))
    a = (np.float64(beta) * ef0.astype(np.float64) + delta.astype(np.float64)).astype(np.float32)
    dec = _decode_dense(payload, scales, n, L, k)
    sent = dec != 0
    assert np.array_equal(ef[~sent], a[~sent])
    err = np.abs(ef[sent].astype(np.float64) + dec[sent] - a[sent])
    assert (err <= 0.5 * np.spacing(np.abs(ef[sent])).astype(np.float64)).all()
    # every full chunk sends k real (nonzero) entries, the 77-value tail min(k, 77)
    assert sent.sum() == k * (oracle.num_chunks(n, (L, k, rule)) - 1) + min(k, 77)


# ---------------------------------------------------------------------------------------------
# The receiver with a variant codec
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("L,k", [(4096, 128), (2048, 32)])
def test_variant_decode_closed_cases(L, k):
    rng = np.random.default_rng(k)
    n = 2 * L
    codec = (L, k, MAX)
    peers = []
    for p in range(4):   # disjoint supports: peer p owns positions = p (mod 4)
        idx = np.sort(np.stack([rng.choice(L // 4, k, replace=False) * 4 + p for _ in range(2)]),
                      axis=1).astype(np.uint16)
        codes = rng.integers(0, 4, size=(2, k)).astype(np.uint8)
        scales = np.array([0.75, 2.0], np.float32)
        peers.append((oracle.pack(idx, codes, codec), scales))
    single, flags = oracle.decode_aggregate([peers[0][0]], [peers[0][1]], n, codec=codec)
    assert flags == 0
    assert np.array_equal(single, _decode_dense(peers[0][0], peers[0][1], n, L, k))
    mean, _ = oracle.decode_aggregate([p[0] for p in peers], [p[1] for p in peers], n,
                                      codec=codec)
    want = sum(_decode_dense(p[0], p[1], n, L, k) for p in peers) / F32(4)
    assert np.array_equal(mean, want.astype(np.float32))
    # a peer and its sign-flipped copy cancel exactly
    i0, c0 = oracle.unpack(peers[0][0], codec)
    flipped = oracle.pack(i0, c0 ^ 2, codec)
    zero, _ = oracle.decode_aggregate([peers[0][0], flipped], [peers[0][1]] * 2, n, codec=codec)
    assert not zero.any()


def test_variant_malformed_records_and_peer_stats():
    L, k = 2048, 32
    codec = (L, k, MAX)
    idx = np.tile(np.arange(0, 64, 2, dtype=np.uint16), (2, 1))
    codes = np.tile(np.array([0, 1, 2, 3], np.uint8), (2, 8))
    good = oracle.pack(idx, codes, codec)
    bad_idx = idx.copy()
    bad_idx[1, [4, 5]] = bad_idx[1, [5, 4]]                # record 1 not ascending
    bad = oracle.pack(bad_idx, codes, codec)
    sc = np.array([2.0, 4.0], np.float32)
    mean, flags = oracle.decode_aggregate([good, bad], [sc, sc], 2 * L, codec=codec)
    assert flags == oracle.FLAG_BAD_RECORD
    st = oracle.peer_stats([good, bad], [sc, sc], 2 * L, codec=codec)
    assert list(st["rejected"]) == [0, 1]
    assert list(st["big"]) == [32, 16] and list(st["negative"]) == [32, 16]
    assert list(st["max_scale"]) == [4.0, 2.0]
    # per record: 16 entries of (0.5 s)^2 and 16 of (1.5 s)^2 = 16 * 2.5 * s^2 = 40 s^2
    assert st["sumsq"][0] == 40 * 4.0 + 40 * 16.0 and st["sumsq"][1] == 40 * 4.0
    # with k = 128 the check covers every entry: a swap at entries 100 and 101
    codec = (4096, 128, MAX)
    idx = np.arange(0, 256, 2, dtype=np.uint16)[None]
    codes = np.zeros((1, 128), np.uint8)
    idx[0, [100, 101]] = idx[0, [101, 100]]
    _, flags = oracle.decode_aggregate([oracle.pack(idx, codes, codec)], [np.ones(1, np.float32)],
                                       4096, codec=codec)
    assert flags == oracle.FLAG_BAD_RECORD


def test_default_codec_argument_is_the_default_codec():
    rng = np.random.default_rng(5)
    n = 3 * 4096 + 9
    delta = rng.laplace(0, 1, n).astype(np.float32)
    e1 = rng.laplace(0, 1, n).astype(np.float32)
    e2 = e1.copy()
    p1, s1, _ = oracle.ef_compress(delta, e1, 0.9)
    p2, s2, _ = oracle.ef_compress(delta, e2, 0.9, codec=(4096, 64, MAX))
    assert np.array_equal(p1, p2) and np.array_equal(s1, s2) and np.array_equal(e1, e2)
