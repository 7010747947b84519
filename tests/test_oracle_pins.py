"""Pins of the CPU oracle to facts fixed outside the oracle itself (CPU only).

Every check here compares the oracle against something it does not compute: a figure the
pages print (tests/golden/page_figures.txt), hand-derived bytes (tests/golden/
pack_known_answer.txt), a characterisation checked by exhaustive enumeration, a library
sort, exact rational arithmetic, or an invariant of the method.  A dropped term, a wrong
sign, a swapped sub-field or a wrong tie rule in the oracle fails at least one of them.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def _figures():
    out = {}
    with open(os.path.join(GOLDEN, "page_figures.txt")) as f:
        for line in f:
            line = line.split(";")[0].strip()
            if line and not line.startswith("#"):
                k, v = (t.strip() for t in line.split("="))
                out[k] = float(v)
    return out


def _decode_dense(payload, scales, n):
    """Dense vector of one peer's decoded values (test-side placement via unpack)."""
    idx, codes = oracle.unpack(payload)
    C = idx.shape[0]
    out = np.zeros(C * 4096, dtype=np.float32)
    for c in range(C):
        for r in range(64):
            out[c * 4096 + int(idx[c, r])] = oracle.level(int(codes[c, r]), float(scales[c]))
    return out[:n]


def _nearest_f32(x: Fraction) -> np.float32:
    """Round an exact rational to the nearest fp32 (ties to even), by exhaustive neighbour check."""
    f = F32(float(x))  # within one fp32 ulp of the answer
    cands = [np.nextafter(f, F32(-np.inf)), f, np.nextafter(f, F32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - x),
                                     int(np.frombuffer(F32(c).tobytes(), np.uint32)[0]) & 1))
    return F32(best)


# ---------------------------------------------------------------------------------------------
# Sizes and figures the pages print
# ---------------------------------------------------------------------------------------------
def test_constants_match_page_figures():
    fig = _figures()
    k = oracle.constants()
    assert k["chunk"] == fig["chunk"]
    assert k["topk"] == fig["topk"]
    assert k["record_bytes"] == fig["bytes_per_chunk"]
    assert k["record_bytes"] * 8 == fig["bits_per_chunk"]
    assert fig["topk"] * (fig["value_bits"] + fig["index_bits"]) == fig["bits_per_chunk"]
    assert 2 ** fig["index_bits"] == fig["chunk"]
    assert fig["chunk"] * 4 == fig["dense_bytes_per_chunk"]
    assert round(fig["dense_bytes_per_chunk"] / k["record_bytes"], 1) == fig["compression_ratio"]


def test_oracle_output_sizes_and_density_match_pages():
    fig = _figures()
    rng = np.random.default_rng(1)
    n = 3 * 4096
    delta = rng.standard_normal(n).astype(np.float32)
    ef = np.zeros(n, np.float32)
    payload, scales, flags = oracle.ef_compress(delta, ef, 1.0)
    assert flags == 0
    assert payload.shape == (3, fig["bytes_per_chunk"])
    dense = _decode_dense(payload, scales, n)
    nnz_per_chunk = (dense.reshape(3, 4096) != 0).sum(axis=1)
    assert (nnz_per_chunk == fig["topk"]).all()
    density = 100.0 * nnz_per_chunk[0] / 4096
    assert density == fig["density_percent"]
    assert round(100.0 - density, 2) == fig["dropped_percent"]


def test_per_peer_payload_arithmetic_matches_pages():
    fig = _figures()
    params = int(fig["params"])
    chunks = oracle.num_chunks(params)
    payload_bytes = chunks * oracle.constants()["record_bytes"]
    assert abs(payload_bytes / 1e9 - fig["payload_per_peer_gb"]) < 0.05       # about 2 GB per peer
    mbps = payload_bytes * 8 / fig["window_seconds"] / 1e6
    assert round(mbps) == fig["uplink_mbps_per_peer"]                           # about 13 Mbps
    assert round(4 * 72.7e9 / 1e9, 1) == fig["dense_fp32_gb"]


# ---------------------------------------------------------------------------------------------
# Top-k selection
# ---------------------------------------------------------------------------------------------
def _rank_key(v, i):
    """Larger is better: NaN above all numbers, then |v|, then the lower index."""
    return (1 if math.isnan(v) else 0, 0.0 if math.isnan(v) else abs(v), -i)


@pytest.mark.parametrize("L,k", [(1, 1), (5, 2), (8, 3), (10, 4), (12, 4), (6, 6)])
def test_topk_matches_exhaustive_enumeration(L, k):
    rng = np.random.default_rng(L * 100 + k)
    for trial in range(40):
        # small integers: many exact ties in magnitude, both signs, signed zeros
        a = rng.integers(-3, 4, size=L).astype(np.float32)
        a[rng.random(L) < 0.15] = -0.0
        if trial % 7 == 3:
            a[rng.integers(L)] = np.nan
        got, _ = oracle.topk_select(a, k)
        keys = [_rank_key(float(a[i]), i) for i in range(L)]
        winners = [S for S in itertools.combinations(range(L), k)
                   if all(keys[i] > keys[j] for i in S for j in range(L) if j not in S)]
        assert len(winners) == 1
        assert list(got) == list(winners[0])


def test_topk_matches_library_sort_full_chunk():
    rng = np.random.default_rng(7)
    for trial in range(20):
        a = rng.standard_normal(4096).astype(np.float32)
        if trial % 2:
            a = np.round(a * 4) / 4  # heavy ties
        order = np.lexsort((np.arange(4096), -np.abs(a).astype(np.float64)))
        got, top = oracle.topk_select(a, 64)
        assert list(got) == sorted(order[:64].tolist())
        assert top == order[0]


def test_topk_closed_cases():
    got, _ = oracle.topk_select(np.full(4096, -2.5, np.float32), 64)
    assert list(got) == list(range(64))                     # all equal: lowest indices
    got, _ = oracle.topk_select(np.arange(4096, dtype=np.float32) * -1.0, 64)
    assert list(got) == list(range(4032, 4096))             # |a| increasing in j
    got, _ = oracle.topk_select(np.zeros(4096, np.float32), 64)
    assert list(got) == list(range(64))                     # all zero
    rng = np.random.default_rng(3)
    spikes = np.sort(rng.choice(4096, 64, replace=False))
    a = (rng.standard_normal(4096) * 1e-3).astype(np.float32)
    a[spikes] = rng.choice([-1.0, 1.0], 64) * (1.0 + rng.random(64))
    got, _ = oracle.topk_select(a, 64)
    assert list(got) == spikes.tolist()                     # planted spikes


# ---------------------------------------------------------------------------------------------
# Quantiser, residual and the compress step on hand-built chunks
# ---------------------------------------------------------------------------------------------
def test_quantiser_closed_cases():
    s = oracle.scale(1.5)
    assert s == F32(1.0)
    assert oracle.code(1.0, s) == 0                         # exactly at s: smaller level
    assert oracle.code(float(np.nextafter(F32(1), F32(2))), s) == 1
    assert oracle.code(-1.5, s) == 3 and oracle.level(3, s) == F32(-1.5)
    assert oracle.code(0.25, s) == 0 and oracle.level(0, s) == F32(0.5)
    assert oracle.code(-0.75, s) == 2 and oracle.level(2, s) == F32(-0.5)
    assert oracle.code(-0.0, s) == 0                        # -0.0 codes as positive
    assert oracle.level(1, s) == F32(1.5)
    assert oracle.scale(3.0) == F32(2.0)
    assert oracle.scale(1.0) == F32(1.0) / F32(1.5)


def test_compress_planted_chunk_by_hand():
    pos = np.array([7 + 61 * r for r in range(64)])
    special = {0: 1.5, 1: 1.0, 2: float(np.nextafter(F32(1), F32(2))), 3: -1.5, 4: 0.25, 5: -0.75}
    rng = np.random.default_rng(11)
    vals = (rng.choice([-1, 1], 64) * (0.1 + 1.3 * rng.random(64))).astype(np.float32)
    for r, v in special.items():
        vals[r] = v
    delta = np.zeros(4096, np.float32)
    delta[pos] = vals
    ef = np.zeros(4096, np.float32)
    payload, scales, flags = oracle.ef_compress(delta, ef, 1.0)
    assert flags == 0 and scales[0] == F32(1.0)
    idx, codes = oracle.unpack(payload)
    assert idx[0].tolist() == pos.tolist()
    expect_codes = {0: 1, 1: 0, 2: 1, 3: 3, 4: 0, 5: 2}
    expect_resid = {0: 0.0, 1: 0.5, 2: float(np.nextafter(F32(1), F32(2))) - 1.5, 3: 0.0,
                    4: -0.25, 5: -0.25}
    for r in expect_codes:
        assert codes[0, r] == expect_codes[r]
        assert ef[pos[r]] == F32(expect_resid[r])
    for r in range(64):                                     # generic entries: rule restated
        v = vals[r]
        c = (2 if v < 0 else 0) | (1 if abs(v) > 1.0 else 0)
        assert codes[0, r] == c
    mask = np.ones(4096, bool)
    mask[pos] = False
    assert (ef[mask] == 0).all()


def test_all_zero_chunk_and_negative_zero():
    for z in (0.0, -0.0):
        delta = np.full(4096, z, np.float32)
        ef = np.zeros(4096, np.float32)
        payload, scales, _ = oracle.ef_compress(delta, ef, 1.0)
        idx, codes = oracle.unpack(payload)
        assert idx[0].tolist() == list(range(64))
        assert (codes == 0).all() and scales[0] == 0.0
        assert (ef == 0).all()


def test_selected_zeros_take_the_small_positive_level():
    delta = np.zeros(4096, np.float32)
    delta[[100, 200, 3000]] = [0.3, -3.0, 1.2]
    ef = np.zeros(4096, np.float32)
    payload, scales, _ = oracle.ef_compress(delta, ef, 1.0)
    s = scales[0]
    assert s == F32(3.0) / F32(1.5)
    idx, codes = oracle.unpack(payload)
    expect = sorted(set(range(61)) | {100, 200, 3000})[:64]
    assert idx[0].tolist() == expect
    zeros = [r for r in range(64) if idx[0, r] not in (100, 200, 3000)]
    assert all(codes[0, r] == 0 for r in zeros)
    assert all(ef[idx[0, r]] == -F32(0.5) * s for r in zeros)


def test_tail_chunk_pads_lose_ties_and_are_not_stored():
    n = 4096 + 10
    rng = np.random.default_rng(5)
    delta = rng.standard_normal(n).astype(np.float32)
    ef_full = np.zeros(n, np.float32)
    payload, scales, _ = oracle.ef_compress(delta, ef_full, 1.0)
    idx, codes = oracle.unpack(payload)
    assert idx[1].tolist() == list(range(64))   # 10 real entries + pads 10..63
    assert (codes[1, 10:] == 0).all()
    # the tail chunk alone gives the same record: chunks are independent
    ef_tail = np.zeros(10, np.float32)
    p2, s2, _ = oracle.ef_compress(delta[4096:], ef_tail, 1.0)
    assert (p2[0] == payload[1]).all() and s2[0] == scales[1]
    assert (ef_tail == ef_full[4096:]).all()
    # pads are dropped on decode
    mean, _ = oracle.decode_aggregate([payload], [scales], n)
    assert np.count_nonzero(mean[4096:]) == 10


def test_tail_chunk_real_zeros_win_ties_against_pads():
    """A tail chunk of 100 real values, only 10 of them nonzero: the 64 chosen are the 10
    nonzero values and the real zeros at the lowest indices; the pads (zeros past n, with
    larger indices) lose every tie to them."""
    n = 4096 + 100
    delta = np.zeros(n, np.float32)
    nz = 4096 + np.array([3, 9, 17, 30, 44, 51, 66, 70, 88, 99])
    delta[nz] = np.arange(1, 11, dtype=np.float32)
    delta[:4096] = 1.0
    ef = np.zeros(n, np.float32)
    payload, scales, _ = oracle.ef_compress(delta, ef, 1.0)
    idx, codes = oracle.unpack(payload)
    zeros = [j for j in range(100) if j + 4096 not in set(nz.tolist())][:54]
    assert idx[1].tolist() == sorted(zeros + (nz - 4096).tolist())
    assert idx[1].max() < 100
    s = F32(10.0) / F32(1.5)
    assert scales[1] == s
    assert all(ef[4096 + j] == -F32(0.5) * s for j in zeros)


@pytest.mark.parametrize("beta", [1.0, 0.5])
def test_ef_conservation_exact_betas(beta):
    """e_new = a off the chosen set and e_new = RN(a - q) on it, with a = RN(beta*e + delta)."""
    rng = np.random.default_rng(int(beta * 10))
    n = 4 * 4096 + 123
    delta = (rng.laplace(size=n) * 1e-4).astype(np.float32)
    ef0 = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    ef = ef0.copy()
    payload, scales, _ = oracle.ef_compress(delta, ef, beta)
    a = (F32(beta) * ef0) + delta                # beta*e is exact for beta in {1, 0.5}
    q = _decode_dense(payload, scales, n)
    chosen = np.zeros(n, bool)
    idx, _ = oracle.unpack(payload)
    for c in range(idx.shape[0]):
        gi = c * 4096 + idx[c].astype(np.int64)
        chosen[gi[gi < n]] = True
    assert (ef[~chosen] == a[~chosen]).all()
    assert (ef[chosen] == (a - q)[chosen]).all()
    # chosen set = library-sort top-64 of |a| per chunk (pads as zeros)
    ap = np.zeros(idx.shape[0] * 4096, np.float32)
    ap[:n] = a
    for c in range(idx.shape[0]):
        blk = ap[c * 4096:(c + 1) * 4096]
        order = np.lexsort((np.arange(4096), -np.abs(blk).astype(np.float64)))
        assert sorted(order[:64].tolist()) == idx[c].tolist()
        assert scales[c] == F32(np.abs(blk).max()) / F32(1.5)


def test_ef_accumulate_is_one_correctly_rounded_fma():
    rng = np.random.default_rng(9)
    n = 4096
    beta = 0.95
    delta = (rng.laplace(size=n) * 1e-4).astype(np.float32)
    ef0 = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    ef = ef0.copy()
    payload, _, _ = oracle.ef_compress(delta, ef, beta)
    chosen = set(oracle.unpack(payload)[0][0].tolist())
    b = Fraction(float(F32(beta)))
    for i in range(0, n, 7):
        if i in chosen:
            continue
        exact = b * Fraction(float(ef0[i])) + Fraction(float(delta[i]))
        assert ef[i] == _nearest_f32(exact), i


def test_bf16_delta_is_widened_exactly():
    rng = np.random.default_rng(4)
    n = 4096
    f = rng.standard_normal(n).astype(np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)          # truncate to bf16
    widened = (bits.astype(np.uint32) << 16).view(np.float32)
    ef_a = np.zeros(n, np.float32)
    ef_b = np.zeros(n, np.float32)
    pa, sa, _ = oracle.ef_compress(bits, ef_a, 1.0, bf16=True)
    pb, sb, _ = oracle.ef_compress(widened, ef_b, 1.0)
    assert (pa == pb).all() and (sa == sb).all() and (ef_a == ef_b).all()


def test_nonfinite_flag():
    delta = np.zeros(8192, np.float32)
    delta[5000] = np.inf
    ef = np.zeros(8192, np.float32)
    _, _, flags = oracle.ef_compress(delta, ef, 1.0)
    assert flags & oracle.FLAG_NONFINITE
    delta[5000] = np.nan
    ef[:] = 0
    payload, _, flags = oracle.ef_compress(delta, ef, 1.0)
    assert flags & oracle.FLAG_NONFINITE
    idx, _ = oracle.unpack(payload)
    assert 5000 - 4096 in idx[1].tolist()                      # NaN ranks first


def test_nan_ranks_above_every_number():
    """NaNs (any payload) rank first, equal among themselves, then index order decides."""
    a = np.arange(4096, dtype=np.float32) - 2048.0
    nan_pos = [5, 4000, 4001, 4090]
    a[nan_pos] = np.nan
    a[4001] = -np.float32(np.nan)
    mag = np.where(np.isnan(a), np.inf, np.abs(a)).astype(np.float64)
    order = np.lexsort((np.arange(4096), -mag))
    got, top = oracle.topk_select(a, 64)
    assert list(got) == sorted(order[:64].tolist())
    assert set(nan_pos) <= set(got.tolist()) and top == 5
    for start in range(0, 4096, 512):                        # NaN in every position class
        b = np.arange(4096, dtype=np.float32)
        b[start + 7] = np.nan
        got, top = oracle.topk_select(b, 64)
        assert top == start + 7 and start + 7 in got.tolist()


# ---------------------------------------------------------------------------------------------
# Record layout
# ---------------------------------------------------------------------------------------------
def _golden_bytes(key):
    with open(os.path.join(GOLDEN, "pack_known_answer.txt")) as f:
        for line in f:
            if line.startswith(key):
                return bytes(int(t, 16) for t in line.split("=")[1].split())
    raise KeyError(key)


def test_pack_known_answer_bytes():
    idx = np.arange(64, dtype=np.uint16)[None]
    codes = np.zeros((1, 64), np.uint8)
    assert bytes(oracle.pack(idx, codes)[0][:13]) == _golden_bytes("A_first13")
    idx = np.zeros((1, 64), np.uint16)
    codes = np.zeros((1, 64), np.uint8)
    idx[0, 63], codes[0, 63] = 4095, 3
    rec = bytes(oracle.pack(idx, codes)[0])
    assert rec[-2:] == _golden_bytes("B_last2") and not any(rec[:-2])


def test_pack_matches_big_integer_definition_and_round_trips():
    rng = np.random.default_rng(2)
    C = 50
    idx = np.sort(np.stack([rng.choice(4096, 64, replace=False) for _ in range(C)]), axis=1)
    idx = idx.astype(np.uint16)
    codes = rng.integers(0, 4, size=(C, 64)).astype(np.uint8)
    payload = oracle.pack(idx, codes)
    for c in range(C):
        big = sum((int(codes[c, r]) | int(idx[c, r]) << 2) << (14 * r) for r in range(64))
        assert bytes(payload[c]) == big.to_bytes(112, "little")
    i2, c2 = oracle.unpack(payload)
    assert (i2 == idx).all() and (c2 == codes).all()


# ---------------------------------------------------------------------------------------------
# Error feedback over rounds
# ---------------------------------------------------------------------------------------------
def test_beta_one_telescopes():
    """With beta = 1: sum_t decode_t + e_T = sum_t delta_t, up to per-round rounding."""
    rng = np.random.default_rng(12)
    n, T = 2 * 4096 + 77, 6
    ef = np.zeros(n, np.float32)
    sent = np.zeros(n, np.float64)
    total = np.zeros(n, np.float64)
    bound = 0.0
    for _ in range(T):
        d = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        payload, scales, _ = oracle.ef_compress(d, ef, 1.0)
        sent += _decode_dense(payload, scales, n)
        total += d
        bound += 2 * np.abs(ef).max() * 2.0 ** -23 + 2 * np.abs(d).max() * 2.0 ** -23
    assert np.abs(sent + ef - total).max() <= bound


def test_every_coordinate_eventually_transmitted():
    """One-shot delta, then zero rounds with beta = 1: the error buffer's max never grows,
    every nonzero coordinate gets sent, and what was sent converges to delta."""
    rng = np.random.default_rng(13)
    n = 2 * 4096
    d0 = rng.standard_normal(n).astype(np.float32)
    ef = np.zeros(n, np.float32)
    ever = np.zeros(n, bool)
    sent = np.zeros(n, np.float64)
    prev_max = np.inf
    zeros = np.zeros(n, np.float32)
    for t in range(400):
        payload, scales, _ = oracle.ef_compress(d0 if t == 0 else zeros, ef, 1.0)
        q = _decode_dense(payload, scales, n)
        ever |= q != 0
        sent += q
        m = np.abs(ef).max()
        assert m <= prev_max
        prev_max = m
    assert ever.all()
    assert np.abs(sent - d0).max() <= 1e-3 * np.abs(d0).max()


# ---------------------------------------------------------------------------------------------
# Decode and aggregation
# ---------------------------------------------------------------------------------------------
def _peer(seed, n, beta=1.0):
    rng = np.random.default_rng(seed)
    d = (rng.laplace(size=n) * 1e-4).astype(np.float32)
    ef = np.zeros(n, np.float32)
    payload, scales, _ = oracle.ef_compress(d, ef, beta)
    return payload, scales


def test_single_peer_mean_is_the_decode():
    n = 3 * 4096 + 500
    p, s = _peer(21, n)
    mean, flags = oracle.decode_aggregate([p], [s], n)
    assert flags == 0
    assert (mean == _decode_dense(p, s, n)).all()


def test_disjoint_peers_give_quarter_values():
    n = 4096
    payloads, scales, dense = [], [], []
    for p in range(4):
        d = np.zeros(n, np.float32)
        pos = np.arange(p, 4096, 4)[:64]
        d[pos] = np.linspace(0.5, 2.0, 64, dtype=np.float32) * (-1) ** p
        ef = np.zeros(n, np.float32)
        pl, sc, _ = oracle.ef_compress(d, ef, 1.0)
        payloads.append(pl)
        scales.append(sc)
        dense.append(_decode_dense(pl, sc, n))
    mean, _ = oracle.decode_aggregate(payloads, scales, n)
    assert (mean == sum(dense) / F32(4)).all()
    assert np.count_nonzero(mean) == 256


def test_sign_flipped_peer_cancels_and_identical_peers_agree():
    n = 2 * 4096
    p, s = _peer(31, n)
    idx, codes = oracle.unpack(p)
    flipped = oracle.pack(idx, codes ^ 2)
    mean, _ = oracle.decode_aggregate([p, flipped], [s, s], n)
    assert (mean == 0).all()
    mean, _ = oracle.decode_aggregate([p, p], [s, s], n)
    assert (mean == _decode_dense(p, s, n)).all()


def test_general_mean_within_tolerance_of_exact_sum():
    n = 5 * 4096 + 1
    peers = [_peer(40 + p, n) for p in range(8)]
    mean, _ = oracle.decode_aggregate([p for p, _ in peers], [s for _, s in peers], n)
    ref = sum(_decode_dense(p, s, n).astype(np.float64) for p, s in peers) / 8
    assert np.abs(mean - ref).max() <= 1e-6 * np.abs(ref).max()


def test_outer_step_is_one_fma():
    n = 4096
    p, s = _peer(50, n)
    rng = np.random.default_rng(51)
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    theta = theta0.copy()
    mean, _ = oracle.decode_aggregate([p], [s], n, theta=theta, lr=0.7)
    lr = Fraction(float(F32(0.7)))
    for i in range(0, n, 5):
        exact = Fraction(float(theta0[i])) - lr * Fraction(float(mean[i]))
        assert theta[i] == _nearest_f32(exact)


def test_malformed_records_are_rejected():
    n = 4096
    p0, s0 = _peer(60, n)
    p1, s1 = _peer(61, n)
    idx, codes = oracle.unpack(p1)
    bad_idx = idx.copy()
    bad_idx[0, [10, 11]] = bad_idx[0, [11, 10]]                  # not ascending
    dup_idx = idx.copy()
    dup_idx[0, 11] = dup_idx[0, 10]                              # duplicate
    good = _decode_dense(p0, s0, n) / F32(2)
    for bad in (oracle.pack(bad_idx, codes), oracle.pack(dup_idx, codes)):
        mean, flags = oracle.decode_aggregate([p0, bad], [s0, s1], n)
        assert flags & oracle.FLAG_BAD_RECORD
        assert (mean == good).all()
    for bad_s in (np.nan, np.inf, -1.0):
        mean, flags = oracle.decode_aggregate([p0, p1], [s0, np.array([bad_s], np.float32)], n)
        assert flags & oracle.FLAG_BAD_RECORD
        assert (mean == good).all()


# ---------------------------------------------------------------------------------------------
# Receiver statistics per peer
# ---------------------------------------------------------------------------------------------
def test_peer_stats_by_hand():
    """A chunk with 64 planted values and scale 1: counts and sum of squares by hand."""
    pos = np.array([7 + 61 * r for r in range(64)])
    vals = np.full(64, 0.75, np.float32)            # |v| <= s: code 0, q = 0.5
    vals[:10] = 1.5                                  # max: code 1, q = 1.5 (s = 1)
    vals[10:14] = -1.25                              # code 3, q = -1.5
    vals[14:20] = -0.5                               # code 2, q = -0.5
    delta = np.zeros(4096, np.float32)
    delta[pos] = vals
    pl, sc, _ = oracle.ef_compress(delta, np.zeros(4096, np.float32), 1.0)
    assert sc[0] == F32(1.0)
    bad_idx, bad_codes = oracle.unpack(pl)
    bad_idx[0, [0, 1]] = bad_idx[0, [1, 0]]
    bad = oracle.pack(bad_idx, bad_codes)
    st = oracle.peer_stats([pl, bad, pl], [sc, sc, np.array([np.nan], np.float32)], 4096)
    assert st["rejected"].tolist() == [0, 1, 1]
    assert st["big"].tolist() == [14, 0, 0]
    assert st["negative"].tolist() == [10, 0, 0]
    assert st["max_scale"].tolist() == [1.0, 0.0, 0.0]
    assert st["sumsq"][0] == 14 * 2.25 + 50 * 0.25
    assert st["sumsq"][1] == 0.0


def test_peer_stats_sum_of_squares_is_the_decode_norm():
    n = 6 * 4096 + 10
    payloads, scales = [], []
    for seed in (70, 71, 72):
        p, s = _peer(seed, n)
        payloads.append(p)
        scales.append(s)
    st = oracle.peer_stats(payloads, scales, n)
    for k, (p, s) in enumerate(zip(payloads, scales)):
        idx, codes = oracle.unpack(p)
        # every entry of the record, pads included, as placed by a dense decode of a padded tensor
        q = np.array([oracle.level(int(c), float(s[ch])) for ch in range(idx.shape[0])
                      for c in codes[ch]], np.float64)
        assert st["sumsq"][k] == pytest.approx(float(np.sum(q * q)), rel=1e-12)
        assert st["big"][k] == int((codes & 1).sum())
        assert st["negative"][k] == int((codes >> 1).sum())
        assert st["max_scale"][k] == s.max()
