"""Helpers for the GPU parity tests: host copies, bit comparisons and sampled-chunk checks.

The oracle runs on host copies of exactly the bytes the GPU consumed.  At full workload sizes
only sampled chunks are checked: chunks are independent, so running the oracle on the
concatenation of the sampled chunks' inputs reproduces those chunks' outputs.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

CHUNK = 4096
TOL = 1e-6   # max-abs error normalised by max |reference|, for the mean and theta


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.detach().cpu().numpy()


def bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a).view(np.uint32 if a.dtype == np.float32 else np.uint8)


def assert_bit_equal(got: np.ndarray, ref: np.ndarray, what: str):
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    g, r = bits(got), bits(ref)
    if not np.array_equal(g, r):
        bad = np.flatnonzero((g != r).reshape(-1))
        raise AssertionError(f"{what}: {bad.size} of {g.size} differ, first at {bad[:8].tolist()}")


def assert_close(got: np.ndarray, ref: np.ndarray, what: str, tol: float = TOL):
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    err = float(np.abs(got.astype(np.float64) - ref.astype(np.float64)).max()) if ref.size else 0.0
    assert err <= tol * max(scale, np.finfo(np.float32).tiny), \
        f"{what}: max err {err:.3e} > {tol:g} x {scale:.3e}"


def sample_chunks(C: int, k: int, seed: int) -> np.ndarray:
    """First, last and k random chunk ids (sorted, unique)."""
    rng = np.random.default_rng(seed)
    ids = set(rng.choice(C, size=min(k, C), replace=False).tolist()) | {0, C - 1}
    return np.array(sorted(ids), dtype=np.int64)


def gather_chunks(x: torch.Tensor, ids: np.ndarray, n: int):
    """Host copy of the chunks `ids` of a flat tensor: (full chunks concatenated, tail or None)."""
    full_ids = [c for c in ids.tolist() if (c + 1) * CHUNK <= n]
    tail = None
    if full_ids:
        idx = (torch.tensor(full_ids, device=x.device)[:, None] * CHUNK +
               torch.arange(CHUNK, device=x.device)[None, :]).reshape(-1)
        body = host(x[idx])
    else:
        body = host(x[:0])
    last = ids[-1]
    if (last + 1) * CHUNK > n:
        tail = host(x[last * CHUNK:n])
    return body, tail, full_ids


def check_compress_sampled(run, delta: torch.Tensor, ef: torch.Tensor, beta: float,
                           ids: np.ndarray, what: str):
    """Snapshot the sampled chunks, call run() (the GPU round returning payload, scales),
    and compare those chunks with the oracle bit for bit."""
    n = delta.numel()
    bf16 = delta.dtype == torch.bfloat16
    d_body, d_tail, full_ids = gather_chunks(delta, ids, n)
    e_body, e_tail, _ = gather_chunks(ef, ids, n)
    payload, scales = run()
    torch.cuda.synchronize()
    e_after_body, e_after_tail, _ = gather_chunks(ef, ids, n)
    pl = host(payload)
    sc = host(scales)
    if full_ids:
        o_pl, o_sc, _ = oracle.ef_compress(d_body, e_body, beta, bf16=bf16)
        assert_bit_equal(pl[full_ids], o_pl, f"{what}: payload")
        assert_bit_equal(sc[full_ids], o_sc, f"{what}: scales")
        assert_bit_equal(e_after_body, e_body, f"{what}: error buffer")
    if d_tail is not None:
        o_pl, o_sc, _ = oracle.ef_compress(d_tail, e_tail, beta, bf16=bf16)
        assert_bit_equal(pl[ids[-1:]], o_pl, f"{what}: tail payload")
        assert_bit_equal(sc[ids[-1:]], o_sc, f"{what}: tail scale")
        assert_bit_equal(e_after_tail, e_tail, f"{what}: tail error buffer")
    return payload, scales


def check_decode_sampled(payloads, scales, n: int, mean: torch.Tensor, theta_before,
                         theta_after, lr: float, ids: np.ndarray, what: str):
    """Compare sampled chunks of a GPU decode (mean, theta) with the oracle on those chunks."""
    full_ids = [c for c in ids.tolist() if (c + 1) * CHUNK <= n]
    has_tail = (ids[-1] + 1) * CHUNK > n
    groups = [(full_ids, len(full_ids) * CHUNK)]
    if has_tail:
        groups.append(([int(ids[-1])], n - int(ids[-1]) * CHUNK))
    m_body, m_tail, _ = gather_chunks(mean, ids, n)
    t_after = gather_chunks(theta_after, ids, n) if theta_after is not None else None
    for gi, (cids, nn) in enumerate(groups):
        if not cids:
            continue
        sel = torch.tensor(cids, device=payloads[0].device)
        pl = [host(p[sel]) for p in payloads]
        sc = [host(s[sel]) for s in scales]
        th = None
        if theta_before is not None:
            th = (theta_before[0] if gi == 0 else theta_before[1]).copy()
        o_mean, _ = oracle.decode_aggregate(pl, sc, nn, theta=th, lr=lr)
        got = m_body if gi == 0 else m_tail
        assert_close(got, o_mean, f"{what}: mean")
        if th is not None:
            got_t = t_after[0] if gi == 0 else t_after[1]
            assert_close(got_t, th, f"{what}: theta")
