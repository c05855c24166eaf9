"""Comparison rules between the CUDA path and the oracle.

Floating point (bf16 inputs, fp32 accumulation on the GPU, fp64 in the
oracle):
  * block scores: |s_gpu - s_ref| <= 1e-2 |s_ref| + 1e-3 rms(row of s_ref)
    (the absolute floor is needed because ReLU produces exact zeros);
  * selected sets: identical, except that a block in the symmetric difference
    must score within 1e-2 (relative) of the oracle's (budget-1)-th best
    score of that row -- a near-tie the two arithmetics may break differently;
  * attention outputs, compared on one and the same selection (the GPU's):
    |O_gpu - O_ref| <= 2e-2 + 1e-2 |O_ref|, and the same for the log-sum-exp.
Integer work (block keys, row layout of idx) is compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

SCORE_RTOL, SCORE_ATOL_RMS = 1e-2, 1e-3
SET_RTOL = 1e-2
OUT_ATOL, OUT_RTOL = 2e-2, 1e-2


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_scores(gpu: np.ndarray, ref: np.ndarray):
    valid = ~np.isnan(ref)
    assert np.array_equal(valid, ~np.isnan(gpu)), "score masks differ"
    r = np.where(valid, ref, 0.0)
    g = np.where(valid, gpu, 0.0)
    cnt = np.maximum(valid.sum(axis=1, keepdims=True), 1)
    rms = np.sqrt((r * r).sum(axis=1, keepdims=True) / cnt)
    err = np.abs(g - r)
    tol = SCORE_RTOL * np.abs(r) + SCORE_ATOL_RMS * rms
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} scores out of tolerance; worst {err[bad].max()}"


def check_row_format(idx_row: np.ndarray, t: int, budget: int):
    """Ascending past blocks, then the current block, then -1 padding."""
    c = t // 4
    n = min(budget, c + 1)
    assert np.all(idx_row[n:] == -1), (t, idx_row)
    sel = idx_row[:n]
    assert sel[-1] == c, (t, sel[-5:])
    assert np.all(np.diff(sel) > 0), (t, "not strictly ascending")
    assert sel[0] >= 0


def check_selection(idx_gpu: np.ndarray, idx_ref: np.ndarray, score_rows: np.ndarray, rows, budget: int):
    """idx_* [nrows, budget]; score_rows [nrows, nb] oracle scores (NaN where b >= c)."""
    nmis = 0
    for r, t in enumerate(rows):
        t = int(t)
        check_row_format(idx_gpu[r], t, budget)
        a = set(int(b) for b in idx_gpu[r] if b >= 0)
        b_ = set(int(b) for b in idx_ref[r] if b >= 0)
        if a == b_:
            continue
        c = t // 4
        s = score_rows[r, :c]
        kth = np.sort(s)[::-1][budget - 2]
        for blk in a ^ b_:
            assert blk != c
            assert abs(s[blk] - kth) <= SET_RTOL * abs(kth) + 1e-9, (t, blk, s[blk], kth)
            nmis += 1
    return nmis


def check_outputs(o_gpu: np.ndarray, o_ref: np.ndarray, what: str = "O"):
    err = np.abs(o_gpu - o_ref)
    tol = OUT_ATOL + OUT_RTOL * np.abs(o_ref)
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} out of tolerance; worst {err.max()}"


def sample_rows(L: int, n: int, seed: int = 0, extra=()) -> np.ndarray:
    """Seeded row sample: the first and last 16 rows, rows around the points
    where the budget starts to bind, and n uniform rows."""
    rng = np.random.default_rng(seed)
    base = set(range(min(16, L))) | set(range(max(0, L - 16), L))
    for edge in (2044, 2048, 2052):
        if edge < L:
            base.add(edge)
    base |= set(int(x) for x in extra if 0 <= x < L)
    base |= set(int(x) for x in rng.integers(0, L, size=n))
    return np.array(sorted(base), dtype=np.int64)


def check_rope(got_bits, ref_bits, x_bits):
    """RoPE'd keys: the GPU rotates in fp32 (angle reduced in fp64), the
    oracle in fp64, both then round to bf16.  Allowed: one bf16 ulp of the
    result (2^-7 relative) plus the fp32 rounding error of the rotation, which
    dominates when x1 cos a and x2 sin a nearly cancel."""
    g = \
        torch.from_numpy(got_bits[..., :64].astype(np.int32) << 16).view(torch.float32).double().numpy()
    r = torch.from_numpy(ref_bits[..., :64].astype(np.int32) << 16).view(torch.float32).double().numpy()
    x = torch.from_numpy(x_bits[..., :64].astype(np.int32) << 16).view(torch.float32).double().numpy()
    mag = np.abs(x[..., :32]) + np.abs(x[..., 32:])
    mag = np.concatenate([mag, mag], axis=-1)
    bound = 2.0 ** -7 * np.abs(r) + 2.0 ** -20 * mag
    assert np.all(np.abs(g - r) <= bound), float(np.max(np.abs(g - r) - bound))
    assert np.mean(got_bits[..., :64] != ref_bits[..., :64]) < 1e-3
