"""Comparison helpers for the GPU parity tests (no arithmetic of the method)."""
from __future__ import annotations

import numpy as np

MAX_ABS = 2e-2    # max-abs tolerance for outputs and gradients (fp32 accumulate, bf16 inputs)
MEAN_ABS = 2e-3   # mean-abs tolerance
# The fine forward's log-sum-exp.  The row sum l adds the n = 64 K softmax
# weights exp2(s - m) rounded to fp16 (the operand the P.V product uses);
# every weight is <= 256 and the largest is >= 1, so l >= 1, and a rounding
# errs by at most 2^-11 of the weight (fp16 normal range) or by 2^-25
# (below it).  Hence |log l - log l_exact| <= 2^-11 + n 2^-25 even if every
# rounding went the same way.  S is an fp32 sum of exact products of the
# 16-bit operands, and exp2 is the hardware approximation (relative error
# ~2^-22): 1e-4 covers both.  Mean-abs 1e-4.
LSE_MEAN_ABS = 1e-4


def lse_max_abs(keys: int) -> float:
    """Max-abs bound on the fine LSE of a row that attends to `keys` keys."""
    return 2.0 ** -11 + keys * 2.0 ** -25 + 1e-4


LSE_MAX_ABS = lse_max_abs(64 * 16)   # the unit tests' lists: at most 16 cubes (6.2e-4)


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half a unit in the last place of bf16 (8 significant bits) at |x|."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.exp2(e - 8)


def round_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def assert_close(gpu, ref, bf16_out: bool = False, max_abs: float = MAX_ABS, mean_abs: float = MEAN_ABS,
                 what: str = ""):
    """Element-by-element parity.  For bf16 outputs the bound applies beyond the
    output format's own rounding (half an ulp at the reference value); the
    mean is taken against the reference rounded to bf16."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite values"
    diff = np.abs(gpu - ref)
    if bf16_out:
        excess = diff - half_ulp_bf16(ref)
        mean = np.abs(gpu - round_bf16(ref)).mean()
    else:
        excess = diff
        mean = diff.mean()
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= max_abs, f"{what}: max-abs {excess.max():.3e} at {worst} (gpu {gpu[worst]}, ref {ref[worst]})"
    assert mean <= mean_abs, f"{what}: mean-abs {mean:.3e}"
    return float(excess.max()), float(mean)


def check_topk_validity(gpu_idx: np.ndarray, ref_scores: np.ndarray, K: int, rel: float = 1e-5):
    """The GPU's selection must be a Top-K of the oracle's float64 scores up to
    near-ties: every picked score >= the oracle's K-th largest - tol and every
    unpicked score <= it + tol (tol = rel * max |score| of the row).  Returns
    the number of rows whose set differs from the oracle's exact set."""
    R = gpu_idx.reshape(-1, K)
    S = ref_scores.reshape(R.shape[0], -1)
    Nc = S.shape[1]
    assert R.min() >= 0 and R.max() < Nc
    kth = -np.sort(-S, axis=1)[:, K - 1]
    tol = rel * np.abs(S).max(axis=1) + 1e-7
    picked = np.zeros_like(S, dtype=bool)
    np.put_along_axis(picked, R.astype(np.int64), True, axis=1)
    assert np.all(picked.sum(1) == K), "repeated cube in a selected row"
    assert np.all(np.where(picked, S, np.inf).min(1) >= kth - tol), "a picked cube scores below the K-th"
    assert np.all(np.where(~picked, S, -np.inf).max(1) <= kth + tol), "an unpicked cube scores above the K-th"
    order = np.lexsort((np.broadcast_to(np.arange(Nc), S.shape), -S), axis=1)[:, :K]
    exact = np.zeros_like(picked)
    np.put_along_axis(exact, order, True, axis=1)
    return int((exact != picked).any(1).sum())


def exact_topk(scores: np.ndarray, K: int) -> np.ndarray:
    """Brute-force Top-K (score descending, lower id on ties) of given scores."""
    S = scores.reshape(-1, scores.shape[-1])
    Nc = S.shape[1]
    order = np.lexsort((np.broadcast_to(np.arange(Nc), S.shape), -S), axis=1)[:, :K]
    return order.reshape(scores.shape[:-1] + (K,))
