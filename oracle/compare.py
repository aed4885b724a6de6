"""Parity criteria between the CUDA path and the oracle — TEST INFRASTRUCTURE.

Scores: |I_gpu - I_ora| <= rtol * max(|I_ora|, mean_s |I_ora[t, :n_t]|) with
rtol = 2e-3. A plain relative bound fails near zero, and with head weights of
both signs the head sum cancels, so the row's mean magnitude is the floor.

Top-k sets: with tau the oracle's k-th score of the row and eps the score
tolerance at tau, every GPU id must score >= tau - eps in the oracle, every
oracle id scoring > tau + eps must be in the GPU set, the numbers of valid ids
agree, ids are distinct and inside [0, n_t), and the tail is -1. Ties within
the tolerance at the k-th boundary may be resolved either way.
"""
from __future__ import annotations

import numpy as np

RTOL = 2e-3


def score_tolerance(ora_row: np.ndarray, rtol: float = RTOL) -> np.ndarray:
    floor = np.abs(ora_row).mean() if ora_row.size else 0.0
    return rtol * np.maximum(np.abs(ora_row), floor)


def check_scores(gpu_row: np.ndarray, ora_row: np.ndarray, rtol: float = RTOL):
    """Returns (ok, worst ratio of error to tolerance, index of the worst)."""
    gpu_row = np.asarray(gpu_row, np.float64)
    if not np.all(np.isfinite(gpu_row)):
        return False, float("inf"), int(np.argmin(np.isfinite(gpu_row)))
    tol = score_tolerance(ora_row, rtol)
    err = np.abs(gpu_row - ora_row)
    ratio = err / np.maximum(tol, 1e-300)
    i = int(np.argmax(ratio)) if ratio.size else 0
    worst = float(ratio[i]) if ratio.size else 0.0
    return worst <= 1.0, worst, i


def check_topk_row(gpu_ids: np.ndarray, ora_scores: np.ndarray, k: int, rtol: float = RTOL):
    """Check one row of GPU top-k ids against the oracle's fp64 scores (length n_t).

    Returns (ok, message)."""
    n = int(ora_scores.shape[0])
    gpu_ids = np.asarray(gpu_ids, np.int64)
    m = min(k, n)
    valid = gpu_ids[gpu_ids >= 0]
    if valid.size != m:
        return False, f"{valid.size} valid ids, expected {m}"
    if np.any(gpu_ids[gpu_ids < 0] != -1):
        return False, "negative id other than -1"
    if np.unique(valid).size != valid.size:
        return False, "duplicate ids"
    if valid.size and (valid.min() < 0 or valid.max() >= n):
        return False, "id outside the row"
    if m == n:
        return (True, "") if set(valid.tolist()) == set(range(n)) else (False, "short row is not every key")
    order = np.argsort(-ora_scores, kind="stable")
    tau = ora_scores[order[k - 1]]
    eps = score_tolerance(np.array([tau]), rtol)[0] if n else 0.0
    eps = max(eps, rtol * np.abs(ora_scores).mean())
    low = ora_scores[valid] < tau - eps
    if np.any(low):
        bad = valid[low][0]
        return False, f"id {bad} scores {ora_scores[bad]:.6g} < tau-eps {tau - eps:.6g}"
    must = np.nonzero(ora_scores > tau + eps)[0]
    missing = np.setdiff1d(must, valid)
    if missing.size:
        return False, f"{missing.size} ids above tau+eps missing, e.g. {missing[0]}"
    return True, ""


def check_topk(gpu_topk: np.ndarray, ora_scores: np.ndarray, row_lens: np.ndarray, k: int, rtol: float = RTOL):
    """All rows; ``ora_scores[i, :row_lens[i]]`` are row i's scores. Returns list of failures."""
    fails = []
    for i in range(gpu_topk.shape[0]):
        ok, msg = check_topk_row(gpu_topk[i], ora_scores[i, : int(row_lens[i])], k, rtol)
        if not ok:
            fails.append((i, msg))
    return fails
