"""Sequential temperature scaling (STS) of the confidence head: the offline fit.

"DSpark" §3.2 (STS): the scheduler consumes the absolute values of the survival
products a_j = prod_{i<=j} c_i, so the confidence head is calibrated after
training on held-out rounds.  One temperature per draft position is searched
left to right; positions already fitted keep their temperature, and position j
takes the t_j on a one-dimensional grid that minimises the expected calibration
error (ECE) of a_j against the event "the first j + 1 drafts were accepted".
Dividing a logit by t_j > 0 preserves the order of the confidences, so the
ranking the scheduler sorts by within one position does not change.

This module is the host-side fitting tool.  The fitted temperatures are applied
on the device by ``dspark_confidence(..., sts_temperature=t)``.

Readings where the pages are silent: ECE uses equal-width bins over [0, 1]
(15 by default), each bin weighted by its share of the samples, the last bin
closed; the grid is log-spaced over [0.05, 20]; on ties the grid point closest
to t = 1 wins (the smallest change to the head).
"""
from __future__ import annotations

import numpy as np

__all__ = ["ece", "default_grid", "logits_from_confidence", "apply_sts", "fit_sts"]


def ece(pred, label, n_bins: int = 15) -> float:
    """Expected calibration error of probabilities `pred` against 0/1 `label`:
    sum over equal-width bins of (bin share) * |mean(pred) - mean(label)|."""
    pred = np.asarray(pred, np.float64).ravel()
    label = np.asarray(label, np.float64).ravel()
    if pred.shape != label.shape:
        raise ValueError("pred and label must have the same number of elements")
    n = pred.size
    if n == 0:
        return 0.0
    if n_bins < 1:
        raise ValueError("n_bins must be positive")
    idx = np.minimum((np.clip(pred, 0.0, 1.0) * n_bins).astype(np.int64), n_bins - 1)
    sum_p = np.bincount(idx, weights=pred, minlength=n_bins)
    sum_y = np.bincount(idx, weights=label, minlength=n_bins)
    return float(np.sum(np.abs(sum_p - sum_y)) / n)


def default_grid(n: int = 241, lo: float = 0.05, hi: float = 20.0) -> np.ndarray:
    """n log-spaced temperatures over [lo, hi], plus t = 1 (the identity)."""
    g = np.exp(np.linspace(np.log(lo), np.log(hi), n))
    return np.unique(np.concatenate([g, [1.0]]))


def logits_from_confidence(c) -> np.ndarray:
    """Inverse sigmoid of confidences in (0, 1), in fp64."""
    c = np.asarray(c, np.float64)
    return np.log(c) - np.log1p(-c)


def _sigmoid(z):
    z = np.asarray(z, np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    e = np.exp(z[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def apply_sts(logits, t) -> tuple[np.ndarray, np.ndarray]:
    """c_j = sigma(logit_j / t_j) and a_j = prod_{i<=j} c_i (fp64), for logits [N, gamma]."""
    logits = np.asarray(logits, np.float64)
    t = np.asarray(t, np.float64)
    if logits.ndim != 2 or t.shape != (logits.shape[1],):
        raise ValueError("logits must be [N, gamma] and t [gamma]")
    c = _sigmoid(logits / t[None, :])
    return c, np.cumprod(c, axis=1)


def fit_sts(logits, n_accept, grid=None, n_bins: int = 15):
    """Fit one temperature per position, left to right.

    logits   [N, gamma]  raw confidence logits of N held-out draft blocks
    n_accept [N]         accepted draft length of each block (0..gamma)
    Returns (t [gamma] float32, ece_before [gamma], ece_after [gamma]), the ECEs
    being those of a_j against 1[n_accept > j] without and with the fitted t.
    """
    logits = np.asarray(logits, np.float64)
    n_accept = np.asarray(n_accept)
    if logits.ndim != 2 or n_accept.shape != (logits.shape[0],):
        raise ValueError("logits must be [N, gamma] and n_accept [N]")
    N, gamma = logits.shape
    if N and (n_accept.min() < 0 or n_accept.max() > gamma):
        raise ValueError("n_accept must lie in [0, gamma]")
    grid = default_grid() if grid is None else np.asarray(grid, np.float64)
    if grid.ndim != 1 or grid.size == 0 or not np.all(grid > 0) or not np.all(np.isfinite(grid)):
        raise ValueError("grid must hold finite positive temperatures")
    # candidates in order of closeness to 1 so that argmin breaks ties towards t = 1
    order = np.argsort(np.abs(np.log(grid)), kind="stable")
    cand = grid[order]
    t = np.ones(gamma, np.float64)
    before = np.empty(gamma)
    after = np.empty(gamma)
    a_raw = np.ones(N)
    a_fit = np.ones(N)
    for j in range(gamma):
        label = n_accept > j
        a_raw = a_raw * _sigmoid(logits[:, j])
        before[j] = ece(a_raw, label, n_bins)
        errs = np.array([ece(a_fit * _sigmoid(logits[:, j] / tj), label, n_bins) for tj in cand])
        t[j] = cand[int(np.argmin(errs))]
        a_fit = a_fit * _sigmoid(logits[:, j] / t[j])
        after[j] = ece(a_fit, label, n_bins)
    return t.astype(np.float32), before, after
