"""Float64 oracle for the SAF calibration reduction (test infrastructure only).

Source: "When Can Attention Heads Be Statically Defined?" (close-reading
notes), §3.1: the per-head sample mean A_hat over N calibration sequences,
the variance score of Eq. (1), and the global ascending sort of all layers'
heads by that score, from which the first k = round(r L H) are taken.
App. B.1 gives the decomposition R(P) = R(E[A]) + ||P - E[A]||_F^2 / T^2 that
``reconstruction_risk`` lets the tests check.

Two-pass, float64, full T x T matrices.  Entries above the diagonal are zero
by causality; the oracle keeps them (they contribute nothing).
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "calib_mean",
    "calib_svar",
    "calib_mean_svar",
    "num_select",
    "select_heads",
    "reconstruction_risk",
    "calib_kl_score",
    "sharp_mean_pattern",
]


def calib_mean(A: np.ndarray) -> np.ndarray:
    """A_hat = (1/N) sum_n A_n for one head.  A: [N, T, T]."""
    A = np.asarray(A, dtype=np.float64)
    return A.sum(axis=0) / A.shape[0]


def calib_svar(A: np.ndarray, A_hat: np.ndarray | None = None) -> float:
    """Eq. (1): s_var = sum_n ||A_n - A_hat||_F^2 / ((N - 1) T^2).  N >= 2."""
    A = np.asarray(A, dtype=np.float64)
    N, T, _ = A.shape
    if N < 2:
        raise ValueError("s_var needs N >= 2 calibration samples")
    if A_hat is None:
        A_hat = calib_mean(A)
    dev = A - A_hat[None]
    return float((dev * dev).sum() / ((N - 1) * T * T))


def calib_mean_svar(A_all: np.ndarray):
    """A_all: [N, heads, T, T] -> (A_hat [heads, T, T], s_var [heads])."""
    A_all = np.asarray(A_all)
    N, nh, T, _ = A_all.shape
    A_hat = np.zeros((nh, T, T))
    s_var = np.zeros(nh)
    for h in range(nh):
        A = A_all[:, h].astype(np.float64)
        A_hat[h] = calib_mean(A)
        s_var[h] = calib_svar(A, A_hat[h])
    return A_hat, s_var


def num_select(r: float, num_heads: int) -> int:
    """k = round(r * L * H), rounding exact halves to even."""
    return int(round(r * num_heads))


def select_heads(s_var, k: int) -> np.ndarray:
    """Heads of all layers sorted ascending by s_var; ties go to the lower
    flat index l * H + h.  Returns the first k flat indices in that order."""
    s_var = np.asarray(s_var)
    order = sorted(range(len(s_var)), key=lambda i: (s_var[i], i))
    return np.asarray(order[:k], dtype=np.int64)


def reconstruction_risk(P: np.ndarray, A: np.ndarray) -> float:
    """R(P) = mean_n ||A_n - P||_F^2 / T^2 under the empirical measure."""
    A = np.asarray(A, dtype=np.float64)
    N, T, _ = A.shape
    dev = A - np.asarray(P, dtype=np.float64)[None]
    return float((dev * dev).sum() / (N * T * T))


def calib_kl_score(A: np.ndarray, A_hat: np.ndarray | None = None) -> float:
    """Row-wise forward-KL score of one head: the mean over the N samples and
    the T rows of KL(A_n(i, :) || A_hat(i, :)), in nats.  This is the
    alternative selector the notes compare against s_var (§3.1 and App. B.2);
    its formula is not printed there, and this mean over samples and rows is
    the reading taken.  Terms with A_n(i, j) = 0 contribute nothing."""
    A = np.asarray(A, dtype=np.float64)
    N, T, _ = A.shape
    if A_hat is None:
        A_hat = calib_mean(A)
    total = 0.0
    for n in range(N):
        m = A[n] > 0
        total += float((A[n][m] * (np.log(A[n][m]) - np.log(A_hat[m]))).sum())
    return total / (N * T)


def sharp_mean_pattern(L: np.ndarray) -> np.ndarray:
    """The sharp-mean fixed pattern of one head (one of the candidate fixed
    patterns listed with the probability mean in §3, compared in §5.1 /
    Fig. 3): the pre-softmax logits are
    averaged over the N samples first, and each row of that mean then goes
    through a causal softmax.  L: [N, T, T]; only j <= i is read.  Returns
    [T, T] with exact zeros above the diagonal."""
    L = np.asarray(L, dtype=np.float64)
    N, T, _ = L.shape
    M = L.sum(axis=0) / N
    P = np.zeros((T, T))
    for i in range(T):
        row = M[i, : i + 1]
        e = np.exp(row - row.max())
        P[i, : i + 1] = e / e.sum()
    return P
