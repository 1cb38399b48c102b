"""Float64 oracle for the compact pattern fit (test infrastructure only).

Source: "When Can Attention Heads Be Statically Defined?" (close-reading
notes), §3 (Eq. (3) and the text around Eq. (4)) and App. A.2:

* the fixed pattern of a chosen head is the calibration mean A_hat; it is
  compressed into the two length-T vectors alpha (absolute key position) and
  rho (distance i - j) of Eq. (3) by minimising the row-wise cross-entropy of
  P_hat(alpha, rho) against A_hat;
* the target's absolute-position and distance marginals are sufficient
  statistics for that fit (Eq. (4)): with dl(i, j) = P_hat(i, j) - A_hat(i, j),
  the gradient of the row-averaged cross-entropy is the column sums (alpha)
  and the diagonal sums (rho) of dl / T, and the A_hat part of those sums is
  just its two marginals;
* each candidate gets 400 Adam steps; a head whose mean row KL(A_hat || P_hat)
  exceeds 0.2 nat is skipped and the next head in variance order is tried.

Readings where the notes are silent: rows are averaged (the loss is
(1/T) sum_i CE_i); Adam uses lr = 1e-2, beta = (0.9, 0.999), eps = 1e-8
(Kingma & Ba's published defaults except the rate); alpha and rho start from
the log of the marginals averaged over their valid entries,
alpha0(j) = log(sum_i A_hat(i,j) / (T - j)), rho0(d) = log(sum_i A_hat(i,i-d) / (T - d)),
floored at 1e-30.
"""

from __future__ import annotations

import numpy as np

from .attention import static_pattern

__all__ = [
    "marginals",
    "fit_loss",
    "fit_gradient",
    "mean_row_kl",
    "adam_step",
    "compact_fit",
    "select_fitted",
]


def marginals(P: np.ndarray):
    """(column sums, diagonal sums) of a T x T matrix: col(j) = sum_i P(i, j),
    diag(d) = sum_i P(i, i - d)."""
    P = np.asarray(P, dtype=np.float64)
    T = P.shape[0]
    return P.sum(axis=0), np.array([np.trace(P, offset=-d) for d in range(T)])


def fit_loss(alpha, rho, A_hat) -> float:
    """Row-averaged cross-entropy -(1/T) sum_i sum_{j<=i} A_hat(i,j) log P_hat(i,j)."""
    P = static_pattern(alpha, rho)
    A = np.asarray(A_hat, dtype=np.float64)
    m = A > 0
    return float(-(A[m] * np.log(P[m])).sum() / A.shape[0])


def fit_gradient(alpha, rho, target_marginals):
    """Gradient of fit_loss from the sufficient statistics of the target."""
    T = len(alpha)
    col_t, diag_t = target_marginals
    col_p, diag_p = marginals(static_pattern(alpha, rho))
    return (col_p - col_t) / T, (diag_p - diag_t) / T


def mean_row_kl(A_hat, P) -> float:
    """(1/T) sum_i KL(A_hat(i, :) || P(i, :)), in nats."""
    A = np.asarray(A_hat, dtype=np.float64)
    P = np.asarray(P, dtype=np.float64)
    m = A > 0
    return float((A[m] * (np.log(A[m]) - np.log(P[m]))).sum() / A.shape[0])


def adam_step(theta, g, m, v, t, lr, beta1, beta2, eps):
    """One Adam update (Kingma & Ba, Algorithm 1) of step number t >= 1:
    moments m, v; bias-corrected mhat, vhat; theta - lr mhat / (sqrt(vhat) + eps).
    Returns (theta, m, v)."""
    m = beta1 * m + (1 - beta1) * g
    v = beta2 * v + (1 - beta2) * g * g
    mhat = m / (1 - beta1 ** t)
    vhat = v / (1 - beta2 ** t)
    return theta - lr * mhat / (np.sqrt(vhat) + eps), m, v


def compact_fit(A_hat, steps=400, lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8):
    """Fit (alpha, rho) to one head's A_hat.  Returns (alpha, rho, mean row KL)."""
    A = np.asarray(A_hat, dtype=np.float64)
    T = A.shape[0]
    col_t, diag_t = marginals(A)
    alpha = np.log(np.maximum(col_t / (T - np.arange(T)), 1e-30))
    rho = np.log(np.maximum(diag_t / (T - np.arange(T)), 1e-30))
    m_a = np.zeros(T)
    v_a = np.zeros(T)
    m_r = np.zeros(T)
    v_r = np.zeros(T)
    for t in range(1, steps + 1):
        g_a, g_r = fit_gradient(alpha, rho, (col_t, diag_t))
        alpha, m_a, v_a = adam_step(alpha, g_a, m_a, v_a, t, lr, beta1, beta2, eps)
        rho, m_r, v_r = adam_step(rho, g_r, m_r, v_r, t, lr, beta1, beta2, eps)
    return alpha, rho, mean_row_kl(A, static_pattern(alpha, rho))


def select_fitted(order, kls, k, kl_max=0.2):
    """Walk the candidates in `order` (ascending s_var) and keep the first k
    whose fitted pattern has mean row KL <= kl_max; `kls[i]` belongs to
    order[i]."""
    out = []
    for h, kl in zip(order, kls):
        if len(out) == k:
            break
        if kl <= kl_max:
            out.append(int(h))
    return np.asarray(out, dtype=np.int64)
