"""Float64 oracle for the hybrid causal attention layer (test infrastructure only).

Source: "When Can Attention Heads Be Statically Defined?" (close-reading
notes).  Indices are 0-based: query i, key j, distance i - j.  The page's
Z(i) sums k = 1..i in 1-based notation; here k runs over 0..i.

All arrays are NumPy float64 and every T x T matrix is materialised.  No
blocking, online softmax or factoring is used: each function is the
definition written out.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "causal_mask",
    "dynamic_head_fwd",
    "dynamic_head_bwd",
    "static_pattern",
    "static_log_normaliser",
    "static_head_fwd",
    "static_head_bwd",
    "hybrid_attn_fwd",
    "hybrid_attn_bwd",
    "dynamic_head_fwd_rows",
    "static_head_fwd_rows",
    "dynamic_head_bwd_rows",
    "static_head_bwd_rows",
]


def causal_mask(T: int) -> np.ndarray:
    """Boolean [T, T] mask, True where key j <= query i (diagonal included)."""
    return np.tril(np.ones((T, T), dtype=bool))


def _causal_row_softmax(L: np.ndarray):
    """Row softmax of a logit matrix whose masked entries are -inf.

    Returns (P, lse) with lse(i) = log sum_j exp L(i, j).  A row whose every
    logit is -inf has no distribution; by the reading recorded for the
    build it yields an all-zero row and lse = -inf.
    """
    m = L.max(axis=1)
    finite = np.isfinite(m)
    shift = np.where(finite, m, 0.0)
    with np.errstate(invalid="ignore"):
        e = np.exp(L - shift[:, None])
    e[~finite, :] = 0.0
    s = e.sum(axis=1)
    P = np.zeros_like(L)
    P[finite] = e[finite] / s[finite, None]
    lse = np.full(L.shape[0], -np.inf)
    lse[finite] = shift[finite] + np.log(s[finite])
    return P, lse


# --------------------------------------------------------------------------
# Dynamic head: A = softmax_causal(Q K^T / sqrt(d_h)), Z = A V   (§1 equation)
# --------------------------------------------------------------------------

def dynamic_head_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray):
    """One dynamic head.  q, k, v: [T, d_h] float64.

    Returns (out [T, d_h], lse [T], A [T, T]).
    """
    T, d = q.shape
    S = (q @ k.T) / np.sqrt(d)
    S = np.where(causal_mask(T), S, -np.inf)
    A, lse = _causal_row_softmax(S)
    return A @ v, lse, A


def dynamic_head_bwd(q, k, v, dout):
    """Gradients of the scalar loss sum(dout * out) for one dynamic head.

    The softmax Jacobian applied to dA = dout V^T gives
    dS(i, j) = A(i, j) * (dA(i, j) - sum_k A(i, k) dA(i, k)); the 1/sqrt(d_h)
    logit scale then carries into dQ and dK.  Returns (dq, dk, dv).
    """
    T, d = q.shape
    _, _, A = dynamic_head_fwd(q, k, v)
    dv = A.T @ dout
    dA = dout @ v.T
    row = (A * dA).sum(axis=1, keepdims=True)
    dS = A * (dA - row)
    dq = dS @ k / np.sqrt(d)
    dk = dS.T @ q / np.sqrt(d)
    return dq, dk, dv


# --------------------------------------------------------------------------
# Static head: P(i,j) = exp(alpha(j) + rho(i-j)) / Z(i), j <= i   (Eq. (3))
# --------------------------------------------------------------------------

def _static_logits(alpha: np.ndarray, rho: np.ndarray) -> np.ndarray:
    """L(i, j) = alpha(j) + rho(i - j) on the causal triangle, -inf above it."""
    T = alpha.shape[0]
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    dist = i - j
    L = np.full((T, T), -np.inf)
    mask = dist >= 0
    L[mask] = (alpha[None, :] + rho[np.clip(dist, 0, T - 1)])[mask]
    return L


def static_pattern(alpha: np.ndarray, rho: np.ndarray) -> np.ndarray:
    """The compact fixed pattern P_hat [T, T] of one frozen head (Eq. (3))."""
    P, _ = _causal_row_softmax(_static_logits(alpha, rho))
    return P


def static_log_normaliser(alpha: np.ndarray, rho: np.ndarray) -> np.ndarray:
    """log Z(i) = log sum_{k<=i} exp(alpha(k) + rho(i-k)), shape [T]."""
    _, lse = _causal_row_softmax(_static_logits(alpha, rho))
    return lse


def static_head_fwd(alpha, rho, v):
    """One frozen head on one sequence: out = P_hat V, and log Z per row."""
    P, logZ = _causal_row_softmax(_static_logits(alpha, rho))
    return P @ v, logZ


def static_head_bwd(alpha, rho, v_list, dout_list):
    """Backward of a frozen head over a batch of sequences.

    v_list, dout_list: sequences of [T, d_h] arrays, one per batch element.
    Returns (dv_list, dalpha [T], drho [T]).

    dV_b = P_hat^T dO_b is the static head's whole attention backward (§3.3 /
    App. D.2).  The alpha/rho gradients (the paper keeps them frozen) are the
    chain rule through Eq. (3): with dP_b = dO_b V_b^T the logit gradient is
    dl = sum_b P_hat * (dP_b - rowsum(P_hat * dP_b)); alpha(j) receives the
    column sums of dl and rho(delta) the sums along each diagonal i - j = delta.
    """
    T = alpha.shape[0]
    P = static_pattern(alpha, rho)
    dv_list = [P.T @ dout for dout in dout_list]
    dl = np.zeros((T, T))
    for v, dout in zip(v_list, dout_list):
        dP = dout @ v.T
        row = (P * dP).sum(axis=1, keepdims=True)
        dl += P * (dP - row)
    dalpha = dl.sum(axis=0)
    drho = np.array([np.trace(dl, offset=-delta) for delta in range(T)])
    return dv_list, dalpha, drho


# --------------------------------------------------------------------------
# The hybrid layer: dynamic and static heads side by side
# --------------------------------------------------------------------------

def _as64(x):
    return np.asarray(x, dtype=np.float64)


def hybrid_attn_fwd(Q, K, V, alpha, rho, head_is_static):
    """Q, K, V: [B, H, T, d_h]; alpha, rho: [H, T]; head_is_static: [H] bools.

    Returns (out [B, H, T, d_h], lse [B, H, T]).  Static heads read only V;
    their lse slot holds log Z(i).
    """
    Q, K, V = _as64(Q), _as64(K), _as64(V)
    alpha, rho = _as64(alpha), _as64(rho)
    B, H, T, d = V.shape
    out = np.zeros((B, H, T, d))
    lse = np.zeros((B, H, T))
    for h in range(H):
        if head_is_static[h]:
            P, logZ = _causal_row_softmax(_static_logits(alpha[h], rho[h]))
            for b in range(B):
                out[b, h] = P @ V[b, h]
                lse[b, h] = logZ
        else:
            for b in range(B):
                o, l, _ = dynamic_head_fwd(Q[b, h], K[b, h], V[b, h])
                out[b, h] = o
                lse[b, h] = l
    return out, lse


def hybrid_attn_bwd(Q, K, V, alpha, rho, head_is_static, dout,
                    want_param_grads=True):
    """Gradients of sum(dout * out) for the hybrid layer.

    Returns (dQ, dK, dV, dalpha, drho).  dQ and dK are zero on static heads
    (those heads have no query/key path).  dalpha/drho are [H, T], summed over
    the batch, zero on dynamic rows; they are None when not requested.
    """
    Q, K, V, dout = _as64(Q), _as64(K), _as64(V), _as64(dout)
    alpha, rho = _as64(alpha), _as64(rho)
    B, H, T, d = V.shape
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    dalpha = np.zeros((H, T)) if want_param_grads else None
    drho = np.zeros((H, T)) if want_param_grads else None
    for h in range(H):
        if head_is_static[h]:
            dvs, da, dr = static_head_bwd(alpha[h], rho[h],
                                          [V[b, h] for b in range(B)],
                                          [dout[b, h] for b in range(B)])
            for b in range(B):
                dV[b, h] = dvs[b]
            if want_param_grads:
                dalpha[h] = da
                drho[h] = dr
        else:
            for b in range(B):
                dq, dk, dv = dynamic_head_bwd(Q[b, h], K[b, h], V[b, h],
                                              dout[b, h])
                dQ[b, h], dK[b, h], dV[b, h] = dq, dk, dv
    return dQ, dK, dV, dalpha, drho


def _kv_expand(X, H):
    """[B, H_kv, T, d] -> [B, H, T, d]: kv head c serves query heads
    c*g .. c*g + g - 1, g = H / H_kv."""
    X = _as64(X)
    H_kv = X.shape[1]
    if H % H_kv != 0:
        raise ValueError("H must be a multiple of H_kv")
    return np.repeat(X, H // H_kv, axis=1)


def gqa_hybrid_attn_fwd(Q, K, V, alpha, rho, head_is_static):
    """Grouped-query form of the hybrid layer (the GQA path of §3.3 / App. D.2:
    K and V are shared by groups of query heads, so freezing a query head
    removes only its query path and it still mixes its group's V).

    Q: [B, H, T, d_h]; K, V: [B, H_kv, T, d_h], H a multiple of H_kv; query
    head h reads kv head h // (H / H_kv).  Same outputs as hybrid_attn_fwd.
    """
    H = np.asarray(Q).shape[1]
    return hybrid_attn_fwd(Q, _kv_expand(K, H), _kv_expand(V, H), alpha, rho, head_is_static)


def gqa_hybrid_attn_bwd(Q, K, V, alpha, rho, head_is_static, dout, want_param_grads=True):
    """Gradients of sum(dout * out) for the grouped-query layer: dK and dV of a
    kv head are the sums over the query heads it serves ([B, H_kv, T, d_h]);
    dQ, dalpha, drho are per query head, as in hybrid_attn_bwd."""
    Q = _as64(Q)
    B, H, T, d = Q.shape
    H_kv = np.asarray(K).shape[1]
    dQ, dKe, dVe, da, dr = hybrid_attn_bwd(Q, _kv_expand(K, H), _kv_expand(V, H), alpha, rho,
                                           head_is_static, dout, want_param_grads)
    g = H // H_kv
    dK = dKe.reshape(B, H_kv, g, T, d).sum(axis=2)
    dV = dVe.reshape(B, H_kv, g, T, d).sum(axis=2)
    return dQ, dK, dV, da, dr


# --------------------------------------------------------------------------
# Row-restricted forms (the same definitions evaluated on a subset of query
# rows), for spot checks of full-size outputs.
# --------------------------------------------------------------------------

def dynamic_head_fwd_rows(q, k, v, rows):
    """Rows ``rows`` of (out, lse) of one dynamic head.  Row i of causal
    attention depends only on q_i and keys/values 0..i."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    T, d = k.shape
    rows = np.asarray(rows)
    S = (q[rows] @ k.T) / np.sqrt(d)
    S = np.where(np.arange(T)[None, :] <= rows[:, None], S, -np.inf)
    A, lse = _causal_row_softmax(S)
    return A @ v, lse


def static_head_fwd_rows(alpha, rho, v, rows):
    """Rows ``rows`` of (out, log Z) of one frozen head."""
    alpha, rho, v = _as64(alpha), _as64(rho), _as64(v)
    T = alpha.shape[0]
    rows = np.asarray(rows)
    j = np.arange(T)[None, :]
    dist = rows[:, None] - j
    L = np.full((len(rows), T), -np.inf)
    m = dist >= 0
    L[m] = (alpha[None, :] + rho[np.clip(dist, 0, T - 1)])[m]
    P, lse = _causal_row_softmax(L)
    return P @ v, lse


def dynamic_head_bwd_rows(q, k, v, dout, rows):
    """Contribution of the query rows ``rows`` to the backward of one dynamic
    head: (dq for those rows, their part of dk, their part of dv).  Summing the
    parts over a partition of all rows gives dynamic_head_bwd."""
    q, k, v, dout = _as64(q), _as64(k), _as64(v), _as64(dout)
    T, d = k.shape
    rows = np.asarray(rows)
    S = (q[rows] @ k.T) / np.sqrt(d)
    S = np.where(np.arange(T)[None, :] <= rows[:, None], S, -np.inf)
    A, _ = _causal_row_softmax(S)
    dv = A.T @ dout[rows]
    dA = dout[rows] @ v.T
    dS = A * (dA - (A * dA).sum(axis=1, keepdims=True))
    return dS @ k / np.sqrt(d), dS.T @ q[rows] / np.sqrt(d), dv


def static_head_bwd_rows(alpha, rho, v, dout, rows):
    """Contribution of the query rows ``rows`` of one sequence to a frozen
    head's backward: (its part of dv, of dalpha, of drho)."""
    alpha, rho, v, dout = _as64(alpha), _as64(rho), _as64(v), _as64(dout)
    T = alpha.shape[0]
    rows = np.asarray(rows)
    j = np.arange(T)[None, :]
    dist = rows[:, None] - j
    L = np.full((len(rows), T), -np.inf)
    m = dist >= 0
    L[m] = (alpha[None, :] + rho[np.clip(dist, 0, T - 1)])[m]
    P, _ = _causal_row_softmax(L)
    dv = P.T @ dout[rows]
    dP = dout[rows] @ v.T
    dl = P * (dP - (P * dP).sum(axis=1, keepdims=True))
    dalpha = dl.sum(axis=0)
    drho = np.zeros(T)
    np.add.at(drho, np.clip(dist, 0, T - 1)[m], dl[m])
    return dv, dalpha, drho
