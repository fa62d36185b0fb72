"""Oracle O2: fp64 numpy restatements of the chunkwise WY algorithm.

TEST INFRASTRUCTURE ONLY (like everything under ``oracle/``). These functions
exist to pin the chunkwise algebra against the token recurrence of
``gdn_recurrence.c``; the GPU path never imports them.

Every function works on one (sequence, value head) chain whose q and k rows are
already L2-normalised:

    qn, kn : [T, K]     v : [T, V]     log_alpha, beta : [T]     S0 : [V, K]

and returns ``(out [T, V], S_final [V, K])``.

Sources
-------
* State transition ``S_t = S_{t-1} alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T``,
  cumulative gate ``gamma^r = prod_{j<=r} alpha_j``, ``Gamma^{r,i} = gamma^r / gamma^i``,
  the chunk transition ``S_[t+1] = S->_[t] + (U~_[t] - W<-_[t] S_[t]^T)^T K->_[t]``,
  ``W = (I + tril(B K K^T, -1))^{-1} B K`` and
  ``U~ = (I + tril(B (Gamma . K K^T), -1))^{-1} B V``:
  "Simple math to speed up GDN prefill", section "Reminder".
* ``M = I + tril(BKK^T,-1)``, ``N = I + tril(B(Gamma . KK^T),-1)``, ``N = G M G^{-1}`` and
  hence ``N^{-1} = G M^{-1} G^{-1}``: same page, section "Save one invert".
* The gamma-scaled form (WY rows with ``beta_i / gamma_i``, output
  ``O = gamma (S0 Q - (S0 W) triu(K^T Q) + U~ triu(K^T Q))`` and state
  ``S_new = gamma_C (S0 - (S0 W) K^T + U~^T K)``): pymllm
  "pymllm.layers.attention.gdn_chunkwise", Algorithm steps 1-3.

Readings
--------
* The page-4 arrows are read as ``S-> = gamma_C S``, ``W<- = G W`` (rows scaled by
  gamma) and ``K-> = diag(gamma_C / gamma) K``; with ``U~ = N^{-1} B V`` this gives
  the recurrence exactly (checked by the tests against the token recurrence).
* The page-3 ``w`` recursion is read as ``w_i = beta_i k_i - W_<i (K_<i^T (beta_i k_i))``
  (the same shape as its ``u~`` line); the literal text, with ``K`` and ``W``
  swapped, is kept as :func:`page3_w_rows_literal` so a test can show that it is
  not ``M^{-1} B K``.
* Rows are tokens (row-stacked); the page-3 formulas are written with tokens as
  columns and are transposed accordingly.
* Decay is kept in log space: ``g = cumsum(log alpha)`` inside the chunk, and every
  factor is ``exp(g_mu - g_nu)`` with ``mu >= nu`` (never ``1/gamma``), except in
  :func:`chunkwise_page3`, which is the page-3 form with ``1/gamma`` on purpose.
"""

from __future__ import annotations

import numpy as np


def _chunks(T: int, C: int):
    for s in range(0, T, C):
        yield s, min(s + C, T)


def gram_factors(kn: np.ndarray, beta: np.ndarray):
    """M = I + tril(diag(beta) K K^T, -1) for one chunk (page 4, "Save one invert")."""
    C = kn.shape[0]
    return np.eye(C) + np.tril(beta[:, None] * (kn @ kn.T), -1)


def decay_matrix(g: np.ndarray) -> np.ndarray:
    """Gamma_{mu,nu} = exp(g_mu - g_nu) on and below the diagonal, 0 above."""
    return np.tril(np.exp(g[:, None] - g[None, :]))


def n_inverse_two_ways(kn: np.ndarray, log_alpha: np.ndarray, beta: np.ndarray):
    """Return (N^{-1} by direct inversion, G M^{-1} G^{-1}) for one chunk.

    The second is formed entrywise as exp(g_mu - g_nu) * (M^{-1})_{mu,nu}, which
    is G M^{-1} G^{-1} without ever forming 1/gamma.
    """
    g = np.cumsum(log_alpha)
    Gam = decay_matrix(g)
    M = gram_factors(kn, beta)
    N = np.eye(len(beta)) + np.tril(beta[:, None] * (Gam * (kn @ kn.T)), -1)
    return np.linalg.inv(N), Gam * np.linalg.inv(M)


def chunk_factors(qn, kn, v, log_alpha, beta):
    """The per-chunk quantities of the page-4 form, for one chunk (rows = its tokens).

    Returns a dict with g = cumsum(log alpha) (chunk-local), Minv = M^{-1},
    A = N^{-1} B = (Gamma . M^{-1}) diag(beta) ("Save one invert"), W<- = A G K,
    U~ = A V and P = Gamma . tril(Q K^T), the masked, decayed scores of the output
    ("Reminder"): the same arithmetic as one iteration of :func:`chunkwise_forward`.
    """
    g = np.cumsum(log_alpha)
    Gam = decay_matrix(g)
    Minv = np.linalg.inv(gram_factors(kn, beta))
    A = (Gam * Minv) * beta[None, :]
    return dict(g=g, Minv=Minv, A=A, W=A @ (np.exp(g)[:, None] * kn), U=A @ v, P=Gam * (qn @ kn.T))


def chunkwise_forward(qn, kn, v, log_alpha, beta, S0, C, scale=1.0, inverses=1):
    """Page-4 chunkwise WY form in log space.

    Per chunk with g = cumsum(log alpha), G = diag(exp(g)), B = diag(beta):
      N^{-1} = G M^{-1} G^{-1}            (inverses=1; inverses=2 inverts N itself)
      W<-   = N^{-1} B G K,   U~ = N^{-1} B V
      U     = U~ - W<- S^T                 (the new values of the chunk)
      O     = G Q S^T + (Gamma . tril(Q K^T)) U
      S     = exp(g_C) S + U^T diag(exp(g_C - g)) K
    """
    T = qn.shape[0]
    S = np.array(S0, dtype=np.float64, copy=True)
    out = np.zeros((T, v.shape[1]))
    for s, e in _chunks(T, C):
        Q, Kc, Vc = qn[s:e], kn[s:e], v[s:e]
        g = np.cumsum(log_alpha[s:e])
        Gam = decay_matrix(g)
        if inverses == 1:
            Ninv = Gam * np.linalg.inv(gram_factors(Kc, beta[s:e]))
        else:
            N = np.eye(e - s) + np.tril(beta[s:e, None] * (Gam * (Kc @ Kc.T)), -1)
            Ninv = np.linalg.inv(N)
        A = Ninv * beta[s:e][None, :]  # N^{-1} B
        W_dec = A @ (np.exp(g)[:, None] * Kc)  # W<- = N^{-1} B G K
        U_tilde = A @ Vc
        U = U_tilde - W_dec @ S.T
        out[s:e] = scale * (np.exp(g)[:, None] * (Q @ S.T) + (Gam * (Q @ Kc.T)) @ U)
        S = np.exp(g[-1]) * S + U.T @ (np.exp(g[-1] - g)[:, None] * Kc)
    return out, S


def chunkwise_page3(qn, kn, v, log_alpha, beta, S0, C, scale=1.0):
    """Page-3 gamma-scaled form with the matrix reading W = M^{-1} B K.

    U~_p3 = M^{-1} B G^{-1} V (the rows beta_i / gamma_i v_i of the WY step), and
      O     = G (Q S^T - tril(Q K^T) (W S^T) + tril(Q K^T) U~_p3)
      S_new = gamma_C (S - (W S^T)^T K + U~_p3^T K)
    Uses 1/gamma, so it overflows for strongly decaying chunks; tests use it
    only on mild gates.
    """
    T = qn.shape[0]
    S = np.array(S0, dtype=np.float64, copy=True)
    out = np.zeros((T, v.shape[1]))
    for s, e in _chunks(T, C):
        Q, Kc, Vc = qn[s:e], kn[s:e], v[s:e]
        gamma = np.exp(np.cumsum(log_alpha[s:e]))
        Minv = np.linalg.inv(gram_factors(Kc, beta[s:e]))
        W = Minv @ (beta[s:e, None] * Kc)
        U3 = Minv @ ((beta[s:e] / gamma)[:, None] * Vc)
        mask_qk = np.tril(Q @ Kc.T)
        out[s:e] = scale * gamma[:, None] * (Q @ S.T - mask_qk @ (W @ S.T) + mask_qk @ U3)
        S = gamma[-1] * (S - (W @ S.T).T @ Kc + U3.T @ Kc)
    return out, S


def wy_rows(kn: np.ndarray, beta: np.ndarray) -> np.ndarray:
    """Row recursion w_i = beta_i k_i - sum_{j<i} (beta_i k_j . k_i) w_j (= M^{-1} B K)."""
    W = np.zeros_like(kn)
    for i in range(kn.shape[0]):
        bk = beta[i] * kn[i]
        W[i] = bk - (kn[:i] @ bk) @ W[:i]
    return W


def page3_w_rows_literal(kn: np.ndarray, beta: np.ndarray) -> np.ndarray:
    """The page-3 line as printed: w_i = beta_i k_i - K_<i (W_<i^T (beta_i k_i)).

    With columns k_j and w_j this is sum_{j<i} (w_j . beta_i k_i) k_j: K and W swap
    roles relative to :func:`wy_rows`. Kept only to document that reading.
    """
    W = np.zeros_like(kn)
    for i in range(kn.shape[0]):
        bk = beta[i] * kn[i]
        W[i] = bk - (W[:i] @ bk) @ kn[:i]
    return W


def brute_force(qn, kn, v, alpha, beta, S0, scale=1.0):
    """The state transition multiplied out as written, one K x K matrix per token."""
    T, K = kn.shape
    S = np.array(S0, dtype=np.float64, copy=True)
    out = np.zeros((T, v.shape[1]))
    for t in range(T):
        k = kn[t][:, None]
        S = S @ (alpha[t] * (np.eye(K) - beta[t] * (k @ k.T))) + beta[t] * (v[t][:, None] @ k.T)
        out[t] = scale * (S @ qn[t])
    return out, S
