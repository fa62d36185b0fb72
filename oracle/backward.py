"""Oracle O3: gradients of the GDN token recurrence, fp64, CPU.

TEST INFRASTRUCTURE ONLY (like everything under ``oracle/``): the GPU library never imports it.

What it differentiates
----------------------
The forward is O1's recurrence, per (sequence, value head) chain with q/k head h = hv // (HV/H):

    q^ = q / sqrt(|q|^2 + 1e-6),  k^ likewise
    log alpha = -exp(A_log) softplus(a + dt_bias),  beta = sigmoid(b)
    S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k^_t) k^_t^T
        (= S_{t-1} alpha_t (I - beta_t k^_t k^_t^T) + beta_t v_t k^_t^T,
         "Simple math to speed up GDN prefill", section "Reminder")
    o_t = scale S_t q^_t      (after the write: "nrm-training-kernels", "General implementation", item 4)

and the scalar whose gradient is taken is

    L = sum_t <dO_t, o_t> + <dS_T, S_T>,

so ``d_out`` and ``d_state`` are the gradients arriving from above: the output's, and the final
state's. The second is the extra incoming state gradient that the bottom level's backward accepts in
"nrm-training-kernels", section "Kernel". The pages print no gradient formulas. Everything below is the
chain rule applied to the forward above, one token at a time, backwards, with the states recomputed by
a forward sweep.

Per token, with u = S_{t-1} k^ and delta = beta (v - alpha u), so that S_t = alpha S_{t-1} + delta k^^T, and
G the gradient of S_t:

    G      += scale dO_t q^^T                   dq^ = scale S_t^T dO_t
    d delta = G k^                              dk^ = G^T delta + S_{t-1}^T du
    d alpha = <G, S_{t-1}> - beta <d delta, u>  d beta = <d delta, v - alpha u>
    dv      = beta d delta                      du = -alpha beta d delta
    G_{t-1} = alpha G + du k^^T

then the gates (d log alpha = alpha d alpha; softplus' = sigmoid; d/dA_log log alpha = log alpha) and the
normalisation (dq = dq^/n - q (q . dq^)/n^3 with n = sqrt(|q|^2 + eps)). GQA: a q/k head collects the
gradients of all its value heads. The gradient of each touched pool slot is G_0 of its chain.
"""

from __future__ import annotations

import numpy as np

EPS = 1e-6


def _softplus(x: float) -> float:
    return max(x, 0.0) + np.log1p(np.exp(-abs(x)))


def _sigmoid(x: float) -> float:
    return 1.0 / (1.0 + np.exp(-x))


def chain_backward(q, k, v, a, b, A_log: float, dt_bias: float, S0, d_out, d_state, scale: float = 1.0):
    """Gradients of one chain (raw inputs, fp64).

    q, k: [T, K] (not normalised); v, d_out: [T, V]; a, b: [T]; A_log, dt_bias: scalars;
    S0, d_state: [V, K]. Returns a dict with dq, dk [T, K], dv [T, V], da, db [T], dA_log, ddt_bias
    (scalars) and dS0 [V, K], plus the forward's out [T, V] and S_final [V, K].
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    a, b = np.asarray(a, dtype=np.float64).reshape(-1), np.asarray(b, dtype=np.float64).reshape(-1)
    d_out = np.asarray(d_out, dtype=np.float64)
    T, K = k.shape
    V = v.shape[1]
    eA = np.exp(float(A_log))

    # forward sweep: keep S_{t-1} and the per-token scalars
    S = np.array(S0, dtype=np.float64, copy=True)
    S_prev = np.zeros((T, V, K))
    qh, kh = np.zeros((T, K)), np.zeros((T, K))
    nq, nk, x, lam, al, be = (np.zeros(T) for _ in range(6))
    out = np.zeros((T, V))
    for t in range(T):
        nq[t] = np.sqrt(q[t] @ q[t] + EPS)
        nk[t] = np.sqrt(k[t] @ k[t] + EPS)
        qh[t], kh[t] = q[t] / nq[t], k[t] / nk[t]
        x[t] = a[t] + float(dt_bias)
        lam[t] = -eA * _softplus(x[t])
        al[t] = np.exp(lam[t])
        be[t] = _sigmoid(b[t])
        S_prev[t] = S
        u = S @ kh[t]
        S = al[t] * S + np.outer(be[t] * (v[t] - al[t] * u), kh[t])
        out[t] = scale * (S @ qh[t])
    S_final = S

    # backward sweep
    G = np.array(d_state, dtype=np.float64, copy=True)
    dq, dk, dv = np.zeros((T, K)), np.zeros((T, K)), np.zeros((T, V))
    da, db = np.zeros(T), np.zeros(T)
    dA_log = ddt_bias = 0.0
    for t in range(T - 1, -1, -1):
        Sp = S_prev[t]
        u = Sp @ kh[t]
        delta = be[t] * (v[t] - al[t] * u)
        St = al[t] * Sp + np.outer(delta, kh[t])
        # o_t = scale S_t q^_t
        G = G + scale * np.outer(d_out[t], qh[t])
        dqh = scale * (St.T @ d_out[t])
        # S_t = alpha S_{t-1} + delta k^^T
        ddelta = G @ kh[t]
        dkh = G.T @ delta
        dal = float(np.sum(G * Sp))
        # delta = beta (v - alpha u)
        dbe = float(ddelta @ (v[t] - al[t] * u))
        dv[t] = be[t] * ddelta
        du = -al[t] * be[t] * ddelta
        dal += -be[t] * float(ddelta @ u)
        # u = S_{t-1} k^
        dkh = dkh + Sp.T @ du
        G = al[t] * G + np.outer(du, kh[t])
        # gates: alpha = exp(lam), lam = -exp(A_log) softplus(x), x = a + dt_bias; beta = sigmoid(b)
        dlam = dal * al[t]
        dA_log += dlam * lam[t]
        dx = dlam * (-eA) * _sigmoid(x[t])
        da[t] = dx
        ddt_bias += dx
        db[t] = dbe * be[t] * (1.0 - be[t])
        # normalisation
        dq[t] = dqh / nq[t] - q[t] * (q[t] @ dqh) / nq[t] ** 3
        dk[t] = dkh / nk[t] - k[t] * (k[t] @ dkh) / nk[t] ** 3
    return dict(dq=dq, dk=dk, dv=dv, da=da, db=db, dA_log=dA_log, ddt_bias=ddt_bias, dS0=G,
                out=out, S_final=S_final)


def gdn_backward(q, k, v, a, b, A_log, dt_bias, state_pool, cache_indices, cu_seqlens, d_out, d_state,
                 scale: float = 1.0):
    """Gradients of a whole call (the layout of gdn_extend_chunkwise), fp64.

    q, k: [T, H, K]; v, d_out: [T, HV, V]; a, b: [T, HV]; A_log, dt_bias: [HV];
    state_pool: [pool, HV, V, K] (the states before the call); cache_indices: [B]; cu_seqlens: [B+1];
    d_state: [B, HV, V, K], the gradient of each sequence's final state.
    Returns dq, dk [T, H, K], dv [T, HV, V], da, db [T, HV], dA_log, ddt_bias [HV] and
    d_state_pool [pool, HV, V, K] (zero for slots the call does not touch).
    """
    f = lambda x: np.asarray(x.double().numpy() if hasattr(x, "double") else x, dtype=np.float64)
    q, k, v, a, b = f(q), f(k), f(v), f(a), f(b)
    A_log, dt_bias, pool = f(A_log), f(dt_bias), f(state_pool)
    d_out, d_state = f(d_out), f(d_state)
    idx = np.asarray(cache_indices.numpy() if hasattr(cache_indices, "numpy") else cache_indices, dtype=np.int64)
    cu = np.asarray(cu_seqlens.numpy() if hasattr(cu_seqlens, "numpy") else cu_seqlens, dtype=np.int64)
    T, H, K = k.shape
    HV = v.shape[1]
    if HV % H != 0:
        raise ValueError("HV must be a multiple of H")
    r = HV // H
    res = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v), da=np.zeros_like(a),
               db=np.zeros_like(b), dA_log=np.zeros(HV), ddt_bias=np.zeros(HV),
               d_state_pool=np.zeros_like(pool))
    for s in range(len(idx)):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        for hv in range(HV):
            h = hv // r
            g = chain_backward(q[t0:t1, h], k[t0:t1, h], v[t0:t1, hv], a[t0:t1, hv], b[t0:t1, hv],
                               A_log[hv], dt_bias[hv], pool[idx[s], hv], d_out[t0:t1, hv], d_state[s, hv],
                               scale)
            res["dq"][t0:t1, h] += g["dq"]
            res["dk"][t0:t1, h] += g["dk"]
            res["dv"][t0:t1, hv] = g["dv"]
            res["da"][t0:t1, hv] = g["da"]
            res["db"][t0:t1, hv] = g["db"]
            res["dA_log"][hv] += g["dA_log"]
            res["ddt_bias"][hv] += g["ddt_bias"]
            res["d_state_pool"][idx[s], hv] = g["dS0"]
    return res
