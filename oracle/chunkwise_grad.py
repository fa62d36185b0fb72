"""Oracle O4: the chunkwise WY forward in fp64 PyTorch (CPU), differentiated by autograd; and the same
backward written out explicitly (numpy fp64), the algorithm a chunkwise backward kernel runs.

TEST INFRASTRUCTURE ONLY (like everything under ``oracle/``): the GPU library never imports it.

It serves the backward pass in two ways. Its gradients pin O3 (``oracle/backward.py``) by a second route:
a different forward algorithm (the chunkwise WY form instead of the token recurrence) and a different
differentiation (autograd instead of the hand-applied chain rule). Its per-chunk intermediates (W<-, U~,
U, the state entering each chunk) keep their gradients, which are the references a chunkwise backward
kernel needs stage by stage.

Forward per chunk, as in O2 (:func:`oracle.chunkwise.chunkwise_forward`), from raw inputs:
    q^ = q / sqrt(|q|^2 + 1e-6), k^ likewise; log alpha = -exp(A_log) softplus(a + dt_bias); beta = sigmoid(b)
    g = cumsum(log alpha) within the chunk, Gamma = exp(g_mu - g_nu) (mu >= nu), B = diag(beta)
    M = I + tril(B K^ K^^T, -1);  A = (Gamma . M^{-1}) B       ("Simple math to speed up GDN prefill",
                                                                sections "Reminder" and "Save one invert")
    W<- = A diag(e^g) K^,  U~ = A V,  U = U~ - W<- S^T
    O = scale (diag(e^g) Q^ S^T + (Gamma . tril(Q^ K^^T)) U)
    S <- e^{g_C} S + U^T diag(e^{g_C - g}) K^
"""

from __future__ import annotations

import numpy as np
import torch


def chunkwise_backward(q, k, v, a, b, A_log, dt_bias, S0, d_out, d_state, C: int = 64, scale: float = 1.0,
                       keep: bool = False):
    """One chain, fp64 torch on the CPU. q, k: [T, K]; v, d_out: [T, V]; a, b: [T]; A_log, dt_bias:
    scalars; S0, d_state: [V, K]. Returns the gradients of L = sum <d_out, o> + <d_state, S_final>
    (dq, dk, dv, da, db, dA_log, ddt_bias, dS0) and, with keep=True, per chunk the gradients of
    W<-, U~, U and of the state entering the chunk ("dW", "dUt", "dU", "dS_in": lists over chunks).
    """
    f = lambda x: torch.as_tensor(x, dtype=torch.float64).clone().requires_grad_(True)
    q, k, v, a, b, S0 = f(q), f(k), f(v), f(a), f(b), f(S0)
    A_log, dt_bias = f(float(A_log)), f(float(dt_bias))
    d_out = torch.as_tensor(d_out, dtype=torch.float64)
    d_state = torch.as_tensor(d_state, dtype=torch.float64)
    T = q.shape[0]
    qn = q / torch.sqrt((q * q).sum(-1, keepdim=True) + 1e-6)
    kn = k / torch.sqrt((k * k).sum(-1, keepdim=True) + 1e-6)
    x = a + dt_bias
    softplus = torch.clamp(x, min=0.0) + torch.log1p(torch.exp(-torch.abs(x)))
    log_alpha = -torch.exp(A_log) * softplus
    beta = 1.0 / (1.0 + torch.exp(-b))
    S = S0
    outs = []
    kept = {"W": [], "Ut": [], "U": [], "S_in": []}
    for s in range(0, T, C):
        e = min(s + C, T)
        n = e - s
        Q, Kc, Vc = qn[s:e], kn[s:e], v[s:e]
        g = torch.cumsum(log_alpha[s:e], 0)
        Gam = torch.tril(torch.exp(g[:, None] - g[None, :]))
        M = torch.eye(n, dtype=torch.float64) + torch.tril(beta[s:e, None] * (Kc @ Kc.T), -1)
        A = (Gam * torch.linalg.inv(M)) * beta[s:e][None, :]
        W = A @ (torch.exp(g)[:, None] * Kc)
        Ut = A @ Vc
        if keep:
            S.retain_grad() if S.requires_grad and not S.is_leaf else None
            W.retain_grad()
            Ut.retain_grad()
            kept["S_in"].append(S)
        U = Ut - W @ S.T
        if keep:
            U.retain_grad()
            kept["W"].append(W)
            kept["Ut"].append(Ut)
            kept["U"].append(U)
        outs.append(scale * (torch.exp(g)[:, None] * (Q @ S.T) + (Gam * (Q @ Kc.T)) @ U))
        S = torch.exp(g[-1]) * S + U.T @ (torch.exp(g[-1] - g)[:, None] * Kc)
    out = torch.cat(outs, 0) if outs else torch.zeros_like(d_out)
    L = (d_out * out).sum() + (d_state * S).sum()
    L.backward()
    res = dict(dq=q.grad.numpy(), dk=k.grad.numpy(), dv=v.grad.numpy(), da=a.grad.numpy(), db=b.grad.numpy(),
               dA_log=float(A_log.grad), ddt_bias=float(dt_bias.grad), dS0=S0.grad.numpy(),
               out=out.detach().numpy(), S_final=S.detach().numpy())
    if keep:
        res["dW"] = [t.grad.numpy() for t in kept["W"]]
        res["dUt"] = [t.grad.numpy() for t in kept["Ut"]]
        res["dU"] = [t.grad.numpy() for t in kept["U"]]
        res["dS_in"] = [t.grad.numpy() for t in kept["S_in"]]
    return res


def chunkwise_backward_explicit(q, k, v, a, b, A_log, dt_bias, S0, d_out, d_state, C: int = 64,
                                scale: float = 1.0):
    """The chunkwise backward written out (numpy fp64), as a kernel would run it.

    Forward sweep over the chunks (keeping each chunk's entering state), then a reverse sweep of the
    state gradient, the only sequential part:
        dU_c    = scale P^T dO_c + K->_c dS_out^T
        dS_in   = e^{g_C} dS_out + scale dO_c^T diag(e^g) Q^ - dU_c^T W<-_c
    and then, per chunk and independent of the others, the local gradients through P, W<-, U~, the
    inverse, the decays and the gates. Same inputs and outputs as :func:`chunkwise_backward`; with the
    per-chunk "dW", "dUt", "dU", "dS_in" lists always returned.
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    a, b = np.asarray(a, dtype=np.float64).reshape(-1), np.asarray(b, dtype=np.float64).reshape(-1)
    d_out = np.asarray(d_out, dtype=np.float64)
    T = q.shape[0]
    eA = float(np.exp(A_log))
    nq = np.sqrt(np.sum(q * q, 1) + 1e-6)
    nk = np.sqrt(np.sum(k * k, 1) + 1e-6)
    qn, kn = q / nq[:, None], k / nk[:, None]
    x = a + float(dt_bias)
    sig_x = 1.0 / (1.0 + np.exp(-x))
    la = -eA * (np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x))))
    beta = 1.0 / (1.0 + np.exp(-b))

    # forward sweep: per chunk factors and the entering state
    chunks = []
    S = np.array(S0, dtype=np.float64, copy=True)
    for s in range(0, T, C):
        e = min(s + C, T)
        n = e - s
        Q, Kc, Vc, bt = qn[s:e], kn[s:e], v[s:e], beta[s:e]
        g = np.cumsum(la[s:e])
        Gam = np.tril(np.exp(g[:, None] - g[None, :]))
        KK, QK = Kc @ Kc.T, Q @ Kc.T
        Minv = np.linalg.inv(np.eye(n) + np.tril(bt[:, None] * KK, -1))
        Z = Gam * Minv
        A = Z * bt[None, :]
        EK = np.exp(g)[:, None] * Kc
        W = A @ EK
        Ut = A @ Vc
        U = Ut - W @ S.T
        P = Gam * np.tril(QK)
        dec = np.exp(g[-1] - g)
        Kr = dec[:, None] * Kc                       # K-> = diag(e^{g_C - g}) K^
        chunks.append(dict(s=s, e=e, Q=Q, Kc=Kc, Vc=Vc, bt=bt, g=g, Gam=Gam, KK=KK, QK=QK, Minv=Minv, Z=Z, A=A,
                           EK=EK, W=W, U=U, P=P, dec=dec, Kr=Kr, S_in=S))
        S = np.exp(g[-1]) * S + U.T @ Kr

    # reverse sweep of the state gradient
    dS = np.array(d_state, dtype=np.float64, copy=True)
    for ch in reversed(chunks):
        dO = d_out[ch["s"]:ch["e"]]
        ch["dS_out"] = dS
        ch["dU"] = scale * ch["P"].T @ dO + ch["Kr"] @ dS.T
        dS = (np.exp(ch["g"][-1]) * dS + scale * dO.T @ (np.exp(ch["g"])[:, None] * ch["Q"])
              - ch["dU"].T @ ch["W"])
        ch["dS_in"] = dS
    dS0 = dS

    # per-chunk local gradients (independent across chunks)
    dqn, dkn, dv = np.zeros_like(qn), np.zeros_like(kn), np.zeros_like(v)
    dbeta, dla = np.zeros(T), np.zeros(T)
    for ch in chunks:
        s, e = ch["s"], ch["e"]
        dO = d_out[s:e]
        Q, Kc, Vc, bt, g, Gam, A, Z, Minv = (ch[n] for n in ("Q", "Kc", "Vc", "bt", "g", "Gam", "A", "Z", "Minv"))
        S_in, dU, dS_out, U = ch["S_in"], ch["dU"], ch["dS_out"], ch["U"]
        eg = np.exp(g)
        dg = np.zeros(e - s)
        dW = -dU @ S_in                              # U = U~ - W<- S^T
        ch["dW"], ch["dUt"] = dW, dU
        # O = scale (diag(e^g) Q S^T + P U)
        SQ = Q @ S_in.T                              # rows: S_in q_i
        dQ = scale * eg[:, None] * (dO @ S_in)
        dg += scale * eg * np.sum(dO * SQ, 1)
        dP = scale * np.tril(dO @ U.T)
        dGam = dP * np.tril(ch["QK"])
        dQ += (Gam * dP) @ Kc
        dK = (Gam * dP).T @ Q
        # S_out = e^{g_C} S_in + U^T K->
        dKr = U @ dS_out
        r = ch["dec"] * np.sum(dKr * Kc, 1)
        dK += ch["dec"][:, None] * dKr
        dgC = float(np.sum(r)) + np.exp(g[-1]) * float(np.sum(dS_out * S_in))
        dg -= r
        # U~ = A V, W<- = A diag(e^g) K^
        dA = dU @ Vc.T + dW @ ch["EK"].T
        dv[s:e] = A.T @ dU
        AtdW = A.T @ dW
        dK += eg[:, None] * AtdW
        dg += eg * np.sum(Kc * AtdW, 1)
        # A = (Gamma . M^{-1}) diag(beta)
        dZ = dA * bt[None, :]
        dbeta[s:e] += np.sum(dA * Z, 0)
        dGam += dZ * Minv
        dMinv = dZ * Gam
        # M^{-1}: dM = -M^{-T} dM^{-1} M^{-T}; M = I + tril(diag(beta) K K^T, -1)
        X = np.tril(-Minv.T @ dMinv @ Minv.T, -1)
        dbeta[s:e] += np.sum(X * ch["KK"], 1)
        dK += bt[:, None] * (X @ Kc) + X.T @ (bt[:, None] * Kc)
        # Gamma_ij = exp(g_i - g_j) on and below the diagonal
        wG = np.tril(dGam * Gam)
        dg += np.sum(wG, 1) - np.sum(wG, 0)
        dg[-1] += dgC
        # g = cumsum(log alpha) within the chunk
        dla[s:e] = np.cumsum(dg[::-1])[::-1]
        dqn[s:e], dkn[s:e] = dQ, dK

    # gates and normalisation
    dA_log = float(np.sum(dla * la))
    dx = dla * (-eA) * sig_x
    db = dbeta * beta * (1.0 - beta)
    dq = dqn / nq[:, None] - q * np.sum(q * dqn, 1)[:, None] / nq[:, None] ** 3
    dk = dkn / nk[:, None] - k * np.sum(k * dkn, 1)[:, None] / nk[:, None] ** 3
    return dict(dq=dq, dk=dk, dv=dv, da=dx, db=db, dA_log=dA_log, ddt_bias=float(np.sum(dx)), dS0=dS0,
                dW=[c["dW"] for c in chunks], dUt=[c["dUt"] for c in chunks], dU=[c["dU"] for c in chunks],
                dS_in=[c["dS_in"] for c in chunks])
