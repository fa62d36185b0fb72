"""Oracle O4: the chunkwise WY forward in fp64 PyTorch (CPU), differentiated by autograd.

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
