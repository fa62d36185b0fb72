"""Pins for the backward oracle (oracle/backward.py): its gradients against facts other than itself.

* Central finite differences of the loss L = sum <dO, o> + <dS, S_final>, where (o, S_final) come from
  O1's C recurrence (oracle.delta_rule) and O1's gate routines. The normalisation q / sqrt(|q|^2 + 1e-6)
  is written out here, as the pages define it.
* Exact linearity: o and S_final are affine in the initial state and in v, so a finite step in either
  changes L by exactly <gradient, step>.
* A closed form: with beta = 0 the state only decays.
* Teeth: plausible mistakes planted in a copy of the backward fail the finite-difference pin.
* A second route: autograd through the chunkwise WY form (O4, oracle/chunkwise_grad.py) gives the same
  gradients as O3's chain rule through the token recurrence, and O4's kept gradients of the state entering
  each chunk pass the exact-linearity check against O1.
"""

import numpy as np
import pytest

import oracle
from oracle import backward as bw


def _norm_rows(x):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + 1e-6)


def o1_chain(q, k, v, a, b, A_log, dt_bias, S0, scale=1.0):
    alpha = np.array([np.exp(oracle.log_alpha(at, A_log, dt_bias)) for at in a])
    beta = np.array([oracle.beta(bt) for bt in b])
    return oracle.delta_rule(_norm_rows(q), _norm_rows(k), v, alpha, beta, S0, scale=scale)


def o1_loss(p, d_out, d_state, scale=1.0):
    out, S = o1_chain(p["q"], p["k"], p["v"], p["a"], p["b"], float(p["A_log"]), float(p["dt_bias"]),
                      p["S0"], scale)
    return float(np.sum(d_out * out) + np.sum(d_state * S))


def random_chain(seed, T=4, K=3, V=2, a_mean=0.0, b_mean=0.0):
    rng = np.random.default_rng(seed)
    p = dict(q=rng.standard_normal((T, K)), k=rng.standard_normal((T, K)), v=rng.standard_normal((T, V)),
             a=rng.standard_normal(T) + a_mean, b=rng.standard_normal(T) + b_mean,
             A_log=np.array(np.log(rng.uniform(0.5, 3.0))), dt_bias=np.array(rng.uniform(-1.0, 1.0)),
             S0=0.5 * rng.standard_normal((V, K)))
    return p, rng.standard_normal((T, V)), rng.standard_normal((V, K))


GRAD_OF = {"q": "dq", "k": "dk", "v": "dv", "a": "da", "b": "db", "A_log": "dA_log", "dt_bias": "ddt_bias",
           "S0": "dS0"}


def finite_differences(loss, p, h=1e-5):
    fd = {}
    for name, x in p.items():
        g = np.zeros(np.shape(x))
        flat = np.array(x, dtype=np.float64).reshape(-1)
        for i in range(flat.size):
            pp = {n: np.array(y, dtype=np.float64, copy=True) for n, y in p.items()}
            for sgn in (1.0, -1.0):
                f2 = flat.copy()
                f2[i] += sgn * h
                pp[name] = f2.reshape(np.shape(x))
                g.reshape(-1)[i] += sgn * loss(pp) / (2 * h)
        fd[name] = g
    return fd


def assert_matches_fd(grads, fd, tol=1e-6):
    for name, g_fd in fd.items():
        g = np.asarray(grads[GRAD_OF[name]], dtype=np.float64).reshape(np.shape(g_fd))
        err = np.max(np.abs(g - g_fd))
        assert err <= tol * (1.0 + np.max(np.abs(g_fd))), (name, err, g, g_fd)


def chain_grads(p, d_out, d_state, scale=1.0, fn=bw.chain_backward):
    return fn(p["q"], p["k"], p["v"], p["a"], p["b"], float(p["A_log"]), float(p["dt_bias"]), p["S0"], d_out,
              d_state, scale)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("scale", [1.0, 0.7])
def test_chain_gradients_match_finite_differences(seed, scale):
    p, d_out, d_state = random_chain(seed)
    g = chain_grads(p, d_out, d_state, scale)
    assert_matches_fd(g, finite_differences(lambda pp: o1_loss(pp, d_out, d_state, scale), p))


@pytest.mark.parametrize("gates", [(3.0, -2.0), (-4.0, 3.0)])
def test_chain_gradients_at_gate_extremes(gates):
    """Strong decay with small beta, and almost no decay with beta near 1."""
    p, d_out, d_state = random_chain(10, a_mean=gates[0], b_mean=gates[1])
    g = chain_grads(p, d_out, d_state)
    assert_matches_fd(g, finite_differences(lambda pp: o1_loss(pp, d_out, d_state), p))


def test_forward_sweep_matches_o1():
    p, d_out, d_state = random_chain(20, T=9, K=5, V=4)
    g = chain_grads(p, d_out, d_state, 0.9)
    out, S = o1_chain(p["q"], p["k"], p["v"], p["a"], p["b"], float(p["A_log"]), float(p["dt_bias"]), p["S0"], 0.9)
    assert np.max(np.abs(g["out"] - out)) < 1e-12 and np.max(np.abs(g["S_final"] - S)) < 1e-12


@pytest.mark.parametrize("which", ["S0", "v"])
def test_exact_linearity_in_state_and_values(which):
    """L is affine in S0 and in v: a finite step of either changes L by exactly <gradient, step>."""
    p, d_out, d_state = random_chain(30, T=12, K=6, V=5)
    g = chain_grads(p, d_out, d_state)
    step = np.random.default_rng(31).standard_normal(np.shape(p[which]))
    p2 = dict(p, **{which: p[which] + step})
    change = o1_loss(p2, d_out, d_state) - o1_loss(p, d_out, d_state)
    predicted = float(np.sum(g[GRAD_OF[which]] * step))
    assert abs(change - predicted) <= 1e-10 * (1.0 + abs(change))


def test_pure_decay_closed_form():
    """beta = 0 (b very negative): S_t = (prod alpha) S0, so dS0 = (prod_t alpha_t) dS_T +
    scale sum_t (prod_{s<=t} alpha_s) dO_t q^_t^T, and v and k get no gradient."""
    p, d_out, d_state = random_chain(40, T=6, K=4, V=3)
    p["b"] = np.full(6, -80.0)
    g = chain_grads(p, d_out, d_state, 0.5)
    alpha = np.array([np.exp(oracle.log_alpha(at, float(p["A_log"]), float(p["dt_bias"]))) for at in p["a"]])
    cum = np.cumprod(alpha)
    qn = _norm_rows(p["q"])
    expect = cum[-1] * d_state + 0.5 * sum(cum[t] * np.outer(d_out[t], qn[t]) for t in range(6))
    assert np.max(np.abs(g["dS0"] - expect)) < 1e-13
    assert np.max(np.abs(g["dv"])) < 1e-30 and np.max(np.abs(g["dk"])) < 1e-30


def test_full_call_layout_gqa_varlen_and_empty_sequence():
    """gdn_backward over a call: H=1, HV=2 (both value heads read one q/k head), three sequences of
    lengths 3, 0, 2 in slots 2, 0, 3 of a 4-slot pool; finite differences of the whole call's loss."""
    rng = np.random.default_rng(50)
    T, H, HV, K, V, pool_n = 5, 1, 2, 3, 2, 4
    cu = np.array([0, 3, 3, 5])
    idx = np.array([2, 0, 3])
    p = dict(q=rng.standard_normal((T, H, K)), k=rng.standard_normal((T, H, K)), v=rng.standard_normal((T, HV, V)),
             a=rng.standard_normal((T, HV)), b=rng.standard_normal((T, HV)),
             A_log=np.log(rng.uniform(0.5, 3.0, HV)), dt_bias=rng.uniform(-1, 1, HV),
             pool=0.5 * rng.standard_normal((pool_n, HV, V, K)))
    d_out = rng.standard_normal((T, HV, V))
    d_state = rng.standard_normal((len(idx), HV, V, K))

    def loss(pp):
        L = 0.0
        for s in range(len(idx)):
            t0, t1 = cu[s], cu[s + 1]
            for hv in range(HV):
                if t1 == t0:
                    S = pp["pool"][idx[s], hv]
                    L += float(np.sum(d_state[s, hv] * S))
                    continue
                out, S = o1_chain(pp["q"][t0:t1, 0], pp["k"][t0:t1, 0], pp["v"][t0:t1, hv], pp["a"][t0:t1, hv],
                                  pp["b"][t0:t1, hv], float(pp["A_log"][hv]), float(pp["dt_bias"][hv]),
                                  pp["pool"][idx[s], hv])
                L += float(np.sum(d_out[t0:t1, hv] * out) + np.sum(d_state[s, hv] * S))
        return L

    g = bw.gdn_backward(p["q"], p["k"], p["v"], p["a"], p["b"], p["A_log"], p["dt_bias"], p["pool"], idx, cu,
                        d_out, d_state)
    fd = finite_differences(loss, p)
    names = {"q": "dq", "k": "dk", "v": "dv", "a": "da", "b": "db", "A_log": "dA_log", "dt_bias": "ddt_bias",
             "pool": "d_state_pool"}
    for n, gn in names.items():
        err = np.max(np.abs(g[gn] - fd[n]))
        assert err <= 1e-6 * (1.0 + np.max(np.abs(fd[n]))), (n, err)
    assert np.all(g["d_state_pool"][1] == 0.0)  # slot 1 is not touched by the call
    assert np.array_equal(g["d_state_pool"][0], d_state[1])  # the empty sequence passes its gradient through


# --------------------------------------------------------------------------- pins have teeth

def _mutant_backward(kind):
    """Plausible mistakes planted in a copy of the chain backward (CPU only)."""
    def run(q, k, v, a, b, A_log, dt_bias, S0, d_out, d_state, scale=1.0):
        T = len(q)
        eA = np.exp(A_log)
        sp = lambda x: max(x, 0.0) + np.log1p(np.exp(-abs(x)))
        sg = lambda x: 1.0 / (1.0 + np.exp(-x))
        nq = np.sqrt(np.sum(q * q, 1) + 1e-6)
        nk = np.sqrt(np.sum(k * k, 1) + 1e-6)
        qh, kh = q / nq[:, None], k / nk[:, None]
        x = a + dt_bias
        lam = np.array([-eA * sp(xi) for xi in x])
        al, be = np.exp(lam), sg(b)
        Ss = [np.array(S0, dtype=np.float64)]
        for t in range(T):
            S = Ss[-1]
            Ss.append(al[t] * S + np.outer(be[t] * (v[t] - al[t] * (S @ kh[t])), kh[t]))
        G = np.array(d_state, dtype=np.float64)
        res = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v), da=np.zeros(T), db=np.zeros(T),
                   dA_log=0.0, ddt_bias=0.0)
        for t in range(T - 1, -1, -1):
            Sp, St = Ss[t], Ss[t + 1]
            u = Sp @ kh[t]
            delta = be[t] * (v[t] - al[t] * u)
            G = G + scale * np.outer(d_out[t], qh[t])
            dqh = scale * ((Sp if kind == "read_before_write" else St).T @ d_out[t])
            ddelta = G @ kh[t]
            dkh = G.T @ delta
            dal = np.sum(G * Sp) - be[t] * (ddelta @ u)
            dbe = ddelta @ (v[t] - al[t] * u)
            res["dv"][t] = be[t] * ddelta
            du = -al[t] * be[t] * ddelta
            dkh = dkh + Sp.T @ du
            G = al[t] * G if kind == "dropped_erase" else al[t] * G + np.outer(du, kh[t])
            dlam = dal * al[t]
            res["dA_log"] += dlam * lam[t]
            dx = dlam * (-eA) * (sp(x[t]) if kind == "softplus_for_sigmoid" else sg(x[t]))
            res["da"][t] = dx
            res["ddt_bias"] += dx
            res["db"][t] = dbe * be[t] * (1.0 - be[t])
            if kind == "no_norm_jacobian":
                res["dq"][t], res["dk"][t] = dqh / nq[t], dkh / nk[t]
            else:
                res["dq"][t] = dqh / nq[t] - q[t] * (q[t] @ dqh) / nq[t] ** 3
                res["dk"][t] = dkh / nk[t] - k[t] * (k[t] @ dkh) / nk[t] ** 3
        res["dS0"] = G
        return res
    return run


@pytest.mark.parametrize("kind", ["read_before_write", "dropped_erase", "softplus_for_sigmoid", "no_norm_jacobian"])
def test_pins_catch_planted_backward_mistakes(kind):
    p, d_out, d_state = random_chain(0)
    fd = finite_differences(lambda pp: o1_loss(pp, d_out, d_state), p)
    assert_matches_fd(chain_grads(p, d_out, d_state, fn=_mutant_backward("none")), fd)  # the unplanted copy passes
    with pytest.raises(AssertionError):
        assert_matches_fd(chain_grads(p, d_out, d_state, fn=_mutant_backward(kind)), fd)


# --------------------------------------------------------------------------- O4: autograd of the chunkwise form

from oracle import chunkwise_grad as cg  # noqa: E402


@pytest.mark.parametrize("C", [16, 64])
@pytest.mark.parametrize("gates", [(0.0, 0.0), (3.0, -2.0), (-4.0, 3.0)])
def test_autograd_of_chunkwise_form_equals_chain_rule_of_recurrence(C, gates):
    """Two independent routes to the same gradients: O3 (hand chain rule, token recurrence) and O4
    (autograd, chunkwise WY form with one inverse), over several chunks and a ragged tail."""
    p, d_out, d_state = random_chain(60, T=150, K=6, V=5, a_mean=gates[0], b_mean=gates[1])
    g3 = chain_grads(p, d_out, d_state, 0.8)
    g4 = cg.chunkwise_backward(p["q"], p["k"], p["v"], p["a"], p["b"], float(p["A_log"]), float(p["dt_bias"]),
                               p["S0"], d_out, d_state, C=C, scale=0.8)
    for name in ("dq", "dk", "dv", "da", "db", "dS0"):
        ref = np.asarray(g3[name])
        assert np.max(np.abs(g4[name] - ref)) <= 1e-9 * (1.0 + np.max(np.abs(ref))), name
    for name in ("dA_log", "ddt_bias"):
        assert abs(g4[name] - g3[name]) <= 1e-9 * (1.0 + abs(g3[name])), name


def test_chunk_boundary_state_gradients_by_exact_linearity():
    """The gradient of the state entering chunk c, kept by O4, checked against O1: the tail of the
    loss (tokens from c C on, and the final state) is affine in that state."""
    C, T = 16, 70
    p, d_out, d_state = random_chain(61, T=T, K=5, V=4)
    g4 = cg.chunkwise_backward(p["q"], p["k"], p["v"], p["a"], p["b"], float(p["A_log"]), float(p["dt_bias"]),
                               p["S0"], d_out, d_state, C=C, keep=True)
    rng = np.random.default_rng(62)
    for c in range(len(g4["dS_in"])):
        t0 = c * C
        head = dict(p, q=p["q"][:t0], k=p["k"][:t0], v=p["v"][:t0], a=p["a"][:t0], b=p["b"][:t0])
        S_c = p["S0"] if t0 == 0 else o1_chain(head["q"], head["k"], head["v"], head["a"], head["b"],
                                               float(p["A_log"]), float(p["dt_bias"]), p["S0"])[1]
        tail = dict(p, q=p["q"][t0:], k=p["k"][t0:], v=p["v"][t0:], a=p["a"][t0:], b=p["b"][t0:])
        step = rng.standard_normal(S_c.shape)
        change = (o1_loss(dict(tail, S0=S_c + step), d_out[t0:], d_state)
                  - o1_loss(dict(tail, S0=S_c), d_out[t0:], d_state))
        assert abs(change - float(np.sum(g4["dS_in"][c] * step))) <= 1e-10 * (1.0 + abs(change)), c
    # U = U~ - W<- S^T: the kept factor gradients follow from dU and the entering state
    for c in range(len(g4["dU"])):
        assert np.allclose(g4["dUt"][c], g4["dU"][c], rtol=0, atol=1e-13)


@pytest.mark.parametrize("C", [16, 64])
@pytest.mark.parametrize("gates", [(0.0, 0.0), (3.0, -2.0), (-4.0, 3.0)])
def test_explicit_chunkwise_backward_stage_by_stage(C, gates):
    """The chunkwise backward written out (reverse sweep of the state gradient, then per-chunk local
    gradients) equals autograd of the chunkwise form in every per-chunk intermediate and every input
    gradient, and hence O3."""
    p, d_out, d_state = random_chain(70, T=150, K=6, V=5, a_mean=gates[0], b_mean=gates[1])
    args = (p["q"], p["k"], p["v"], p["a"], p["b"], float(p["A_log"]), float(p["dt_bias"]), p["S0"], d_out,
            d_state)
    g4 = cg.chunkwise_backward(*args, C=C, scale=0.8, keep=True)
    gx = cg.chunkwise_backward_explicit(*args, C=C, scale=0.8)
    for name in ("dW", "dUt", "dU", "dS_in"):
        for c, (x, y) in enumerate(zip(gx[name], g4[name])):
            assert np.max(np.abs(x - y)) <= 1e-11 * (1.0 + np.max(np.abs(y))), (name, c)
    g3 = chain_grads(p, d_out, d_state, 0.8)
    for name in ("dq", "dk", "dv", "da", "db", "dS0", "dA_log", "ddt_bias"):
        ref = np.asarray(g3[name])
        assert np.max(np.abs(np.asarray(gx[name]) - ref)) <= 1e-9 * (1.0 + np.max(np.abs(ref))), name
