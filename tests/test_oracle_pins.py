"""Pins for the oracle: checks against facts the pages and the mathematics fix.

Nothing here compares the oracle with itself. Each test checks it against one of:
a worked example (tests/golden), a closed form, a textbook/library routine, an
invariant of the recurrence, brute force on tiny inputs, or an independent
algorithm that the pages say reaches the same result (the chunkwise WY form).
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import chunkwise as cw
from gated_deltanet_chunkwise_gdn_gb300 import workloads as wl


def _unit_rows(rng, T, K):
    x = rng.standard_normal((T, K))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def _random_chain(rng, T, K, V, strong=True):
    qn, kn = _unit_rows(rng, T, K), _unit_rows(rng, T, K)
    v = rng.standard_normal((T, V))
    log_alpha = -rng.uniform(0.0, 1.5 if strong else 0.05, T)
    beta = rng.uniform(0.0, 1.0, T)
    S0 = 0.3 * rng.standard_normal((V, K))
    return qn, kn, v, log_alpha, beta, S0


# --------------------------------------------------------------------------- widening, gates

def test_bf16_widening_matches_torch_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_bits_to_double(int(b)) for b in bits[::97]])
    r = ref[::97]
    both_nan = np.isnan(got) & np.isnan(r)
    assert np.array_equal(got[~both_nan], r[~both_nan])


def test_fp16_widening_matches_numpy_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_bits_to_double(int(b)) for b in bits])
    both_nan = np.isnan(got) & np.isnan(ref)
    assert np.array_equal(got[~both_nan], ref[~both_nan])


def test_gates_match_library_routines():
    from scipy.special import expit
    xs = np.concatenate([np.linspace(-60, 60, 241), [-745.0, -30.5, 1e-9, 30.5, 700.0]])
    for x in xs:
        # softplus(x) = log(1 + e^x) = logaddexp(0, x)
        assert oracle.softplus(x) == pytest.approx(np.logaddexp(0.0, x), rel=1e-15, abs=1e-300)
        assert oracle.beta(x) == pytest.approx(expit(x), rel=1e-15, abs=1e-300)
    rng = np.random.default_rng(0)
    for _ in range(200):
        a, A_log, dt = rng.normal() * 3, np.log(rng.uniform(1, 16)), np.log(np.expm1(rng.uniform(1e-3, 0.1)))
        want = -np.exp(A_log) * np.logaddexp(0.0, a + dt)
        assert oracle.log_alpha(a, A_log, dt) == pytest.approx(want, rel=1e-14)
    # decay is a contraction for every finite input: alpha in (0, 1]
    assert oracle.log_alpha(-1e3, 0.0, 0.0) <= 0.0
    assert oracle.log_alpha(5.0, float("-inf"), 0.0) == 0.0  # A_log = -inf: no decay


# --------------------------------------------------------------------------- the recurrence

def test_worked_two_token_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "two_token_k2.json")))
    out, S = oracle.delta_rule(np.array(g["q"]), np.array(g["k"]), np.array(g["v"]),
                               np.array(g["alpha"]), np.array(g["beta"]), np.array(g["S0"]))
    np.testing.assert_allclose(out, np.array(g["out"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(S, np.array(g["S_final"]), rtol=0, atol=1e-14)


@pytest.mark.parametrize("T", [1, 2, 5, 6])
def test_brute_force_transition_matrices(T):
    rng = np.random.default_rng(T)
    qn, kn, v, la, beta, S0 = _random_chain(rng, T, 4, 4)
    S0 = rng.standard_normal((4, 4))  # non-symmetric, so a transposed S is caught
    out, S = oracle.delta_rule(qn, kn, v, np.exp(la), beta, S0)
    out_bf, S_bf = cw.brute_force(qn, kn, v, np.exp(la), beta, S0)
    np.testing.assert_allclose(out, out_bf, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S, S_bf, rtol=0, atol=1e-13)


def test_pure_decay_when_beta_is_zero():
    """beta = 0: S_T = exp(sum log alpha) S0 and o_t = exp(sum_{<=t} log alpha) S0 q_t."""
    rng = np.random.default_rng(1)
    T, K, V = 40, 8, 6
    qn, kn, v, la, _, S0 = _random_chain(rng, T, K, V)
    out, S = oracle.delta_rule(qn, kn, v, np.exp(la), np.zeros(T), S0)
    cum = np.cumsum(la)
    np.testing.assert_allclose(S, np.exp(cum[-1]) * S0, rtol=1e-13, atol=0)
    np.testing.assert_allclose(out, np.exp(cum)[:, None] * (qn @ S0.T), rtol=1e-12, atol=1e-300)


def test_delta_writes_with_orthonormal_keys_and_no_decay():
    """alpha = 1, orthonormal keys: S_n = S0 + sum_i beta_i (v_i - S0 k_i) k_i^T,
    and every prefix obeys the same formula."""
    rng = np.random.default_rng(2)
    K, V, n = 8, 5, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    kn = Qm[:, :n].T.copy()
    qn = _unit_rows(rng, n, K)
    v = rng.standard_normal((n, V))
    beta = rng.uniform(0, 1, n)
    S0 = rng.standard_normal((V, K))
    out, S = oracle.delta_rule(qn, kn, v, np.ones(n), beta, S0)
    St = S0.copy()
    for t in range(n):
        St = St + beta[t] * np.outer(v[t] - S0 @ kn[t], kn[t])
        np.testing.assert_allclose(out[t], St @ qn[t], rtol=0, atol=1e-13)
    np.testing.assert_allclose(S, St, rtol=0, atol=1e-13)


def test_perfect_recall_and_read_after_write():
    """alpha = beta = 1, S0 = 0, orthonormal keys: reading with q = k_j returns v_j,
    including at the token that wrote it (the token sees its own write)."""
    rng = np.random.default_rng(3)
    K, V, n = 6, 4, 6
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    kn = Qm[:, :n].T.copy()
    v = rng.standard_normal((n, V))
    out, S = oracle.delta_rule(kn, kn, v, np.ones(n), np.ones(n), np.zeros((V, K)))
    np.testing.assert_allclose(out, v, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S @ kn.T, v.T, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S, v.T @ kn, rtol=0, atol=1e-13)  # linear attention, beta=1


def test_linearity_in_state_and_values():
    rng = np.random.default_rng(4)
    T, K, V = 30, 8, 8
    qn, kn, v, la, beta, S0 = _random_chain(rng, T, K, V)
    v2, S02 = rng.standard_normal((T, V)), rng.standard_normal((V, K))
    o1, s1 = oracle.delta_rule(qn, kn, v, np.exp(la), beta, S0)
    o2, s2 = oracle.delta_rule(qn, kn, v2, np.exp(la), beta, S02)
    o3, s3 = oracle.delta_rule(qn, kn, v + 2 * v2, np.exp(la), beta, S0 + 2 * S02)
    np.testing.assert_allclose(o3, o1 + 2 * o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s3, s1 + 2 * s2, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- chunkwise algebra

@pytest.mark.parametrize("C", [1, 2, 4, 8, 64])
@pytest.mark.parametrize("inverses", [1, 2])
def test_chunkwise_wy_equals_recurrence(C, inverses):
    """The chunkwise WY form computes what sequential application gives."""
    rng = np.random.default_rng(10 + C)
    T, K, V = 150, 16, 12
    qn, kn, v, la, beta, S0 = _random_chain(rng, T, K, V)
    o_ref, s_ref = oracle.delta_rule(qn, kn, v, np.exp(la), beta, S0)
    o, s = cw.chunkwise_forward(qn, kn, v, la, beta, S0, C, inverses=inverses)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-11)
    np.testing.assert_allclose(s, s_ref, rtol=0, atol=1e-11)


def test_one_inverse_identity():
    """N^{-1} = G M^{-1} G^{-1} ("Save one invert"), at C = 64 and C = 128."""
    rng = np.random.default_rng(5)
    for C in (64, 128):
        kn = _unit_rows(rng, C, 128)
        la = -rng.uniform(0.0, 0.4, C)
        beta = rng.uniform(0, 1, C)
        direct, one = cw.n_inverse_two_ways(kn, la, beta)
        assert np.max(np.abs(direct - one)) < 1e-13
        # and it really is the inverse of N
        Gam = cw.decay_matrix(np.cumsum(la))
        N = np.eye(C) + np.tril(beta[:, None] * (Gam * (kn @ kn.T)), -1)
        assert np.max(np.abs(N @ one - np.eye(C))) < 1e-12


def test_page3_gamma_form_on_mild_gates_and_overflow_on_strong():
    rng = np.random.default_rng(6)
    T, K, V = 130, 16, 8
    qn, kn, v, la, beta, S0 = _random_chain(rng, T, K, V, strong=False)
    o_ref, s_ref = oracle.delta_rule(qn, kn, v, np.exp(la), beta, S0)
    o, s = cw.chunkwise_page3(qn, kn, v, la, beta, S0, 64)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-10)
    np.testing.assert_allclose(s, s_ref, rtol=0, atol=1e-10)
    # fp32 1/gamma overflows once a chunk's sum of log alpha is below about -88
    la_strong = np.full(128, -1.0)
    assert not np.isfinite(np.float32(1.0) / np.exp(np.cumsum(la_strong)).astype(np.float32)).all()


def test_page3_literal_w_line_is_not_m_inverse_bk():
    rng = np.random.default_rng(7)
    C, K = 8, 16
    kn = _unit_rows(rng, C, K)
    beta = rng.uniform(0.2, 1.0, C)
    W = np.linalg.inv(cw.gram_factors(kn, beta)) @ (beta[:, None] * kn)
    np.testing.assert_allclose(cw.wy_rows(kn, beta), W, rtol=0, atol=1e-13)
    lit = cw.page3_w_rows_literal(kn, beta)
    np.testing.assert_allclose(lit[:2], W[:2], rtol=0, atol=1e-13)  # rows 1-2 agree
    assert np.max(np.abs(lit[2:] - W[2:])) > 1e-6                   # from row 3 on they differ


# --------------------------------------------------------------------------- the full call

def _small_inputs(lengths, H, HV, K, V, seed, **kw):
    w = wl.custom("pin", lengths, H=H, HV=HV, K=K, V=V, chunk_size=64, seed=seed, **kw)
    return wl.make_inputs(w)


def test_full_call_matches_explicit_chain():
    """gdn_forward = gates + normalisation + delta_rule on each (seq, hv) chain."""
    d = _small_inputs([5, 9], H=2, HV=4, K=8, V=6, seed=11)
    res = oracle.gdn_forward(**{k: d[k] for k in d if k != "chunk_size"})
    cu, idx = d["cu_seqlens"].numpy(), d["cache_indices"].numpy()
    for i, (s, hv) in enumerate(res.chains):
        h = hv // 2
        t0, t1 = cu[s], cu[s + 1]
        q = d["q"][t0:t1, h].double().numpy()
        k = d["k"][t0:t1, h].double().numpy()
        qn = q / np.sqrt((q * q).sum(1, keepdims=True) + 1e-6)
        kn = k / np.sqrt((k * k).sum(1, keepdims=True) + 1e-6)
        a = d["a"][t0:t1, hv].double().numpy()
        la = -np.exp(float(d["A_log"][hv])) * np.logaddexp(0.0, a + float(d["dt_bias"][hv]))
        beta = 1.0 / (1.0 + np.exp(-d["b"][t0:t1, hv].double().numpy()))
        S0 = d["state_pool"][idx[s], hv].double().numpy()
        o, S = cw.brute_force(qn, kn, d["v"][t0:t1, hv].double().numpy(), np.exp(la), beta, S0)
        np.testing.assert_allclose(res.chain_output(i), o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(res.states[i], S, rtol=0, atol=1e-12)


def test_gqa_equals_repeated_heads():
    """Value head hv reads q/k head hv // (HV/H): HV = 2H equals q/k repeated per head."""
    d = _small_inputs([20, 7], H=2, HV=4, K=8, V=8, seed=12)
    args = {k: d[k] for k in d if k != "chunk_size"}
    r1 = oracle.gdn_forward(**args)
    args2 = dict(args, q=d["q"].repeat_interleave(2, dim=1), k=d["k"].repeat_interleave(2, dim=1))
    r2 = oracle.gdn_forward(**args2)
    np.testing.assert_array_equal(r1.out, r2.out)
    np.testing.assert_array_equal(r1.states, r2.states)
    args3 = dict(args, q=d["q"].repeat(1, 2, 1), k=d["k"].repeat(1, 2, 1))  # the other mapping
    assert np.max(np.abs(oracle.gdn_forward(**args3).out - r1.out)) > 1e-3


def test_varlen_equals_per_sequence_calls():
    d = _small_inputs([13, 1, 40], H=1, HV=2, K=8, V=4, seed=13)
    args = {k: d[k] for k in d if k != "chunk_size"}
    whole = oracle.gdn_forward(**args)
    cu = d["cu_seqlens"]
    for s in range(3):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        one = oracle.gdn_forward(
            q=d["q"][t0:t1], k=d["k"][t0:t1], v=d["v"][t0:t1], a=d["a"][t0:t1], b=d["b"][t0:t1],
            A_log=d["A_log"], dt_bias=d["dt_bias"], state_pool=d["state_pool"],
            cache_indices=d["cache_indices"][s:s + 1], cu_seqlens=torch.tensor([0, t1 - t0]))
        for hv in range(2):
            i = s * 2 + hv
            np.testing.assert_array_equal(whole.chain_output(i), one.chain_output(hv))
            np.testing.assert_array_equal(whole.states[i], one.states[hv])


def test_zero_length_sequence_keeps_state_and_split_calls_continue():
    d = _small_inputs([0, 30], H=1, HV=1, K=8, V=8, seed=14)
    args = {k: d[k] for k in d if k != "chunk_size"}
    r = oracle.gdn_forward(**args)
    np.testing.assert_array_equal(r.states[0], d["state_pool"][d["cache_indices"][0], 0].double().numpy())
    # split the 30-token sequence in two calls, carrying the state
    slot = int(d["cache_indices"][1])
    first = oracle.gdn_forward(**dict(args, q=d["q"][:12], k=d["k"][:12], v=d["v"][:12], a=d["a"][:12],
                                      b=d["b"][:12], cache_indices=d["cache_indices"][1:],
                                      cu_seqlens=torch.tensor([0, 12])))
    pool2 = d["state_pool"].clone()
    pool2[slot, 0] = torch.from_numpy(first.states[0]).float()
    second = oracle.gdn_forward(**dict(args, q=d["q"][12:], k=d["k"][12:], v=d["v"][12:], a=d["a"][12:],
                                       b=d["b"][12:], state_pool=pool2, cache_indices=d["cache_indices"][1:],
                                       cu_seqlens=torch.tensor([0, 18])))
    whole = r.chain_output(1)
    np.testing.assert_allclose(whole[:12], first.out, rtol=0, atol=0)
    np.testing.assert_allclose(whole[12:], second.out, rtol=0, atol=1e-6)  # fp32 state hand-over


def test_normalisation_makes_q_and_k_scale_free():
    d = _small_inputs([33], H=1, HV=1, K=16, V=8, seed=15)
    args = {k: d[k] for k in d if k != "chunk_size"}
    r1 = oracle.gdn_forward(**args)
    r2 = oracle.gdn_forward(**dict(args, q=d["q"] * 4, k=d["k"] * 0.25))  # powers of 2: exact in bf16
    np.testing.assert_allclose(r2.out, r1.out, rtol=0, atol=2e-6 * np.abs(r1.out).max())
    zero_q = oracle.gdn_forward(**dict(args, q=torch.zeros_like(d["q"])))
    assert np.all(zero_q.out == 0.0)


def test_oracle_rejects_bad_slots():
    d = _small_inputs([3, 4], H=1, HV=1, K=4, V=4, seed=16, pool_size=4)
    args = {k: d[k] for k in d if k != "chunk_size"}
    with pytest.raises(ValueError):
        oracle.gdn_forward(**dict(args, cache_indices=torch.tensor([1, 1])))
    with pytest.raises(ValueError):
        oracle.gdn_forward(**dict(args, cache_indices=torch.tensor([0, 4])))


# --------------------------------------------------------------------------- pins have teeth

def _mutant(kind):
    """Plausible mistakes planted in a copy of the recurrence (CPU only)."""
    def run(qn, kn, v, alpha, beta, S0):
        S = S0.copy()
        out = np.zeros((len(qn), v.shape[1]))
        for t in range(len(qn)):
            if kind == "read_before_write":
                out[t] = S @ qn[t]
            a = 1.0 if kind == "dropped_decay" else alpha[t]
            S = a * S
            Sk = (S.T @ kn[t]) if kind == "transposed_state" else (S @ kn[t])
            sign = -1.0 if kind == "wrong_sign" else 1.0
            S = S + np.outer(beta[t] * (v[t] - sign * Sk), kn[t])
            if kind != "read_before_write":
                out[t] = S @ qn[t]
        return out, S
    return run


@pytest.mark.parametrize("kind", ["read_before_write", "dropped_decay", "transposed_state", "wrong_sign"])
def test_pins_catch_planted_mistakes(kind, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "two_token_k2.json")))
    out, S = _mutant(kind)(np.array(g["q"]), np.array(g["k"]), np.array(g["v"]),
                           np.array(g["alpha"]), np.array(g["beta"]), np.array(g["S0"]))
    assert (np.max(np.abs(out - np.array(g["out"]))) > 1e-3
            or np.max(np.abs(S - np.array(g["S_final"]))) > 1e-3)


def test_chunk_factors_against_independent_routes():
    """O2's per-chunk factors: W<- against the row recursion, U~ against the direct N^{-1},
    P entry by entry, and the chunk step built from them against the token recurrence."""
    rng = np.random.default_rng(7)
    C, K, V = 12, 6, 5
    kn = rng.standard_normal((C, K)); kn /= np.linalg.norm(kn, axis=1, keepdims=True)
    qn = rng.standard_normal((C, K)); qn /= np.linalg.norm(qn, axis=1, keepdims=True)
    v = rng.standard_normal((C, V))
    la = -rng.uniform(0.05, 0.8, C)
    be = rng.uniform(0.1, 0.9, C)
    f = cw.chunk_factors(qn, kn, v, la, be)
    g = np.cumsum(la)
    np.testing.assert_allclose(f["g"], g, rtol=0, atol=1e-15)
    np.testing.assert_allclose(f["W"], np.exp(g)[:, None] * cw.wy_rows(kn, be), rtol=1e-12, atol=1e-13)
    Ninv, _ = cw.n_inverse_two_ways(kn, la, be)
    np.testing.assert_allclose(f["U"], Ninv @ (be[:, None] * v), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(f["Minv"] @ cw.gram_factors(kn, be), np.eye(C), atol=1e-13)
    for i in range(C):
        for j in range(C):
            want = np.exp(g[i] - g[j]) * (qn[i] @ kn[j]) if j <= i else 0.0
            assert abs(f["P"][i, j] - want) <= 1e-13
    S0 = rng.standard_normal((V, K))
    U = f["U"] - f["W"] @ S0.T
    out = np.exp(g)[:, None] * (qn @ S0.T) + f["P"] @ U
    S1 = np.exp(g[-1]) * S0 + U.T @ (np.exp(g[-1] - g)[:, None] * kn)
    ref_out, ref_S = oracle.delta_rule(qn, kn, v, np.exp(la), be, S0)
    np.testing.assert_allclose(out, ref_out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(S1, ref_S, rtol=1e-11, atol=1e-12)
