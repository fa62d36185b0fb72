"""The per-chunk factors the intra-chunk kernel leaves in the workspace, chunk by chunk,
against the fp64 chunkwise oracle (O2, :func:`oracle.chunkwise.chunk_factors`).

For every chunk of every sequence and every value head this reads, through
gdn_workspace_layout, the chunk-local cumulative log decay g and beta (gates kernel), 1/|q|
and 1/|k| (the diagonal of the Gram product), and the WY factors W<-, U~ and the masked,
decayed scores P ("Simple math to speed up GDN prefill", sections "Reminder" and "Save one
invert": A = N^{-1} B = (Gamma . M^{-1}) B, W<- = A G K^, U~ = A V). M^{-1} itself never
leaves the chip; it is checked through W<- and U~, which are products of it. For K = V = 128
the factors carry the exact split exp(g_last - g_t)/|k_t| = m_t 2^e_t (rows of W<-, U~ times
m_t, columns of P divided by it, ks_t = 2^e_t stored), so the comparison undoes it with the
oracle's own exp(g_last - g_t)/|k_t| and the stored power of two.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import chunkwise as o2
from gated_deltanet_chunkwise_gdn_gb300 import _lib, gdn_extend_chunkwise, workloads as wl
from gpu_helpers import INPUT_KEYS, rel_l2

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

EPS = 1e-6  # q^ = q / sqrt(|q|^2 + eps)


def _f64(x: torch.Tensor) -> np.ndarray:
    return x.float().numpy().astype(np.float64)


def _region(ws: torch.Tensor, off: int, n: int, dtype) -> torch.Tensor:
    nbytes = n * torch.tensor([], dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_intra_factors_match_the_chunkwise_oracle(D):
    w = wl.custom("intermediates", [100, 64, 1, 150], H=2, HV=4, K=D, V=D, chunk_size=64, seed=61)
    d = wl.make_inputs(w)
    T, H, K = d["q"].shape
    HV, V = d["v"].shape[1], d["v"].shape[2]
    B = d["cache_indices"].shape[0]
    lay = _lib.workspace_layout(T, B, H, HV, K, V, 64)
    assert lay.block == 64 and lay.affine_factors == (1 if D == 128 else 0)
    ws = torch.zeros(lay.total + 256, dtype=torch.uint8, device="cuda")
    g = {k: d[k].cuda() for k in INPUT_KEYS}
    gdn_extend_chunkwise(*[g[k] for k in INPUT_KEYS], chunk_size=64, workspace=ws, check=True)
    torch.cuda.synchronize()
    ws = ws.cpu()
    C = lay.block
    n_chunks = int(_region(ws, lay.status, 2, torch.int32)[1])
    tab = _region(ws, lay.chunk_tab, 4 * n_chunks, torch.int32).view(n_chunks, 4).numpy()
    mc = int(lay.max_chunks)
    G = _region(ws, lay.g, mc * HV * C, torch.float32).view(mc, HV, C)
    Be = _region(ws, lay.beta, mc * HV * C, torch.float32).view(mc, HV, C)
    RQ = _region(ws, lay.rq, mc * H * C, torch.float32).view(mc, H, C)
    RK = _region(ws, lay.rk, mc * H * C, torch.float32).view(mc, H, C)
    et = d["q"].dtype
    Wg = _region(ws, lay.w, mc * HV * C * K, et).view(mc, HV, C, K)
    Ug = _region(ws, lay.u, mc * HV * C * V, et).view(mc, HV, C, V)
    Pg = _region(ws, lay.p, mc * HV * C * C, et).view(mc, HV, C, C)
    KS = _region(ws, lay.ks, mc * HV * C, torch.float32).view(mc, HV, C) if lay.affine_factors else None

    cu = d["cu_seqlens"].numpy()
    assert n_chunks == sum(-(-int(cu[s + 1] - cu[s]) // C) for s in range(B))
    q, k, v = _f64(d["q"]), _f64(d["k"]), _f64(d["v"])
    a, b = d["a"].numpy(), d["b"].numpy()
    A_log, dt_bias = d["A_log"].numpy(), d["dt_bias"].numpy()
    worst = dict(W=0.0, U=0.0, P=0.0)
    for j in range(n_chunks):
        seq, t0, L, c = (int(x) for x in tab[j])
        assert t0 == cu[seq] + c * C and L == min(C, cu[seq + 1] - t0) and L > 0
        for hv in range(HV):
            h = hv // (HV // H)
            rows = slice(t0, t0 + L)
            nq = np.sqrt((q[rows, h] ** 2).sum(1) + EPS)
            nk = np.sqrt((k[rows, h] ** 2).sum(1) + EPS)
            qn, kn = q[rows, h] / nq[:, None], k[rows, h] / nk[:, None]
            la = np.array([oracle.log_alpha(a[t, hv], A_log[hv], dt_bias[hv]) for t in range(t0, t0 + L)])
            be = np.array([oracle.beta(b[t, hv]) for t in range(t0, t0 + L)])
            f = o2.chunk_factors(qn, kn, v[rows, hv], la, be)
            # gates, and zeros past the chunk's length
            np.testing.assert_allclose(G[j, hv, :L].double().numpy(), f["g"], rtol=1e-5, atol=1e-4)
            np.testing.assert_allclose(Be[j, hv, :L].double().numpy(), be, rtol=1e-6, atol=1e-7)
            assert float(Be[j, hv, L:].abs().sum()) == 0.0
            np.testing.assert_allclose(RQ[j, h, :L].double().numpy(), 1 / nq, rtol=1e-5)
            np.testing.assert_allclose(RK[j, h, :L].double().numpy(), 1 / nk, rtol=1e-5)
            assert float(RQ[j, h, L:].abs().sum()) == 0.0 and float(RK[j, h, L:].abs().sum()) == 0.0
            W = _f64(Wg[j, hv, :L])
            U = _f64(Ug[j, hv, :L])
            P = _f64(Pg[j, hv, :L, :L])
            fW, fU, fP = f["W"], f["U"], f["P"]
            if KS is not None:
                # undo the split: row t of W, U times ks_t / sk_t (= 1 / m_t), column t of P times m_t.
                # With strong decay sk_t of the first rows falls below fp32's normal range: ks_t is
                # then a subnormal power of two (m_t has lost bits; those rows are left out) or 0
                # with m_t = 1 (the row is stored unscaled).
                sk = np.exp(f["g"][-1] - f["g"]) / nk
                ks = KS[j, hv, :L].double().numpy()
                pos = ks > 0
                assert np.all(ks >= 0) and np.all(np.log2(ks[pos]) == np.round(np.log2(ks[pos])))
                keep = (ks == 0) | (ks >= 2.0 ** -126)
                m = np.where(pos, sk / np.where(pos, ks, 1.0), 1.0)
                assert np.all((m[keep] > 0.499) & (m[keep] < 1.001)), m
                W, U, P = W[keep] / m[keep, None], U[keep] / m[keep, None], P[np.ix_(keep, keep)] * m[None, keep]
                fW, fU, fP = fW[keep], fU[keep], fP[np.ix_(keep, keep)]
            worst["W"] = max(worst["W"], rel_l2(W, fW))
            worst["U"] = max(worst["U"], rel_l2(U, fU))
            worst["P"] = max(worst["P"], rel_l2(P, fP))
            assert np.all(np.triu(_f64(Pg[j, hv, :L, :L]), 1) == 0)  # causal: nothing above the diagonal
    print(f"intermediates D={D}: worst per-tile rel-L2 W {worst['W']:.2e} U {worst['U']:.2e} P {worst['P']:.2e}")
    # 16-bit tiles (8-bit mantissa for bf16): about 2e-3 from the final rounding alone
    assert worst["W"] <= 1e-2 and worst["U"] <= 1e-2 and worst["P"] <= 1e-2, worst


def _seg_range(n, nseg, r16, part):
    """Chunk range of segment `part` when a sequence of n chunks is cut into nseg segments, segment 0
    r16/16 as long as the others (the scan's cut; returns (c0, c1, number of non-empty segments))."""
    if nseg <= 1 or n <= 0:
        return (0 if part == 0 else n), n, (1 if n > 0 else 0)
    den = (nseg - 1) * 16 + r16
    L0 = min(max(-(-n * r16 // den), 1), n)
    rest = n - L0
    L1 = -(-rest // (nseg - 1)) if rest > 0 else 1
    ns = 1 + -(-rest // L1)
    if part == 0:
        return 0, L0, ns
    c0 = L0 + (part - 1) * L1
    return min(c0, n), min(c0 + L1, n), ns


@pytest.mark.parametrize("D,decay", [(64, "weak"), (128, "weak"), (128, "strong"), (128, "switch")])
def test_segment_start_states_match_the_recurrence(D, decay):
    """A long sequence of one head runs through the segmented scan (per-segment affine maps chained
    into start states), and every segment's start state must equal the oracle's state after the
    prefix before it, to the state tolerance. Weak decay (A_log = -7): each start state carries the
    whole prefix. Strong: the default gates. Switch: weak decay for the first half of the sequence
    and strong after it, so one chain mixes both."""
    T = 8192
    w = wl.custom("segstates", [T], H=1, HV=1, K=D, V=D, chunk_size=64, seed=62)
    d = wl.make_inputs(w)
    if decay == "weak":
        d["A_log"].fill_(-7.0)
    elif decay == "switch":
        d["a"][: T // 2] = -12.0  # softplus(-12) ~ 6e-6: almost no decay in the first half
    lay = _lib.workspace_layout(T, 1, 1, 1, D, D, 64)
    assert lay.nseg > 2
    ws = torch.zeros(lay.total + 256, dtype=torch.uint8, device="cuda")
    g = {k: d[k].cuda() for k in INPUT_KEYS}
    gdn_extend_chunkwise(*[g[k] for k in INPUT_KEYS], chunk_size=64, workspace=ws, check=True)
    torch.cuda.synchronize()
    ws = ws.cpu()
    st = _region(ws, lay.seg_state, lay.nseg * D * D, torch.float32).view(lay.nseg, D, D).double().numpy()
    n = T // 64
    r16 = 8 if D == 128 else 16
    _, _, ns = _seg_range(n, lay.nseg, r16, 0)
    assert ns == lay.nseg
    for s in range(1, ns):
        c0, _, _ = _seg_range(n, lay.nseg, r16, s)
        t = 64 * c0  # the state entering segment s is the state after the first t tokens
        dp = dict(d)
        for k in ("q", "k", "v", "a", "b"):
            dp[k] = d[k][:t]
        dp["cu_seqlens"] = torch.tensor([0, t], dtype=torch.int64)
        ref = oracle.gdn_forward(*[dp[k] for k in INPUT_KEYS]).states[0]
        err = rel_l2(st[s], ref)
        print(f"segment {s} of {ns} (token {t}): start-state rel-L2 {err:.3e}")
        assert err <= 5e-3, (s, err)
