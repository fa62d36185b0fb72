"""GPU parity of the backward pass (gdn_chunkwise_backward) against the fp64 oracles.

The reference gradients come from oracle/backward.py (the chain rule applied to the token
recurrence, pinned on the CPU by finite differences and by autograd of the chunkwise form) and,
for long chains, from the explicit chunkwise backward of oracle/chunkwise_grad.py (pinned against
the former on the CPU). Inputs are the seeded workloads of the forward tests; the gradients
arriving from above (d_out, d_state) are drawn from their own seeded generator.

Tolerance: every gradient is fp32 and the kernels carry fp32 operands as bf16 hi + lo pairs
(about 16 bits), so the backward is held to the forward's state tolerance (5e-3 relative L2 per
gradient tensor) and, per (sequence, value head) chain, to twice that.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from gated_deltanet_chunkwise_gdn_gb300 import (GatedDeltaNetChunkwise, GdnError, gdn_chunkwise_backward,
                                                workloads as wl)
from oracle import backward as bw
from oracle import chunkwise_grad as cg

pytestmark = pytest.mark.gpu

GRAD_TOL = 5e-3
CHAIN_FACTOR = 2.0
KEYS = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state_pool", "cache_indices", "cu_seqlens")


def upstream(d: dict, seed: int, with_state: bool = True):
    """Seeded gradients from above: d_out like v (same dtype), d_state like the pool (fp32)."""
    gen = torch.Generator().manual_seed(10_000 + seed)
    d_out = torch.randn(d["v"].shape, generator=gen).to(d["v"].dtype)
    d_state = 0.1 * torch.randn(d["state_pool"].shape, generator=gen) if with_state else None
    return d_out, d_state


def run_backward(d, d_out, d_state, chunk_size=None, scale=1.0):
    g = {k: d[k].cuda() for k in KEYS}
    res = gdn_chunkwise_backward(*[g[k] for k in KEYS], d_out.cuda(),
                                 d_state.cuda() if d_state is not None else None,
                                 chunk_size=chunk_size or d["chunk_size"], scale=scale, check=True)
    torch.cuda.synchronize()
    return {k: getattr(res, k).cpu().double().numpy() for k in res._fields}


def oracle_backward(d, d_out, d_state, scale=1.0):
    idx = d["cache_indices"].numpy()
    ds = d_state if d_state is not None else torch.zeros_like(d["state_pool"])
    ds_seq = ds.double().numpy()[idx]
    return bw.gdn_backward(*[d[k] for k in KEYS], d_out.double(), ds_seq, scale=scale)


def rel(x, y):
    den = float(np.linalg.norm(y))
    return float(np.linalg.norm(x - y)) / (den if den > 0 else 1.0)


def compare(d, got, ref, tol=GRAD_TOL):
    """Relative L2 per gradient tensor, and the worst (sequence, value head) chain."""
    cu = d["cu_seqlens"].numpy()
    idx = d["cache_indices"].numpy()
    H, HV = d["q"].shape[1], d["v"].shape[1]
    r = HV // H
    errs = {}
    names = {"dq": "dq", "dk": "dk", "dv": "dv", "da": "da", "db": "db", "dA_log": "dA_log",
             "ddt_bias": "ddt_bias", "d_state_pool": "d_state_pool"}
    for gk, rk in names.items():
        x, y = got[gk], ref[rk]
        if gk == "d_state_pool":
            x, y = x[idx], y[idx]
        errs[gk] = rel(x, y)
    worst = 0.0
    for s in range(len(idx)):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        for hv in range(HV):
            h = hv // r
            for gk, sl in (("dv", (slice(t0, t1), hv)), ("da", (slice(t0, t1), hv)),
                           ("db", (slice(t0, t1), hv))):
                if t1 > t0:
                    worst = max(worst, rel(got[gk][sl], ref[gk][sl]))
            worst = max(worst, rel(got["d_state_pool"][idx[s], hv], ref["d_state_pool"][idx[s], hv]))
            if t1 > t0 and hv % r == 0:
                for gk in ("dq", "dk"):
                    worst = max(worst, rel(got[gk][t0:t1, h], ref[gk][t0:t1, h]))
    errs["worst_chain"] = worst
    print({k: f"{v:.2e}" for k, v in errs.items()})
    for k, v in errs.items():
        lim = tol * CHAIN_FACTOR if k == "worst_chain" else tol
        assert v <= lim, (k, v, errs)
    return errs


CASES = {
    # name: (lengths, H, HV, K, chunk_size, extra workload args)
    "d64_gqa_ragged": ([100, 64, 1, 130], 2, 4, 64, 64, {}),
    "d128_ragged": ([300, 65, 7], 2, 2, 128, 64, {}),
    "d128_gqa4": ([129, 200], 1, 4, 128, 64, {}),
    "d64_strong_decay": ([200, 77], 2, 2, 64, 64, dict(a_mean=4.0)),
    "d128_weak_decay": ([257, 190], 2, 2, 128, 64, dict(a_mean=-6.0)),
    "d64_chunk128": ([300, 5], 2, 2, 64, 128, {}),
}


@pytest.mark.parametrize("name", list(CASES))
def test_backward_matches_oracle(name):
    lengths, H, HV, K, C, extra = CASES[name]
    seed = 300 + list(CASES).index(name)
    d = wl.make_inputs(wl.custom(name, lengths, H=H, HV=HV, K=K, V=K, chunk_size=C, seed=seed, **extra))
    d_out, d_state = upstream(d, seed)
    got = run_backward(d, d_out, d_state)
    compare(d, got, oracle_backward(d, d_out, d_state))


@pytest.mark.parametrize("H,HV,K", [(2, 2, 128), (1, 2, 64), (2, 4, 128)])
def test_backward_fp16_inputs(H, HV, K):
    """fp16 q, k, v, dO: the generic local kernel, and with grouped heads the norm kernel."""
    d = wl.make_inputs(wl.custom("bwd_fp16", [150, 40], H=H, HV=HV, K=K, V=K, chunk_size=64, seed=320 + HV + K,
                                 dtype=torch.float16))
    d_out, d_state = upstream(d, 320)
    compare(d, run_backward(d, d_out, d_state), oracle_backward(d, d_out, d_state))


def test_backward_scale_and_no_state_gradient():
    d = wl.make_inputs(wl.custom("bwd_scale", [90, 33], H=1, HV=2, K=64, V=64, chunk_size=64, seed=321))
    d_out, _ = upstream(d, 321, with_state=False)
    got = run_backward(d, d_out, None, scale=0.3)
    compare(d, got, oracle_backward(d, d_out, None, scale=0.3))


def test_backward_untouched_slots_and_empty_sequence():
    """A zero-length sequence passes its state gradient through unchanged; slots outside the batch
    stay as the caller left them."""
    d = wl.make_inputs(wl.custom("bwd_empty", [70, 0, 20], H=2, HV=2, K=64, V=64, chunk_size=64, seed=322,
                                 pool_size=6))
    d_out, d_state = upstream(d, 322)
    g = {k: d[k].cuda() for k in KEYS}
    sentinel = torch.full(d["state_pool"].shape, 7.0, device="cuda")
    res = gdn_chunkwise_backward(*[g[k] for k in KEYS], d_out.cuda(), d_state.cuda(), chunk_size=64, check=True,
                                 d_state_pool=sentinel)
    torch.cuda.synchronize()
    idx = d["cache_indices"].tolist()
    dsp = res.d_state_pool.cpu()
    for slot in range(6):
        if slot not in idx:
            assert torch.all(dsp[slot] == 7.0)
    assert torch.equal(dsp[idx[1]], d_state[idx[1]])
    got = {k: getattr(res, k).cpu().double().numpy() for k in res._fields}
    compare(d, got, oracle_backward(d, d_out, d_state))


def test_backward_in_place_state_gradient():
    """d_state_pool may be d_state itself: each slot's gradient is read before it is written."""
    d = wl.make_inputs(wl.custom("bwd_inplace", [120, 64], H=2, HV=2, K=128, V=128, chunk_size=64, seed=323))
    d_out, d_state = upstream(d, 323)
    ref = run_backward(d, d_out, d_state)
    g = {k: d[k].cuda() for k in KEYS}
    buf = d_state.cuda().clone()
    res = gdn_chunkwise_backward(*[g[k] for k in KEYS], d_out.cuda(), buf, chunk_size=64, check=True,
                                 d_state_pool=buf)
    torch.cuda.synchronize()
    idx = d["cache_indices"].numpy()
    assert np.array_equal(res.d_state_pool.cpu().numpy()[idx], ref["d_state_pool"][idx].astype(np.float32))


def test_backward_is_deterministic():
    d = wl.make_inputs(wl.custom("bwd_det", [200, 31], H=2, HV=4, K=128, V=128, chunk_size=64, seed=324))
    d_out, d_state = upstream(d, 324)
    a = run_backward(d, d_out, d_state)
    b = run_backward(d, d_out, d_state)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_backward_bad_index_is_reported_and_writes_nothing():
    d = wl.make_inputs(wl.custom("bwd_bad", [40, 40], H=1, HV=1, K=64, V=64, chunk_size=64, seed=325))
    d["cache_indices"] = torch.tensor([1, 1], dtype=torch.int64)  # repeated slot
    d_out, d_state = upstream(d, 325)
    g = {k: d[k].cuda() for k in KEYS}
    sentinel = torch.full(d["state_pool"].shape, 3.0, device="cuda")
    with pytest.raises(GdnError):
        gdn_chunkwise_backward(*[g[k] for k in KEYS], d_out.cuda(), d_state.cuda(), chunk_size=64, check=True,
                               d_state_pool=sentinel)
    torch.cuda.synchronize()
    assert torch.all(sentinel == 3.0)


def test_backward_long_chains_sampled_heads():
    """The long-prefill shape (B = 1, T = 65536, H = HV = 16, K = V = 128) in the launch configuration of
    a full call; two value heads compared with the explicit chunkwise oracle, chain by chain."""
    w = wl.custom("bwd_long", [65536], H=16, HV=16, K=128, V=128, chunk_size=64, seed=326, pool_size=1,
                  state_std=0.0)
    d = wl.make_inputs(w)
    d_out, d_state = upstream(d, 326)
    got = run_backward(d, d_out, d_state)
    slot = int(d["cache_indices"][0])
    f = lambda x: x.double().numpy()
    for hv in (0, 11):
        ref = cg.chunkwise_backward_explicit(
            f(d["q"][:, hv]), f(d["k"][:, hv]), f(d["v"][:, hv]), f(d["a"][:, hv]), f(d["b"][:, hv]),
            float(d["A_log"][hv]), float(d["dt_bias"][hv]), f(d["state_pool"][slot, hv]), f(d_out[:, hv]),
            f(d_state[slot, hv]), C=64)
        errs = {"dq": rel(got["dq"][:, hv], ref["dq"]), "dk": rel(got["dk"][:, hv], ref["dk"]),
                "dv": rel(got["dv"][:, hv], ref["dv"]), "da": rel(got["da"][:, hv], ref["da"]),
                "db": rel(got["db"][:, hv], ref["db"]),
                "dS0": rel(got["d_state_pool"][slot, hv], ref["dS0"]),
                "dA_log": abs(got["dA_log"][hv] - ref["dA_log"]) / max(abs(ref["dA_log"]), 1e-30),
                "ddt_bias": abs(got["ddt_bias"][hv] - ref["ddt_bias"]) / max(abs(ref["ddt_bias"]), 1e-30)}
        print(hv, {k: f"{v:.2e}" for k, v in errs.items()})
        for k, v in errs.items():
            assert v <= GRAD_TOL, (hv, k, v)


def test_autograd_function_against_the_oracle():
    """torch.autograd through GatedDeltaNetChunkwise: a weighted loss on the output and the final states,
    gradients of every input compared with the fp64 oracle."""
    d = wl.make_inputs(wl.custom("bwd_autograd", [150, 70], H=2, HV=2, K=64, V=64, chunk_size=64, seed=327,
                                 index_rule="arange"))
    d_out, d_state = upstream(d, 327)
    B = 2
    leaf = {k: d[k].cuda().requires_grad_(True) for k in ("q", "k", "v", "a", "b", "A_log", "dt_bias")}
    init = d["state_pool"][:B].cuda().requires_grad_(True)
    out, final = GatedDeltaNetChunkwise.apply(leaf["q"], leaf["k"], leaf["v"], leaf["a"], leaf["b"],
                                              leaf["A_log"], leaf["dt_bias"], init, d["cu_seqlens"].cuda(), 64)
    loss = (out.float() * d_out.float().cuda()).sum() + (final * d_state[:B].cuda()).sum()
    loss.backward()
    torch.cuda.synchronize()
    ref = oracle_backward(d, d_out, d_state)
    pairs = {"dq": leaf["q"], "dk": leaf["k"], "dv": leaf["v"], "da": leaf["a"], "db": leaf["b"],
             "dA_log": leaf["A_log"], "ddt_bias": leaf["dt_bias"]}
    for name, t in pairs.items():
        e = rel(t.grad.double().cpu().numpy(), ref[name])
        tol = 1e-2 if name in ("dq", "dk", "dv") else GRAD_TOL  # q, k, v gradients come back in bf16
        assert e <= tol, (name, e)
    e = rel(init.grad.double().cpu().numpy(), ref["d_state_pool"][:B])
    assert e <= GRAD_TOL, e


def _guarded(shape, fill, guard=4096):
    """A tensor of `shape` inside a larger buffer with `guard` elements of `fill` on each side."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * guard,), fill, dtype=torch.float32, device="cuda")
    return buf, buf[guard:guard + n].view(shape)


def test_backward_writes_nothing_outside_its_buffers():
    """Guard regions around every gradient buffer and around the workspace stay as they were."""
    from gated_deltanet_chunkwise_gdn_gb300 import GdnGrads, gdn_backward_workspace_size
    d = wl.make_inputs(wl.custom("bwd_guard", [130, 64, 5], H=2, HV=4, K=128, V=128, chunk_size=64, seed=328))
    d_out, d_state = upstream(d, 328)
    g = {k: d[k].cuda() for k in KEYS}
    T, H, K = d["q"].shape
    HV = d["v"].shape[1]
    shapes = ((T, H, K), (T, H, K), (T, HV, K), (T, HV), (T, HV), (HV,), (HV,), tuple(d["state_pool"].shape))
    bufs = [_guarded(s, 11.0) for s in shapes]
    grads = GdnGrads(*[v for _, v in bufs])
    need = gdn_backward_workspace_size(T, 3, H, HV, K, K, 64)
    guard = 1 << 16
    ws_buf = torch.full((need + 2 * guard,), 0x5A, dtype=torch.uint8, device="cuda")
    ws = ws_buf[guard:guard + need]
    gdn_chunkwise_backward(*[g[k] for k in KEYS], d_out.cuda(), d_state.cuda(), chunk_size=64, check=True,
                           workspace=ws, grads=grads)
    torch.cuda.synchronize()
    for buf, view in bufs:
        n = view.numel()
        assert torch.all(buf[:4096] == 11.0) and torch.all(buf[4096 + n:] == 11.0)
    assert torch.all(ws_buf[:guard] == 0x5A) and torch.all(ws_buf[guard + need:] == 0x5A)
    got = {k: getattr(grads, k).cpu().double().numpy() for k in grads._fields}
    compare(d, got, oracle_backward(d, d_out, d_state))


def test_backward_replays_in_a_cuda_graph():
    """With its workspace and gradient buffers given, the backward call is captured in a CUDA graph and
    replayed on new input contents; the replay equals a direct call bit for bit."""
    from gated_deltanet_chunkwise_gdn_gb300 import GdnGrads, gdn_backward_workspace_size
    d1 = wl.make_inputs(wl.custom("bwd_graph", [150, 90], H=2, HV=2, K=64, V=64, chunk_size=64, seed=329))
    d2 = wl.make_inputs(wl.custom("bwd_graph", [150, 90], H=2, HV=2, K=64, V=64, chunk_size=64, seed=330))
    o1, s1 = upstream(d1, 329)
    o2, s2 = upstream(d2, 330)
    T, H, K = d1["q"].shape
    HV = d1["v"].shape[1]
    g = {k: d1[k].cuda() for k in KEYS}
    d_out, d_state = o1.cuda(), s1.cuda()
    ws = torch.empty(gdn_backward_workspace_size(T, 2, H, HV, K, K, 64), dtype=torch.uint8, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    grads = GdnGrads(torch.empty((T, H, K), **f32), torch.empty((T, H, K), **f32), torch.empty((T, HV, K), **f32),
                     torch.empty((T, HV), **f32), torch.empty((T, HV), **f32), torch.empty((HV,), **f32),
                     torch.empty((HV,), **f32), torch.zeros_like(g["state_pool"]))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside the capture (kernel attributes are set on first use)
        gdn_chunkwise_backward(*[g[k] for k in KEYS], d_out, d_state, chunk_size=64, workspace=ws, grads=grads)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn_chunkwise_backward(*[g[k] for k in KEYS], d_out, d_state, chunk_size=64, workspace=ws, grads=grads)
    for k in KEYS:
        g[k].copy_(d2[k])
    d_out.copy_(o2)
    d_state.copy_(s2)
    graph.replay()
    torch.cuda.synchronize()
    replay = {k: getattr(grads, k).cpu().numpy().copy() for k in grads._fields}
    direct = run_backward(d2, o2, s2)
    idx2 = d2["cache_indices"].numpy()
    replay["d_state_pool"], direct["d_state_pool"] = replay["d_state_pool"][idx2], direct["d_state_pool"][idx2]
    for k in replay:
        assert np.array_equal(replay[k].astype(np.float64), direct[k]), k


def test_backward_of_a_call_without_tokens():
    """Every sequence empty (total_tokens = 0): each slot's state gradient passes through unchanged, and the
    gate-parameter gradients are zero."""
    d = wl.make_inputs(wl.custom("bwd_empty_all", [0, 0, 0], H=2, HV=2, K=64, V=64, chunk_size=64, seed=331,
                                 pool_size=5))
    d_out, d_state = upstream(d, 331)
    g = {k: d[k].cuda() for k in KEYS}
    res = gdn_chunkwise_backward(*[g[k] for k in KEYS], d_out.cuda(), d_state.cuda(), chunk_size=64, check=True)
    torch.cuda.synchronize()
    idx = d["cache_indices"].tolist()
    for slot in range(5):
        want = d_state[slot] if slot in idx else torch.zeros_like(d_state[slot])
        assert torch.equal(res.d_state_pool[slot].cpu(), want)
    assert torch.all(res.dA_log == 0) and torch.all(res.ddt_bias == 0)
    assert res.dq.shape[0] == 0 and res.dv.shape[0] == 0
