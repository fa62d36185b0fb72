"""Helpers shared by the GPU tests: run the CUDA path through the binding and
compare it with the oracle, element by element, on the same seeded inputs."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from gated_deltanet_chunkwise_gdn_gb300 import gdn_extend_chunkwise

# Tolerances (relative L2 over all compared elements): 16-bit outputs vs the fp64
# oracle, and the final fp32 state vs the fp64 oracle.
OUT_TOL = 1e-2
STATE_TOL = 5e-3

INPUT_KEYS = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state_pool", "cache_indices", "cu_seqlens")


def to_device(d: dict, device="cuda") -> dict:
    return {k: (d[k].to(device) if isinstance(d[k], torch.Tensor) else d[k]) for k in d}


def run_gpu(d: dict, chunk_size=None, scale=1.0, check=True, out=None):
    """Runs the CUDA path; returns (out [T,HV,V] on CPU, state_pool after the call on CPU)."""
    g = to_device(d)
    pool = g["state_pool"]
    o = gdn_extend_chunkwise(*[g[k] for k in INPUT_KEYS[:7]], pool, g["cache_indices"], g["cu_seqlens"],
                             chunk_size=chunk_size or d["chunk_size"], scale=scale, check=check, out=out)
    torch.cuda.synchronize()
    return o.cpu(), pool.cpu()


def rel_l2(x: np.ndarray, y: np.ndarray) -> float:
    den = float(np.linalg.norm(y))
    return float(np.linalg.norm(x - y)) / (den if den > 0 else 1.0)


def oracle_for(d: dict, chains=None, scale=1.0):
    return oracle.gdn_forward(*[d[k] for k in INPUT_KEYS], scale=scale, chains=chains,
                              is_fp16=d["q"].dtype == torch.float16)


# A single chain may be up to this many times its whole-tensor tolerance: one norm over a
# whole call could otherwise hide a chain (or a segment of one) that is wrong.
CHAIN_FACTOR = 2.0


def compare(d: dict, out_gpu: torch.Tensor, pool_gpu: torch.Tensor, res, out_tol=OUT_TOL,
            state_tol=STATE_TOL) -> dict:
    """Element-by-element comparison of the GPU result with the oracle's chains: relative L2
    over all compared elements, and the same per (sequence, value head) chain."""
    cu = d["cu_seqlens"].numpy()
    idx = d["cache_indices"].numpy()
    og, ro, sg, rs = [], [], [], []
    out_np = out_gpu.float().numpy()
    pool_np = pool_gpu.numpy()
    worst_out = worst_state = 0.0
    worst_chain = None
    for i, (s, hv) in enumerate(res.chains):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        og.append(out_np[t0:t1, hv].astype(np.float64).reshape(-1))
        ro.append(res.chain_output(i).reshape(-1))
        sg.append(pool_np[idx[s], hv].astype(np.float64).reshape(-1))
        rs.append(res.states[i].reshape(-1))
        eo = rel_l2(og[-1], ro[-1]) if t1 > t0 else 0.0
        es = rel_l2(sg[-1], rs[-1])
        if eo / out_tol + es / state_tol > worst_out / out_tol + worst_state / state_tol:
            worst_chain = (int(s), int(hv))
        worst_out, worst_state = max(worst_out, eo), max(worst_state, es)
    og, ro = np.concatenate(og), np.concatenate(ro)
    sg, rs = np.concatenate(sg), np.concatenate(rs)
    stats = dict(out_rel_l2=rel_l2(og, ro), state_rel_l2=rel_l2(sg, rs),
                 chain_out_rel_l2=worst_out, chain_state_rel_l2=worst_state, worst_chain=worst_chain,
                 out_finite=bool(np.isfinite(og).all()), state_finite=bool(np.isfinite(sg).all()))
    print(f"parity: out rel-L2 {stats['out_rel_l2']:.3e}  state rel-L2 {stats['state_rel_l2']:.3e}  "
          f"worst chain {worst_chain}: out {worst_out:.3e} state {worst_state:.3e}")
    assert stats["out_finite"] and stats["state_finite"], stats
    assert stats["out_rel_l2"] <= out_tol, stats
    assert stats["state_rel_l2"] <= state_tol, stats
    assert worst_out <= CHAIN_FACTOR * out_tol, stats
    assert worst_state <= CHAIN_FACTOR * state_tol, stats
    return stats


def untouched_slots_equal(d: dict, pool_gpu: torch.Tensor):
    used = set(int(x) for x in d["cache_indices"])
    for s in range(d["state_pool"].shape[0]):
        if s not in used:
            assert torch.equal(pool_gpu[s], d["state_pool"][s]), f"slot {s} was modified"
