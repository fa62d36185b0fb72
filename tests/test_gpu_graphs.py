"""Both entry points captured in CUDA graphs and replayed, against the fp64 oracle.

A serving loop replays captured steps instead of issuing each launch from the host. The calls
keep no host state between launches: tensor maps are kernel arguments, the work counters live
in the workspace and are reset by the call's first kernel, and the decode update kernel's
programmatic launch becomes a programmatic edge of the graph. So a replay with new contents in
the captured buffers must give the oracle's result for those contents.
"""

import numpy as np
import pytest
import torch

from gated_deltanet_chunkwise_gdn_gb300 import gdn_decode_step, gdn_extend_chunkwise
from gated_deltanet_chunkwise_gdn_gb300 import workloads as wl

from gpu_helpers import INPUT_KEYS, OUT_TOL, STATE_TOL, compare, oracle_for, rel_l2, to_device

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU runs, skipped there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def test_decode_steps_replayed_from_a_graph():
    """One captured decode step, replayed for tokens 0..3 of 64 sequences (inputs copied into the
    captured buffers before each replay): outputs of every token and final states match the oracle."""
    B, n_tok = 64, 4
    w = wl.custom("graph_dec", [n_tok] * B, H=2, HV=4, K=128, V=128, chunk_size=64, seed=81)
    d = wl.make_inputs(w)
    res = oracle_for(d)
    g = to_device(d)
    cu = d["cu_seqlens"]
    tok = lambda j: torch.tensor([int(cu[s]) + j for s in range(B)], dtype=torch.int64, device="cuda")
    live = {k: g[k][tok(0)].clone() for k in ("q", "k", "v", "a", "b")}
    out = torch.empty((B, 4, 128), dtype=torch.bfloat16, device="cuda")
    pool = g["state_pool"]
    pool0 = pool.clone()
    args = lambda: [live["q"], live["k"], live["v"], live["a"], live["b"], g["A_log"], g["dt_bias"], pool,
                    g["cache_indices"]]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture (loads the library, caches the status word)
        gdn_decode_step(*args(), out=out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    pool.copy_(pool0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn_decode_step(*args(), out=out)
    pool.copy_(pool0)  # capture does not run the kernels, but start from the original states anyway
    outs = []
    for j in range(n_tok):
        ix = tok(j)
        for k2 in live:
            live[k2].copy_(g[k2][ix])
        graph.replay()
        outs.append(out.float().cpu().numpy())
    torch.cuda.synchronize()
    got_o, ref_o = [], []
    for i, (s, hv) in enumerate(res.chains):
        ro = res.chain_output(i)
        for j in range(n_tok):
            got_o.append(outs[j][s, hv])
            ref_o.append(ro[j])
    assert rel_l2(np.concatenate(got_o), np.concatenate(ref_o)) <= OUT_TOL
    pool_np = pool.cpu().numpy()
    idx = d["cache_indices"].numpy()
    got_s = np.concatenate([pool_np[idx[s], hv].reshape(-1) for (s, hv) in res.chains])
    ref_s = np.concatenate([res.states[i].reshape(-1) for i in range(len(res.chains))])
    assert rel_l2(got_s, ref_s) <= STATE_TOL


@pytest.mark.parametrize("lengths", [[300, 129, 64, 1], [9000]])
def test_prefill_replayed_from_a_graph(lengths):
    """A captured prefill call replayed on a second input set of the same shape; the second case
    is long enough for the segmented scan."""
    ws = [wl.custom("graph_pre", lengths, H=2, HV=4, K=128, V=128, chunk_size=64, seed=s) for s in (82, 83)]
    d0, d1 = wl.make_inputs(ws[0]), wl.make_inputs(ws[1])
    g = to_device(d0)
    T = sum(lengths)
    out = torch.empty((T, 4, 128), dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up: loads the library and sizes the cached workspace
        gdn_extend_chunkwise(*[g[k] for k in INPUT_KEYS], chunk_size=64, out=out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn_extend_chunkwise(*[g[k] for k in INPUT_KEYS], chunk_size=64, out=out)
    for k in INPUT_KEYS:  # the second input set, in the captured buffers
        g[k].copy_(d1[k].to("cuda"))
    graph.replay()
    torch.cuda.synchronize()
    compare(d1, out.cpu(), g["state_pool"].cpu(), oracle_for(d1))
