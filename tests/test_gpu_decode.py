"""Single-token step (gdn_decode_step) on the GPU against the fp64 oracle.

A decode batch is the recurrence with one token per sequence (cu_seqlens = 0, 1, ..., B), so
the oracle is the same token-by-token recurrence the prefill tests use. Outputs and states are
compared element by element with the prefill tolerances.
"""

import numpy as np
import pytest
import torch

from gated_deltanet_chunkwise_gdn_gb300 import GdnError, gdn_decode_step, gdn_extend_chunkwise
from gated_deltanet_chunkwise_gdn_gb300 import workloads as wl

from gpu_helpers import (INPUT_KEYS, OUT_TOL, STATE_TOL, compare, oracle_for, rel_l2, to_device,
                         untouched_slots_equal)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU runs, skipped there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

DEC_KEYS = ("q", "k", "v", "a", "b", "A_log", "dt_bias", "state_pool", "cache_indices")


def run_decode(d: dict, scale=1.0, check=True):
    g = to_device(d)
    out = gdn_decode_step(*[g[k] for k in DEC_KEYS], scale=scale, check=check)
    torch.cuda.synchronize()
    return out.cpu(), g["state_pool"].cpu()


def decode_inputs(B, H, HV, D, seed, dtype=torch.bfloat16, pool_size=None, a_mean=0.0, b_mean=0.0):
    w = wl.custom("decode", [1] * B, H=H, HV=HV, K=D, V=D, chunk_size=64, seed=seed, pool_size=pool_size,
                  a_mean=a_mean, b_mean=b_mean, dtype=dtype)
    return wl.make_inputs(w)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_decode_matches_oracle(D, dtype):
    d = decode_inputs(37, 2, 4, D, seed=60 + D, dtype=dtype)
    out, pool = run_decode(d)
    compare(d, out, pool, oracle_for(d))
    untouched_slots_equal(d, pool)


def test_decode_workload_full_size():
    """The benchmarked decode batch (256 sequences, H=16, HV=32, K=V=128), every output and state."""
    d = wl.make_inputs(wl.BY_NAME["decode"])
    out, pool = run_decode(d)
    compare(d, out, pool, oracle_for(d))
    untouched_slots_equal(d, pool)


def test_decode_gqa_ratio_four_and_gate_extremes():
    d = decode_inputs(300, 2, 8, 128, seed=71, a_mean=3.0, b_mean=-3.0)   # strong decay, small beta
    out, pool = run_decode(d)
    compare(d, out, pool, oracle_for(d))
    d = decode_inputs(300, 2, 8, 128, seed=72, a_mean=-6.0, b_mean=3.0)   # almost no decay, beta near 1
    out, pool = run_decode(d)
    compare(d, out, pool, oracle_for(d))


def test_decode_scale_argument():
    d = decode_inputs(16, 2, 2, 128, seed=73)
    out, pool = run_decode(d, scale=0.125)
    compare(d, out, pool, oracle_for(d, scale=0.125))


def test_decode_steps_continue_a_prefill():
    """Prefill 100 tokens of each sequence, then decode tokens 100, 101, 102 one step at a time:
    the decode outputs and the final states match the oracle over all 103 tokens."""
    B, L, n_dec = 5, 100, 3
    w = wl.custom("cont", [L + n_dec] * B, H=2, HV=4, K=128, V=128, chunk_size=64, seed=74)
    d = wl.make_inputs(w)
    res = oracle_for(d)
    cu = d["cu_seqlens"]
    g = to_device(d)
    pool = g["state_pool"]
    tok = lambda j: torch.tensor([int(cu[s]) + j for s in range(B)], dtype=torch.int64)
    pre = torch.cat([torch.arange(int(cu[s]), int(cu[s]) + L) for s in range(B)])
    cu_pre = torch.arange(0, B * L + 1, L, dtype=torch.int64)
    gdn_extend_chunkwise(*[g[k][pre.to(g[k].device)] for k in ("q", "k", "v", "a", "b")], g["A_log"], g["dt_bias"],
                         pool, g["cache_indices"], cu_pre.cuda(), chunk_size=64, check=True)
    outs = []
    for j in range(L, L + n_dec):
        ix = tok(j).cuda()
        outs.append(gdn_decode_step(*[g[k][ix] for k in ("q", "k", "v", "a", "b")], g["A_log"], g["dt_bias"],
                                    pool, g["cache_indices"], check=True).float().cpu().numpy())
    torch.cuda.synchronize()
    got_o, ref_o = [], []
    for i, (s, hv) in enumerate(res.chains):
        ro = res.chain_output(i)
        for jj in range(n_dec):
            got_o.append(outs[jj][s, hv])
            ref_o.append(ro[L + jj])
    assert rel_l2(np.concatenate(got_o), np.concatenate(ref_o)) <= OUT_TOL
    pool_np = pool.cpu().numpy()
    idx = d["cache_indices"].numpy()
    got_s = np.concatenate([pool_np[idx[s], hv].reshape(-1) for (s, hv) in res.chains])
    ref_s = np.concatenate([res.states[i].reshape(-1) for i in range(len(res.chains))])
    assert rel_l2(got_s, ref_s) <= STATE_TOL


@pytest.mark.parametrize("bad", ["repeat_across_tiles", "repeat_in_tile", "negative", "past_end"])
def test_decode_bad_cache_indices_rejected_on_device(bad):
    d = decode_inputs(300, 2, 2, 64, seed=75, pool_size=700)
    idx = d["cache_indices"].clone()
    if bad == "repeat_across_tiles":
        idx[290] = idx[5]
    elif bad == "repeat_in_tile":
        idx[7] = idx[6]
    elif bad == "negative":
        idx[299] = -1
    else:
        idx[0] = 700
    d["cache_indices"] = idx
    g = to_device(d)
    sentinel = torch.full((300, 2, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(GdnError) as e:
        gdn_decode_step(*[g[k] for k in DEC_KEYS], out=sentinel, check=True)
    assert e.value.status == 3
    assert torch.equal(g["state_pool"].cpu(), d["state_pool"]), "a rejected step changed the pool"
    assert bool((sentinel == 7.0).all()), "a rejected step wrote its output"


def test_decode_empty_batch():
    d = decode_inputs(4, 2, 2, 64, seed=76)
    g = to_device(d)
    e = {k: (g[k][:0] if k in ("q", "k", "v", "a", "b", "cache_indices") else g[k]) for k in DEC_KEYS}
    out = gdn_decode_step(*[e[k] for k in DEC_KEYS], check=True)
    assert tuple(out.shape) == (0, 2, 64)
    assert torch.equal(g["state_pool"].cpu(), d["state_pool"])


def test_decode_equals_chunkwise_call_with_unit_lengths():
    """The dedicated step and the chunkwise call over the same one-token sequences agree
    (both within the oracle's tolerance, and with each other closely)."""
    d = decode_inputs(64, 4, 8, 128, seed=77)
    o1, p1 = run_decode(d)
    g = to_device(d)
    o2 = gdn_extend_chunkwise(*[g[k] for k in INPUT_KEYS], chunk_size=64, check=True)
    torch.cuda.synchronize()
    res = oracle_for(d)
    compare(d, o2.cpu(), g["state_pool"].cpu(), res)
    assert rel_l2(o1.float().numpy().astype(np.float64), o2.float().cpu().numpy().astype(np.float64)) <= OUT_TOL


def test_decode_batch_above_one_block_check():
    """Above 1024 sequences the slot check runs as a grid of tile pairs after a memset."""
    d = decode_inputs(1300, 1, 2, 64, seed=78, pool_size=2700)
    out, pool = run_decode(d)
    compare(d, out, pool, oracle_for(d))
    untouched_slots_equal(d, pool)


@pytest.mark.parametrize("pos", [(3, 1290), (1100, 1299), (1025, 1026)])
def test_decode_batch_above_one_block_check_rejects_repeats(pos):
    d = decode_inputs(1300, 1, 2, 64, seed=79, pool_size=2700)
    idx = d["cache_indices"].clone()
    idx[pos[1]] = idx[pos[0]]
    d["cache_indices"] = idx
    g = to_device(d)
    with pytest.raises(GdnError) as e:
        gdn_decode_step(*[g[k] for k in DEC_KEYS], check=True)
    assert e.value.status == 3
    assert torch.equal(g["state_pool"].cpu(), d["state_pool"]), "a rejected step changed the pool"
    # the status word is reset by the next good step
    d2 = decode_inputs(1300, 1, 2, 64, seed=80, pool_size=2700)
    g2 = to_device(d2)
    gdn_decode_step(*[g2[k] for k in DEC_KEYS], check=True)
