"""GPU parity: the CUDA path through the C ABI vs the fp64 oracle, same seeded inputs.

Bar: relative L2 <= 1e-2 on the bf16 outputs and <= 5e-3 on the final fp32 states,
element by element over every compared chain; untouched pool slots bit-identical.
"""

import numpy as np
import pytest
import torch

from gated_deltanet_chunkwise_gdn_gb300 import GdnError, gdn_extend_chunkwise, workloads as wl
from gpu_helpers import (INPUT_KEYS, compare, oracle_for, rel_l2, run_gpu, to_device,
                         untouched_slots_equal)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU runs, skipped there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


# ----------------------------------------------------------------------------- the five configs

def test_config_tiny_full():
    d = wl.make_inputs(wl.BY_NAME["tiny"])
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))


def test_config_varlen_full():
    d = wl.make_inputs(wl.BY_NAME["varlen"])
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))
    untouched_slots_equal(d, pool)


def test_config_long_full():
    """B=1, T=65536, H=HV=16, K=V=128: every chain, every token."""
    d = wl.make_inputs(wl.BY_NAME["long"])
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))


def test_config_long_weak_decay_full():
    """The long prefill with A_log = -7 (log alpha about -6e-4 per token): the state carries
    across hundreds of chunks, so every segment of the scan starts from a state that matters
    (10 segments x 16 heads); every chain, every token."""
    d = wl.make_inputs(wl.BY_NAME["long"])
    d["A_log"].fill_(-7.0)
    d["state_pool"].normal_(0.0, 0.1, generator=torch.Generator().manual_seed(99))
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))


def test_segmented_scan_with_mixed_decay_across_heads():
    """Two value heads of one long sequence in one call (the segmented scan), one with weak decay
    (A_log = -7: every segment's start state carries the whole prefix) and one with the default
    gates; every token of both."""
    w = wl.custom("mixed", [8192, 200], H=1, HV=2, K=128, V=128, chunk_size=64, seed=33)
    d = wl.make_inputs(w)
    d["A_log"][0] = -7.0
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))
    untouched_slots_equal(d, pool)


def test_exact_linearity_in_state_and_values():
    """The recurrence is linear in (S0, v): doubling both doubles out and the final state. Every
    scaling on the GPU path is by a power of two, so the results double bit for bit (the
    segmented scan is included: 8192 tokens of one head run in segments)."""
    w = wl.custom("linear", [8192, 300, 1], H=1, HV=2, K=128, V=128, chunk_size=64, seed=31)
    d = wl.make_inputs(w)
    out1, pool1 = run_gpu(d)
    d2 = dict(d)
    d2["v"] = (d["v"].float() * 2).to(d["v"].dtype)
    d2["state_pool"] = d["state_pool"] * 2
    assert torch.equal(d2["v"].float(), d["v"].float() * 2)
    out2, pool2 = run_gpu(d2)
    assert torch.equal(out2.float(), out1.float() * 2)
    assert torch.equal(pool2, pool1 * 2)


def test_config_throughput_every_chain():
    """B=32 x 8192, H=HV=32: all 1024 (sequence, head) chains, every token, the oracle run four sequences
    (128 chains) at a time so that its fp64 outputs stay small; each batch is held to the tolerances."""
    d = wl.make_inputs(wl.BY_NAME["throughput"])
    out, pool = run_gpu(d)
    B, HV = len(d["cache_indices"]), d["v"].shape[1]
    for s0 in range(0, B, 4):
        chains = np.array([(s, hv) for s in range(s0, min(B, s0 + 4)) for hv in range(HV)])
        compare(d, out, pool, oracle_for(d, chains=chains))
    untouched_slots_equal(d, pool)


def test_config_wide_full():
    """B=4 x 16384, H=HV=4, K=V=256, 128-token chunks, a shifted by -2: every chain, every token."""
    d = wl.make_inputs(wl.BY_NAME["wide"])
    assert d["chunk_size"] == 128 and d["q"].shape[-1] == 256
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))


# ----------------------------------------------------------------------------- shapes and edge cases

@pytest.mark.parametrize("D", [64, 128, 256])
def test_ragged_lengths_and_gqa(D):
    """Lengths around the chunk size (1, C-1, C, C+1, 0, several chunks + tail), GQA 1:2."""
    w = wl.custom("ragged", [1, 63, 64, 65, 0, 200, 130], H=2, HV=4, K=D, V=D, chunk_size=64, seed=21)
    d = wl.make_inputs(w)
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))
    untouched_slots_equal(d, pool)
    # the zero-length sequence left its slot exactly as it was
    s_empty = int(d["cache_indices"][4])
    assert torch.equal(pool[s_empty], d["state_pool"][s_empty])


def test_gqa_ratio_four():
    w = wl.custom("gqa4", [300, 77], H=1, HV=4, K=128, V=128, chunk_size=64, seed=22)
    d = wl.make_inputs(w)
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))


def test_many_short_sequences():
    rng = np.random.default_rng(23)
    lens = rng.integers(1, 40, 100).tolist()
    w = wl.custom("short", lens, H=2, HV=2, K=64, V=64, chunk_size=64, seed=23, pool_size=128)
    d = wl.make_inputs(w)
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))


def test_strong_decay_stays_finite():
    """a ~ N(4, 1): sum of log alpha per chunk far below -87 (1/gamma would overflow fp32)."""
    w = wl.custom("strong", [500, 129], H=2, HV=2, K=128, V=128, chunk_size=64, seed=24, a_mean=4.0)
    d = wl.make_inputs(w)
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))


def test_weak_decay_long_memory():
    """A_log very negative: alpha ~ 1, the state carries across many chunks."""
    w = wl.custom("weak", [700], H=1, HV=2, K=64, V=64, chunk_size=64, seed=25)
    d = wl.make_inputs(w)
    d["A_log"] = torch.full_like(d["A_log"], -8.0)
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))


def test_scale_argument():
    w = wl.custom("scale", [100], H=1, HV=1, K=64, V=64, chunk_size=64, seed=26)
    d = wl.make_inputs(w)
    s = 64 ** -0.5
    out, pool = run_gpu(d, scale=s)
    compare(d, out, pool, oracle_for(d, scale=s))


def test_split_call_continuation():
    """extend(T1) then extend(T - T1) on the same slot equals extend(T)."""
    w = wl.custom("split", [333], H=2, HV=2, K=128, V=128, chunk_size=64, seed=27)
    d = wl.make_inputs(w)
    out_all, pool_all = run_gpu(d)
    T1 = 130
    d1 = dict(d, **{k: d[k][:T1] for k in ("q", "k", "v", "a", "b")}, cu_seqlens=torch.tensor([0, T1]))
    out1, pool1 = run_gpu(d1)
    d2 = dict(d, **{k: d[k][T1:] for k in ("q", "k", "v", "a", "b")}, cu_seqlens=torch.tensor([0, 333 - T1]),
              state_pool=pool1)
    out2, pool2 = run_gpu(d2)
    res = oracle_for(d)
    compare(d, out_all, pool_all, res)
    compare(d, torch.cat([out1, out2]), pool2, res)   # the split calls meet the same bar


def test_deterministic():
    w = wl.custom("det", [257, 31], H=2, HV=4, K=128, V=128, chunk_size=64, seed=28)
    d = wl.make_inputs(w)
    o1, p1 = run_gpu(d)
    o2, p2 = run_gpu(d)
    assert torch.equal(o1, o2) and torch.equal(p1, p2)


# ----------------------------------------------------------------------------- error paths

def _sentinel_call(d, **over):
    g = to_device(dict(d, **over))
    out = torch.full((d["q"].shape[0], d["v"].shape[1], d["v"].shape[2]), 7.0, dtype=torch.bfloat16,
                     device="cuda")
    pool = g["state_pool"]
    with pytest.raises(GdnError) as ei:
        gdn_extend_chunkwise(*[g[k] for k in INPUT_KEYS[:7]], pool, g["cache_indices"], g["cu_seqlens"],
                             chunk_size=64, out=out, check=True)
    torch.cuda.synchronize()
    assert torch.equal(pool.cpu(), d["state_pool"]), "state_pool modified by a rejected call"
    assert bool((out == 7.0).all()), "out written by a rejected call"
    return ei.value.status


def test_bad_cache_indices_rejected_on_device():
    w = wl.custom("bad", [40, 50], H=1, HV=2, K=64, V=64, chunk_size=64, seed=29, pool_size=4)
    d = wl.make_inputs(w)
    assert _sentinel_call(d, cache_indices=torch.tensor([1, 1])) == 3
    assert _sentinel_call(d, cache_indices=torch.tensor([0, 4])) == 3
    assert _sentinel_call(d, cache_indices=torch.tensor([-1, 2])) == 3


def test_bad_cu_seqlens_rejected_on_device():
    w = wl.custom("badcu", [40, 50], H=1, HV=2, K=64, V=64, chunk_size=64, seed=30, pool_size=4)
    d = wl.make_inputs(w)
    assert _sentinel_call(d, cu_seqlens=torch.tensor([0, 60, 50])) == 7   # last != total, decreasing
    assert _sentinel_call(d, cu_seqlens=torch.tensor([1, 41, 90])) == 7   # does not start at 0
    # and a good call afterwards works on the same workspace
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))


def test_host_errors_raise():
    w = wl.custom("hosterr", [10], H=2, HV=2, K=64, V=64, chunk_size=64, seed=31)
    d = to_device(wl.make_inputs(w))
    with pytest.raises(GdnError):
        gdn_extend_chunkwise(*[d[k] for k in INPUT_KEYS], chunk_size=48)
    with pytest.raises(TypeError):
        gdn_extend_chunkwise(d["q"].float(), *[d[k] for k in INPUT_KEYS[1:]])


# ----------------------------------------------------------------------------- segment-parallel scan

def test_segmented_scan_long_sequence():
    """Few heads, one long sequence: the scan splits it into segments, computes the affine
    map of the middle one, chains it, and re-runs the segments from their start states."""
    w = wl.custom("seg", [6400], H=1, HV=2, K=128, V=128, chunk_size=64, seed=32)
    d = wl.make_inputs(w)
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))


def test_segmented_scan_weak_decay():
    """alpha ~ 1: the segment transition maps are far from zero, so the chaining matters."""
    w = wl.custom("segweak", [6400], H=1, HV=2, K=128, V=128, chunk_size=64, seed=33)
    d = wl.make_inputs(w)
    d["A_log"] = torch.full_like(d["A_log"], -7.0)
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))


@pytest.mark.parametrize("dtype,a_log", [(torch.bfloat16, None), (torch.bfloat16, -7.0), (torch.float16, -7.0)])
def test_segmented_scan_many_segments_gqa(dtype, a_log):
    """K = V = 128, GQA 1:2, nonzero start states, sequences of very different lengths: the
    longest is cut into nine segments (a shorter segment 0 with outputs and seven affine
    maps in the first pass, the chaining, the re-runs), a two-chunk sequence into two
    segments (no map), a one-token sequence into one."""
    w = wl.custom("segmany", [12000, 7000, 65, 1], H=1, HV=2, K=128, V=128, chunk_size=64, seed=37,
                  dtype=dtype)
    d = wl.make_inputs(w)
    if a_log is not None:
        d["A_log"] = torch.full_like(d["A_log"], a_log)
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))
    untouched_slots_equal(d, pool)


@pytest.mark.parametrize("a_log", [None, -7.0])
def test_segmented_scan_short_middle_segments(a_log):
    """K = V = 128 with one long sequence next to sequences of 8, 9 and 11 chunks, cut into eight
    segments each: the 8-chunk sequence's middle segments are one chunk long (the affine map pass runs
    a single transition: no second -M buffer, no reuse), the others two chunks (one reuse of each)."""
    w = wl.custom("segshort", [16000, 500, 576, 700], H=1, HV=2, K=128, V=128, chunk_size=64, seed=43)
    d = wl.make_inputs(w)
    if a_log is not None:
        d["A_log"] = torch.full_like(d["A_log"], a_log)
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))
    untouched_slots_equal(d, pool)


def test_segmented_scan_wide_heads():
    """K = V = 256 with one long sequence: segment maps, the chaining over four middle
    segments (state staged 32 key rows at a time) and the segment re-runs."""
    w = wl.custom("segwide", [12800], H=1, HV=1, K=256, V=256, chunk_size=64, seed=35)
    d = wl.make_inputs(w)
    d["A_log"] = torch.full_like(d["A_log"], -6.0)
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))


def test_chunk_size_128_matches_oracle():
    """chunk_size=128 (two 64-token WY blocks per chunk) against the oracle, on ragged
    lengths around both block lengths."""
    w = wl.custom("c128", [1, 127, 128, 129, 300], H=2, HV=4, K=128, V=128, chunk_size=128, seed=36)
    d = wl.make_inputs(w)
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))
    untouched_slots_equal(d, pool)


# ----------------------------------------------------------------------------- fp16 inputs

@pytest.mark.parametrize("D", [64, 128, 256])
def test_fp16_ragged_lengths_and_gqa(D):
    """fp16 q/k/v (and output): every tensor-core operand in fp16, lengths around the
    chunk size, GQA 1:2."""
    w = wl.custom("ragged16", [1, 63, 64, 65, 0, 200, 130], H=2, HV=4, K=D, V=D, chunk_size=64, seed=41,
                  dtype=torch.float16)
    d = wl.make_inputs(w)
    assert d["q"].dtype == torch.float16
    out, pool = run_gpu(d)
    assert out.dtype == torch.float16
    compare(d, out, pool, oracle_for(d))
    untouched_slots_equal(d, pool)


def test_fp16_segmented_long_sequence_weak_decay():
    """fp16 through the segment-parallel scan, with alpha ~ 1 so errors would accumulate."""
    w = wl.custom("seg16", [6400], H=1, HV=2, K=128, V=128, chunk_size=64, seed=42, dtype=torch.float16)
    d = wl.make_inputs(w)
    d["A_log"] = torch.full_like(d["A_log"], -7.0)
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))


def test_fp16_and_bf16_of_the_same_values():
    """The bf16 inputs and their fp16 conversion (nearly all values exact in fp16), each
    against the oracle on its own input bits; the two GPU outputs agree to 16-bit rounding."""
    w = wl.custom("same", [300, 129], H=2, HV=2, K=128, V=128, chunk_size=64, seed=43)
    d = wl.make_inputs(w)
    d16 = dict(d)
    for k in ("q", "k", "v"):
        d16[k] = d[k].to(torch.float16)
    out_b, pool_b = run_gpu(d)
    out_h, pool_h = run_gpu(d16)
    compare(d, out_b, pool_b, oracle_for(d))
    compare(d16, out_h, pool_h, oracle_for(d16))
    assert rel_l2(out_h.float().numpy(), out_b.float().numpy()) < 1e-2


def test_segmented_scan_mixed_lengths():
    w = wl.custom("segmix", [5000, 700, 1], H=1, HV=1, K=64, V=64, chunk_size=64, seed=34)
    d = wl.make_inputs(w)
    d["A_log"] = torch.full_like(d["A_log"], -6.0)
    out, pool = run_gpu(d)
    compare(d, out, pool, oracle_for(d))
    untouched_slots_equal(d, pool)
