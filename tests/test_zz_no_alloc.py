"""The allocation-free entry point gives the same results as the regular one.

gdn_extend_chunkwise_noalloc exists for callers that are handed device buffers but may
not allocate device memory themselves (a plugin inside a runtime that owns all device
memory, or a serving loop that forbids cudaMalloc/cudaFree once running). It runs on a
64 MiB scratch array built into the library instead of a caller workspace. This test
calls it through the C ABI several times in a row and checks each call against
gdn_extend_chunkwise on the same inputs and the same starting state: within the
tolerance the parity tests use, and in fact bit for bit, since both entry points run the
same deterministic kernels. The scratch keeps what the previous call left, so a call with
another shape (other head size, more segments) follows the first ones, and a call with a
repeated cache index must report GDN_ERR_BAD_INDEX through the caller's status word and
leave the pool untouched. It sits in its own file, collected last, and passes both alone in
a fresh process and after the other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

from gated_deltanet_chunkwise_gdn_gb300 import _lib, gdn_extend_chunkwise, workloads as wl
from gpu_helpers import INPUT_KEYS, OUT_TOL, STATE_TOL, rel_l2

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _noalloc(lib, g, pool, out, status, chunk_size=64):
    T, H, K = g["q"].shape
    HV, V = g["v"].shape[1], g["v"].shape[2]
    return lib.gdn_extend_chunkwise_noalloc(
        g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(), _lib.GDN_BF16,
        g["a"].data_ptr(), g["b"].data_ptr(), g["A_log"].data_ptr(), g["dt_bias"].data_ptr(),
        pool.data_ptr(), pool.shape[0], g["cache_indices"].data_ptr(), g["cu_seqlens"].data_ptr(),
        g["cache_indices"].shape[0], out.data_ptr(), T, H, HV, K, V, chunk_size, 1.0,
        status.data_ptr() if status is not None else None, torch.cuda.current_stream().cuda_stream)


def _check_pair(lib, w, calls, status):
    """`calls` calls in a row on workload w through both entry points, compared after each."""
    d = wl.make_inputs(w)
    g = {k: d[k].cuda() for k in INPUT_KEYS}
    pool_ref = g["state_pool"].clone()
    pool_new = g["state_pool"].clone()
    for call in range(calls):  # each call continues from the state the previous one left
        out_ref = gdn_extend_chunkwise(*[g[k] for k in INPUT_KEYS[:7]], pool_ref, g["cache_indices"],
                                       g["cu_seqlens"], chunk_size=w.chunk_size, check=True)
        out_new = torch.empty_like(out_ref)
        status.fill_(-1)
        st = _noalloc(lib, g, pool_new, out_new, status, chunk_size=w.chunk_size)
        assert st == 0, _lib.status_string(st)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert rel_l2(out_new.float().cpu().numpy(), out_ref.float().cpu().numpy()) <= OUT_TOL, call
        assert rel_l2(pool_new.cpu().numpy(), pool_ref.cpu().numpy()) <= STATE_TOL, call
        # the same kernels on the same inputs: identical bits
        assert torch.equal(out_new, out_ref), call
        assert torch.equal(pool_new, pool_ref), call


def test_noalloc_matches_regular_entry_point_on_two_calls():
    lib = _lib.load()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    w = wl.custom("noalloc", [300, 77, 64, 1], H=2, HV=4, K=128, V=128, chunk_size=64, seed=41)
    _check_pair(lib, w, 2, status)
    # then other shapes on the same scratch: a smaller head size, and a long sequence whose
    # scan runs in segments (segment states and maps in the scratch, none of them zeroed)
    _check_pair(lib, wl.custom("noalloc64", [5, 190, 64], H=1, HV=2, K=64, V=64, chunk_size=64, seed=43),
                1, status)
    _check_pair(lib, wl.custom("noalloc_seg", [8192], H=1, HV=1, K=128, V=128, chunk_size=64, seed=44),
                2, status)


def test_noalloc_reports_a_repeated_slot_through_the_status_word():
    lib = _lib.load()
    w = wl.custom("noalloc_bad", [70, 40], H=1, HV=2, K=128, V=128, chunk_size=64, seed=45)
    d = wl.make_inputs(w)
    g = {k: d[k].cuda() for k in INPUT_KEYS}
    g["cache_indices"] = torch.tensor([0, 0], dtype=torch.int64, device="cuda")
    pool = g["state_pool"].clone()
    out = torch.zeros_like(g["v"])
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    st = _noalloc(lib, g, pool, out, status)
    assert st == 0, _lib.status_string(st)  # detected on the device, not on the host
    torch.cuda.synchronize()
    assert int(status.item()) == 3  # GDN_ERR_BAD_INDEX
    assert torch.equal(pool, g["state_pool"])
    assert bool((out == 0).all())
    # a misaligned status pointer is refused on the host and nothing is enqueued
    raw = torch.zeros(4, dtype=torch.int32, device="cuda")
    bad = ctypes.c_void_p(raw.data_ptr() + 2)
    good_idx = d["cache_indices"].cuda()
    T, H, K = g["q"].shape
    st = lib.gdn_extend_chunkwise_noalloc(
        g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(), _lib.GDN_BF16,
        g["a"].data_ptr(), g["b"].data_ptr(), g["A_log"].data_ptr(), g["dt_bias"].data_ptr(),
        pool.data_ptr(), pool.shape[0], good_idx.data_ptr(), g["cu_seqlens"].data_ptr(), 2,
        out.data_ptr(), T, H, 2, K, 128, 64, 1.0, bad, torch.cuda.current_stream().cuda_stream)
    assert st == 1  # GDN_ERR_INVALID_ARG
    # and a good call afterwards on the same scratch succeeds
    _check_pair(lib, w, 1, status)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _lib.load()
    # 65536 tokens x 16 heads needs far more than the 64 MiB built-in scratch
    assert lib.gdn_workspace_size(65536, 1, 16, 16, 128, 128, 64) > 64 << 20
    w = wl.custom("noalloc_small", [16], H=1, HV=1, K=128, V=128, chunk_size=64, seed=42)
    d = wl.make_inputs(w)
    g = {k: d[k].cuda() for k in INPUT_KEYS}
    out = torch.zeros((16, 1, 128), dtype=torch.bfloat16, device="cuda")
    st = lib.gdn_extend_chunkwise_noalloc(
        g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(), _lib.GDN_BF16,
        g["a"].data_ptr(), g["b"].data_ptr(), g["A_log"].data_ptr(), g["dt_bias"].data_ptr(),
        g["state_pool"].data_ptr(), 1, g["cache_indices"].data_ptr(), g["cu_seqlens"].data_ptr(), 1,
        out.data_ptr(), 65536, 16, 16, 128, 128, 64, 1.0, None, torch.cuda.current_stream().cuda_stream)
    assert st == 4  # GDN_ERR_WORKSPACE, returned before anything is enqueued
    torch.cuda.synchronize()
    assert bool((out == 0).all())
