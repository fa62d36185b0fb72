"""The allocation-free entry point gives the same results as the regular one.

gdn_extend_chunkwise_noalloc exists for callers that are handed device buffers but may
not allocate device memory themselves (a plugin inside a runtime that owns all device
memory, or a serving loop that forbids cudaMalloc/cudaFree once running). It runs on a
64 MiB scratch array built into the library instead of a caller workspace. This test
calls it through the C ABI twice in a row and checks each call against
gdn_extend_chunkwise on the same inputs and the same starting state, with the tolerance
the parity tests use. It sits in its own file, collected last, and passes both alone in a
fresh process and after the other tests.
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


def test_noalloc_matches_regular_entry_point_on_two_calls():
    lib = _lib.load()
    w = wl.custom("noalloc", [300, 77, 64, 1], H=2, HV=4, K=128, V=128, chunk_size=64, seed=41)
    d = wl.make_inputs(w)
    g = {k: d[k].cuda() for k in INPUT_KEYS}
    pool_ref = g["state_pool"].clone()
    pool_new = g["state_pool"].clone()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):  # the second call continues from the state the first one left
        out_ref = gdn_extend_chunkwise(*[g[k] for k in INPUT_KEYS[:7]], pool_ref, g["cache_indices"],
                                       g["cu_seqlens"], chunk_size=64, check=True)
        out_new = torch.empty_like(out_ref)
        st = _noalloc(lib, g, pool_new, out_new, status)
        assert st == 0, _lib.status_string(st)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert rel_l2(out_new.float().cpu().numpy(), out_ref.float().cpu().numpy()) <= OUT_TOL, call
        assert rel_l2(pool_new.cpu().numpy(), pool_ref.cpu().numpy()) <= STATE_TOL, call


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
