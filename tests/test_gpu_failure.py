"""Failure handling on the GPU without faulting it.

* Bounded waits: a test hook makes one kernel's CTAs issue none of their tile loads, so every
  mbarrier wait in them has nothing to wait for and runs out after a short budget. The call
  must record GDN_ERR_TIMEOUT, leave the state pool (and here the output) untouched, every
  role must leave through the kernel's final barrier (where TMEM is freed), and the next call
  on the same workspace must succeed and match the oracle.
* Guard words: the output and the workspace sit between canary regions, which must come back
  unchanged after a call: nothing is written outside the caller's buffers.
"""

import pytest
import torch

from gated_deltanet_chunkwise_gdn_gb300 import GdnError, _lib, gdn_extend_chunkwise, workloads as wl
from gpu_helpers import INPUT_KEYS, compare, oracle_for, run_gpu, to_device

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

GDN_ERR_TIMEOUT = 5
SHORT_BUDGET = 1 << 20  # SM clock cycles, about half a millisecond


def _stall_case(kernel):
    if kernel in (1, 2):  # K = 64, one whole-sequence scan
        return wl.custom("stall", [200, 64], H=2, HV=4, K=64, V=64, chunk_size=64, seed=71)
    # K = V = 128, long enough for the segmented scan (its first pass is the stalled kernel)
    return wl.custom("stall_seg", [8192], H=1, HV=1, K=128, V=128, chunk_size=64, seed=72)


@pytest.mark.parametrize("kernel", [1, 2, 3], ids=["intra", "scan", "affine_scan"])
def test_a_wait_that_runs_out_reports_timeout_and_touches_nothing(kernel):
    lib = _lib.load()
    d = wl.make_inputs(_stall_case(kernel))
    g = to_device(d)
    pool0 = g["state_pool"].clone()
    sentinel = torch.full_like(g["v"], 7.0)
    out = sentinel.clone()
    ws = torch.zeros(lib.gdn_workspace_size(*d["q"].shape[:1], d["cache_indices"].shape[0], d["q"].shape[1],
                                            d["v"].shape[1], d["q"].shape[2], d["v"].shape[2], 64) + 256,
                     dtype=torch.uint8, device="cuda")
    assert lib.gdn_test_set_stall(kernel, SHORT_BUDGET) == 0
    try:
        with pytest.raises(GdnError) as e:
            gdn_extend_chunkwise(*[g[k] for k in INPUT_KEYS], chunk_size=64, out=out, workspace=ws, check=True)
    finally:
        assert lib.gdn_test_set_stall(0, 1) == 0
    assert e.value.status == GDN_ERR_TIMEOUT, str(e.value)
    torch.cuda.synchronize()  # the context is still usable
    assert torch.equal(g["state_pool"], pool0)
    assert torch.equal(out, sentinel)
    # the next call on the same workspace runs normally and matches the oracle
    o = gdn_extend_chunkwise(*[g[k] for k in INPUT_KEYS], chunk_size=64, workspace=ws, check=True)
    torch.cuda.synchronize()
    compare(d, o.cpu(), g["state_pool"].cpu(), oracle_for(d))


def test_the_stall_hook_rejects_bad_arguments():
    lib = _lib.load()
    assert lib.gdn_test_set_stall(4, 100) == 1
    assert lib.gdn_test_set_stall(1, 0) == 1
    assert lib.gdn_test_set_stall(0, 1) == 0


@pytest.mark.parametrize("D,lengths", [(64, [100, 64, 1]), (128, [8192, 37]), (256, [300, 5])])
def test_nothing_is_written_outside_the_callers_buffers(D, lengths):
    lib = _lib.load()
    d = wl.make_inputs(wl.custom("guard", lengths, H=2, HV=2, K=D, V=D, chunk_size=64, seed=73))
    g = to_device(d)
    T, HV = d["v"].shape[0], d["v"].shape[1]
    B = d["cache_indices"].shape[0]
    GUARD = 4096  # bytes on each side; keeps the workspace 256-byte aligned
    n_out = T * HV * D
    out_buf = torch.full((n_out + 2 * GUARD // 2,), -3.0, dtype=torch.bfloat16, device="cuda")
    out = out_buf[GUARD // 2:GUARD // 2 + n_out].view(T, HV, D)
    need = lib.gdn_workspace_size(T, B, 2, HV, D, D, 64)
    ws_buf = torch.full((need + 2 * GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    base = ws_buf.data_ptr()
    assert base % 256 == 0
    ws = ws_buf[GUARD:GUARD + need]
    gdn_extend_chunkwise(*[g[k] for k in INPUT_KEYS], chunk_size=64, out=out, workspace=ws, check=True)
    torch.cuda.synchronize()
    assert bool((out_buf[:GUARD // 2] == -3.0).all()) and bool((out_buf[GUARD // 2 + n_out:] == -3.0).all())
    assert bool((ws_buf[:GUARD] == 0xA5).all()) and bool((ws_buf[GUARD + need:] == 0xA5).all())
    compare(d, out.cpu(), g["state_pool"].cpu(), oracle_for(d))
