"""The C-ABI library builds, loads, and exports every symbol include/gdn.h declares.

CPU only: the calls made here return from host-side validation before any CUDA
call (null pointers, unsupported sizes, bad workspace).
"""

import ctypes
import os
import re

import pytest

from gated_deltanet_chunkwise_gdn_gb300 import _lib, build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    return re.findall(r"GDN_API\s+[\w\s\*]*?\b(gdn_\w+)\s*\(", text)


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_header_declares_the_abi():
    names = _declared_functions()
    assert {"gdn_extend_chunkwise", "gdn_workspace_size", "gdn_get_device_status",
            "gdn_status_string", "gdn_version"} <= set(names)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in gdn.h but not exported"


def test_only_the_abi_is_exported(lib):
    import subprocess
    r = subprocess.run(["nm", "-D", "--defined-only", gbuild.LIB_PATH], capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("nm not available")
    exported = {ln.split()[-1] for ln in r.stdout.splitlines() if " T " in ln}
    assert exported == set(_declared_functions())


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        s = lib.gdn_status_string(code).decode()
        assert s.startswith(name)
    assert lib.gdn_status_string(99).decode() == "GDN_ERR_UNKNOWN"
    assert lib.gdn_version() >= 100


def test_workspace_size_rules(lib):
    ws = lib.gdn_workspace_size
    assert ws(65536, 1, 16, 16, 128, 128, 64) > 0
    assert ws(0, 0, 1, 1, 64, 64, 64) > 0
    assert ws(100, 2, 3, 4, 128, 128, 64) == 0     # HV not a multiple of H
    assert ws(100, 2, 2, 4, 96, 96, 64) == 0       # head size not built
    assert ws(100, 2, 2, 4, 128, 64, 64) == 0      # K != V
    assert ws(100, 2, 2, 4, 128, 128, 32) == 0     # chunk size not built
    assert ws(-1, 2, 2, 4, 128, 128, 64) == 0
    assert ws(100, 2, 2, 4, 256, 256, 128) > 0     # wide heads, 128-token chunks
    # a 128-token chunk runs as two 64-token WY blocks: the same workspace
    assert ws(1000, 2, 2, 4, 128, 128, 128) == ws(1000, 2, 2, 4, 128, 128, 64)
    # grows with tokens and value heads
    assert ws(2000, 2, 2, 4, 128, 128, 64) > ws(1000, 2, 2, 4, 128, 128, 64)
    assert ws(1000, 2, 2, 8, 128, 128, 64) > ws(1000, 2, 2, 4, 128, 128, 64)


def _call(lib, **over):
    args = dict(q=1, k=1, v=1, dtype=0, a=1, b=1, A_log=1, dt_bias=1, pool=1, pool_size=4, idx=1, cu=1,
                batch=2, out=1, T=100, H=2, HV=4, K=128, V=128, C=64, scale=1.0, ws=256, ws_bytes=1 << 40,
                stream=None)
    args.update(over)
    return lib.gdn_extend_chunkwise(*[args[k] for k in (
        "q", "k", "v", "dtype", "a", "b", "A_log", "dt_bias", "pool", "pool_size", "idx", "cu", "batch",
        "out", "T", "H", "HV", "K", "V", "C", "scale", "ws", "ws_bytes", "stream")])


def test_host_side_errors_return_before_any_device_work(lib):
    assert _call(lib, HV=3) == 1             # HV % H != 0
    assert _call(lib, q=None) == 1           # null input
    assert _call(lib, cu=None) == 1
    assert _call(lib, batch=-1) == 1
    assert _call(lib, dtype=7) == 1
    assert _call(lib, K=96, V=96) == 2       # not built
    assert _call(lib, C=32) == 2
    assert _call(lib, dtype=-1) == 1         # no such dtype
    assert _call(lib, ws=None) == 4          # workspace
    assert _call(lib, ws=264) == 4           # misaligned
    assert _call(lib, ws_bytes=16) == 4      # too small


def test_product_path_has_no_fallback(monkeypatch):
    """With the library missing, the binding raises instead of computing anything."""
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(gbuild, "LIB_PATH", "/nonexistent/libgdn_gb300.so")
    with pytest.raises(RuntimeError):
        _lib.load(build_if_missing=False)


def _decode(lib, **over):
    args = dict(q=16, k=16, v=16, dtype=0, a=16, b=16, A_log=16, dt_bias=16, pool=16, pool_size=4, idx=16,
                batch=2, out=16, H=2, HV=4, K=128, V=128, scale=1.0, status=16, stream=None)
    args.update(over)
    return lib.gdn_decode_step(*[args[k] for k in (
        "q", "k", "v", "dtype", "a", "b", "A_log", "dt_bias", "pool", "pool_size", "idx", "batch", "out",
        "H", "HV", "K", "V", "scale", "status", "stream")])


def test_decode_host_side_errors_return_before_any_device_work(lib):
    assert _decode(lib, HV=3) == 1             # HV % H != 0
    assert _decode(lib, q=None) == 1           # null input
    assert _decode(lib, status=None) == 1      # no status word
    assert _decode(lib, status=18) == 1        # misaligned status word
    assert _decode(lib, pool=24) == 1          # state pool not 16-byte aligned
    assert _decode(lib, out=8) == 1            # output not 16-byte aligned
    assert _decode(lib, batch=-1) == 1
    assert _decode(lib, batch=(1 << 20) + 1) == 1
    assert _decode(lib, batch=1 << 20, HV=4096, H=1) == 1  # grid would exceed 2^31 - 1 blocks
    assert _decode(lib, dtype=5) == 1
    assert _decode(lib, pool_size=0) == 1
    assert _decode(lib, K=96, V=96) == 2       # not built
    assert _decode(lib, K=128, V=64) == 2


def test_calls_beyond_the_factor_row_limit_are_refused(lib):
    """(T/64 + B + 1) * HV * 64 rows of per-chunk factors must fit 32-bit TMA coordinates."""
    ws = lib.gdn_workspace_size
    assert ws(1 << 25, 1 << 25, 1, 1, 64, 64, 64) == 0          # 2^25 one-token sequences, one head
    assert ws(1 << 20, 1 << 20, 1, 4, 64, 64, 64) > 0
    assert ws(1 << 28, 1, 1, 8, 64, 64, 64) == 0                # 2^28 tokens x 8 value heads
    assert _call(lib, T=1 << 25, batch=1 << 25, H=1, HV=1, K=64, V=64) == 2


def test_kernel_kinds_named_for_the_profiler(lib):
    names = [lib.gdn_kernel_name(i) for i in range(8)]
    assert [n.decode() for n in names[:7]] == ["schedule", "gates", "intra", "scan", "decode_check", "decode",
                                               "backward"]
    assert names[7] is None and lib.gdn_kernel_name(-1) is None


def test_backward_workspace_size_rules(lib):
    ws = lib.gdn_backward_workspace_size
    assert ws(65536, 1, 16, 16, 128, 128, 64) > 0
    assert ws(0, 0, 1, 1, 64, 64, 64) > 0
    assert ws(100, 2, 3, 4, 128, 128, 64) == 0     # HV not a multiple of H
    assert ws(100, 2, 2, 4, 256, 256, 128) == 0    # wide heads: no backward
    assert ws(100, 2, 2, 4, 128, 64, 64) == 0      # K != V
    assert ws(100, 2, 2, 4, 128, 128, 32) == 0     # chunk size
    assert ws(100, 2, 1, 1 << 16, 64, 64, 64) == 0  # HV above the grid's y limit
    assert ws((1 << 31) - 64, 1, 16, 16, 64, 64, 64) == 0  # (T H + 7) / 8 norm blocks above the grid limit
    assert ws(1000, 2, 2, 4, 128, 128, 128) == ws(1000, 2, 2, 4, 128, 128, 64)
    # (C*C*2 + C*D*7 + D*D*2) 4-byte words per (chunk, value head); per (token, value head) one word, plus
    # 2*D for the per-value-head q/k gradients when value heads share a q/k head
    per_item = (64 * 64 * 2 + 64 * 128 * 7 + 128 * 128 * 2) * 4
    assert ws(65536, 1, 16, 16, 128, 128, 64) >= 1025 * 16 * per_item + 65536 * 16 * 4
    assert ws(65536, 1, 16, 16, 128, 128, 64) < 1025 * 16 * per_item + 65536 * 16 * 2 * 128 * 4
    assert ws(65536, 1, 8, 16, 128, 128, 64) >= 1025 * 16 * per_item + 65536 * 16 * (2 * 128 + 1) * 4


def _bwd(lib, **over):
    args = dict(q=16, k=16, v=16, dtype=0, a=16, b=16, A_log=16, dt_bias=16, pool=16, pool_size=4, idx=16, cu=16,
                batch=2, d_out=16, d_state=None, dq=16, dk=16, dv=16, da=16, db=16, dA_log=16, ddt_bias=16,
                d_pool=16, T=100, H=2, HV=4, K=128, V=128, C=64, scale=1.0, ws=256, ws_bytes=1 << 40, stream=None)
    args.update(over)
    return lib.gdn_chunkwise_backward(*[args[k] for k in (
        "q", "k", "v", "dtype", "a", "b", "A_log", "dt_bias", "pool", "pool_size", "idx", "cu", "batch",
        "d_out", "d_state", "dq", "dk", "dv", "da", "db", "dA_log", "ddt_bias", "d_pool",
        "T", "H", "HV", "K", "V", "C", "scale", "ws", "ws_bytes", "stream")])


def test_backward_host_side_errors_return_before_any_device_work(lib):
    assert _bwd(lib, HV=3) == 1              # HV % H != 0
    assert _bwd(lib, q=None) == 1            # null input
    assert _bwd(lib, d_out=None) == 1
    assert _bwd(lib, dq=None) == 1           # null output
    assert _bwd(lib, dA_log=None) == 1
    assert _bwd(lib, d_pool=None) == 1
    assert _bwd(lib, dtype=3) == 1
    assert _bwd(lib, q=24) == 1              # tiles are copied in 16-byte pieces
    assert _bwd(lib, dv=12) == 1             # 8-byte stores
    assert _bwd(lib, dq=24) == 1             # 16-byte stores
    assert _bwd(lib, K=256, V=256) == 2      # not built for the backward
    assert _bwd(lib, C=32) == 2
    assert _bwd(lib, ws=None) == 4
    assert _bwd(lib, ws=264) == 4
    assert _bwd(lib, ws_bytes=16) == 4
