"""GB300-native chunkwise Gated DeltaNet (GDN) prefill.

Python binding of the C ABI in include/gdn.h. Argument marshalling only: every
step of the computation runs in the CUDA kernels of libgdn_gb300.so, and there
is no CPU or PyTorch fallback (a missing library raises).

The entry point mirrors ``gdn_extend_chunkwise(q, k, v, a, b, A_log, dt_bias,
state_pool, cache_indices, cu_seqlens, chunk_size=64)`` of the pymllm page
"pymllm.layers.attention.gdn_chunkwise" (Module Contents): same arguments, same
shapes, state_pool updated in place, output returned in v's dtype.
``gdn_decode_step`` advances the same pooled states by one token per sequence.
"""

from __future__ import annotations

from typing import NamedTuple

import torch

from . import _lib
from ._lib import GdnError

__all__ = ["gdn_extend_chunkwise", "gdn_decode_step", "gdn_chunkwise_backward", "GdnGrads", "GatedDeltaNetChunkwise",
           "gdn_workspace_size",
           "gdn_backward_workspace_size", "gdn_get_device_status", "GdnError", "library_path", "version"]

_ws_cache: dict = {}
_status_cache: dict = {}


def library_path() -> str:
    return _lib.lib_path()


def version() -> int:
    return int(_lib.load().gdn_version())


def gdn_workspace_size(total_tokens: int, batch: int, H: int, HV: int, K: int, V: int, chunk_size: int) -> int:
    return int(_lib.load().gdn_workspace_size(total_tokens, batch, H, HV, K, V, chunk_size))


def _workspace(device: torch.device, stream: torch.cuda.Stream, nbytes: int) -> torch.Tensor:
    """The cached workspace of (device, stream).

    One buffer per stream: calls on one stream are ordered, so they may share it, while calls
    on two streams of a device run concurrently and must not. The buffer is allocated on the
    call's stream, so when it is replaced by a larger one, the caching allocator reuses the old
    memory only in that stream's order, after the calls already enqueued there.
    """
    key = (device.index, stream.cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        with torch.cuda.stream(stream):
            buf = torch.empty(max(nbytes, 256) + 256, dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def _aligned_ptr(buf: torch.Tensor) -> int:
    p = buf.data_ptr()
    return (p + 255) & ~255


def _req(t: torch.Tensor, name: str, dtype, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def gdn_extend_chunkwise(q, k, v, a, b, A_log, dt_bias, state_pool, cache_indices, cu_seqlens,
                         chunk_size: int = 64, *, scale: float = 1.0, out: torch.Tensor = None,
                         workspace: torch.Tensor = None, check: bool = False, stream=None) -> torch.Tensor:
    """Chunkwise GDN prefill; returns ``out [total_tokens, HV, V]`` in v's dtype.

    q, k ``[T, H, K]``, v ``[T, HV, V]`` bf16 or fp16 (one dtype) on one CUDA device; a, b ``[T, HV]``,
    A_log, dt_bias ``[HV]`` fp32; state_pool ``[pool, HV, V, K]`` fp32 (updated in
    place); cache_indices ``[B]`` and cu_seqlens ``[B+1]`` int64 on the same device.
    ``check=True`` waits for the device and raises on a device-detected error
    (bad cache index or cu_seqlens).
    """
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("gdn_extend_chunkwise runs on a CUDA device; move the inputs there first")
    act = (torch.bfloat16, torch.float16)
    _req(q, "q", act, dev)
    _req(k, "k", q.dtype, dev)
    _req(v, "v", q.dtype, dev)
    for name, t in (("a", a), ("b", b), ("A_log", A_log), ("dt_bias", dt_bias), ("state_pool", state_pool)):
        _req(t, name, torch.float32, dev)
    _req(cache_indices, "cache_indices", torch.int64, dev)
    _req(cu_seqlens, "cu_seqlens", torch.int64, dev)
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or v.shape[0] != q.shape[0]:
        raise ValueError(f"bad q/k/v shapes {tuple(q.shape)} {tuple(k.shape)} {tuple(v.shape)}")
    T, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    if a.shape != (T, HV) or b.shape != (T, HV) or A_log.shape != (HV,) or dt_bias.shape != (HV,):
        raise ValueError("a, b must be [T, HV] and A_log, dt_bias [HV]")
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (HV, V, K):
        raise ValueError(f"state_pool must be [pool, {HV}, {V}, {K}], got {tuple(state_pool.shape)}")
    B = cache_indices.shape[0]
    if cu_seqlens.shape != (B + 1,):
        raise ValueError("cu_seqlens must have batch + 1 entries")
    if out is None:
        out = torch.empty((T, HV, V), dtype=v.dtype, device=dev)
    else:
        _req(out, "out", v.dtype, dev)
        if tuple(out.shape) != (T, HV, V):
            raise ValueError("out must be [T, HV, V]")
    L = _lib.load()
    need = int(L.gdn_workspace_size(T, B, H, HV, K, V, chunk_size))
    if need == 0:
        raise GdnError(2, f"unsupported sizes (K={K}, V={V}, chunk_size={chunk_size}, H={H}, HV={HV})")
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    elif not hasattr(stream, "cuda_stream"):
        stream = torch.cuda.ExternalStream(int(stream), device=dev)
    sp = stream.cuda_stream
    if workspace is None:
        ws = _workspace(dev, stream, need)
        ws_ptr, ws_bytes = _aligned_ptr(ws), ws.numel() - (_aligned_ptr(ws) - ws.data_ptr())
    else:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    dtype_code = _lib.GDN_BF16 if q.dtype == torch.bfloat16 else _lib.GDN_FP16
    st = L.gdn_extend_chunkwise(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), dtype_code,
        a.data_ptr(), b.data_ptr(), A_log.data_ptr(), dt_bias.data_ptr(),
        state_pool.data_ptr(), state_pool.shape[0], cache_indices.data_ptr(), cu_seqlens.data_ptr(), B,
        out.data_ptr(), T, H, HV, K, V, int(chunk_size), float(scale), ws_ptr, ws_bytes, sp)
    _lib.check(st, "gdn_extend_chunkwise")
    if check:
        _lib.check(L.gdn_get_device_status(ws_ptr, sp), "gdn_extend_chunkwise (device)")
    return out


class GdnGrads(NamedTuple):
    """Gradients returned by :func:`gdn_chunkwise_backward` (all fp32)."""
    dq: torch.Tensor            # [T, H, K]
    dk: torch.Tensor            # [T, H, K]
    dv: torch.Tensor            # [T, HV, V]
    da: torch.Tensor            # [T, HV]
    db: torch.Tensor            # [T, HV]
    dA_log: torch.Tensor        # [HV]
    ddt_bias: torch.Tensor      # [HV]
    d_state_pool: torch.Tensor  # [pool, HV, V, K]: zero except at the batch's slots


def gdn_backward_workspace_size(total_tokens: int, batch: int, H: int, HV: int, K: int, V: int,
                                chunk_size: int) -> int:
    return int(_lib.load().gdn_backward_workspace_size(total_tokens, batch, H, HV, K, V, chunk_size))


def gdn_chunkwise_backward(q, k, v, a, b, A_log, dt_bias, state_pool, cache_indices, cu_seqlens, d_out,
                           d_state=None, chunk_size: int = 64, *, scale: float = 1.0, check: bool = False,
                           stream=None, workspace: torch.Tensor = None,
                           d_state_pool: torch.Tensor = None, grads: GdnGrads = None) -> GdnGrads:
    """Gradients of :func:`gdn_extend_chunkwise` for ``L = <d_out, out> + <d_state, final states>``.

    Same inputs as the forward call, except that ``state_pool`` holds the INITIAL states (the pool
    as the forward found it) and is only read. ``d_out [T, HV, V]`` has v's dtype; ``d_state``
    (optional, fp32, shaped like the pool) is the gradient of the final states at the batch's
    slots. Returns :class:`GdnGrads`. Its ``d_state_pool`` is a new zero tensor written at the
    batch's slots, or the given ``d_state_pool``, written at those slots only; that may be
    ``d_state`` itself, for a caller that carries the state gradient back through earlier calls.
    ``check=True`` waits and raises on a device-detected error (bad cache index or cu_seqlens).
    ``grads``: a :class:`GdnGrads` of the right shapes to write into instead of new tensors (its
    ``d_state_pool`` is then written at the batch's slots only).
    """
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("gdn_chunkwise_backward runs on a CUDA device; move the inputs there first")
    _req(q, "q", (torch.bfloat16, torch.float16), dev)
    _req(k, "k", q.dtype, dev)
    _req(v, "v", q.dtype, dev)
    _req(d_out, "d_out", q.dtype, dev)
    for name, t in (("a", a), ("b", b), ("A_log", A_log), ("dt_bias", dt_bias), ("state_pool", state_pool)):
        _req(t, name, torch.float32, dev)
    _req(cache_indices, "cache_indices", torch.int64, dev)
    _req(cu_seqlens, "cu_seqlens", torch.int64, dev)
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or v.shape[0] != q.shape[0] or d_out.shape != v.shape:
        raise ValueError(f"bad q/k/v/d_out shapes {tuple(q.shape)} {tuple(k.shape)} {tuple(v.shape)} "
                         f"{tuple(d_out.shape)}")
    T, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    if a.shape != (T, HV) or b.shape != (T, HV) or A_log.shape != (HV,) or dt_bias.shape != (HV,):
        raise ValueError("a, b must be [T, HV] and A_log, dt_bias [HV]")
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (HV, V, K):
        raise ValueError(f"state_pool must be [pool, {HV}, {V}, {K}], got {tuple(state_pool.shape)}")
    if d_state is not None:
        _req(d_state, "d_state", torch.float32, dev)
        if d_state.shape != state_pool.shape:
            raise ValueError("d_state must have the shape of state_pool")
    if d_state_pool is not None:
        _req(d_state_pool, "d_state_pool", torch.float32, dev)
        if d_state_pool.shape != state_pool.shape:
            raise ValueError("d_state_pool must have the shape of state_pool")
    B = cache_indices.shape[0]
    if cu_seqlens.shape != (B + 1,):
        raise ValueError("cu_seqlens must have batch + 1 entries")
    L = _lib.load()
    need = int(L.gdn_backward_workspace_size(T, B, H, HV, K, V, chunk_size))
    if need == 0:
        raise GdnError(2, f"unsupported sizes for the backward (K={K}, V={V}, chunk_size={chunk_size}, H={H}, HV={HV})")
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    elif not hasattr(stream, "cuda_stream"):
        stream = torch.cuda.ExternalStream(int(stream), device=dev)
    sp = stream.cuda_stream
    if grads is not None:
        shapes = ((T, H, K), (T, H, K), (T, HV, V), (T, HV), (T, HV), (HV,), (HV,), tuple(state_pool.shape))
        for name, t, shp in zip(GdnGrads._fields, grads, shapes):
            _req(t, name, torch.float32, dev)
            if tuple(t.shape) != shp:
                raise ValueError(f"grads.{name} must have shape {shp}")
        if d_state_pool is not None and d_state_pool.data_ptr() != grads.d_state_pool.data_ptr():
            raise ValueError("give the state gradient's buffer once: as d_state_pool or in grads")
    with torch.cuda.stream(stream):
        f32 = dict(dtype=torch.float32, device=dev)
        g = grads if grads is not None else GdnGrads(torch.empty((T, H, K), **f32), torch.empty((T, H, K), **f32), torch.empty((T, HV, V), **f32),
                     torch.empty((T, HV), **f32), torch.empty((T, HV), **f32), torch.empty((HV,), **f32),
                     torch.empty((HV,), **f32),
                     d_state_pool if d_state_pool is not None else torch.zeros_like(state_pool))
        if workspace is None:
            ws = torch.empty(need + 256, dtype=torch.uint8, device=dev)
            ws_ptr = _aligned_ptr(ws)
            ws_bytes = ws.numel() - (ws_ptr - ws.data_ptr())
        else:
            ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    dtype_code = _lib.GDN_BF16 if q.dtype == torch.bfloat16 else _lib.GDN_FP16
    st = L.gdn_chunkwise_backward(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), dtype_code,
        a.data_ptr(), b.data_ptr(), A_log.data_ptr(), dt_bias.data_ptr(),
        state_pool.data_ptr(), state_pool.shape[0], cache_indices.data_ptr(), cu_seqlens.data_ptr(), B,
        d_out.data_ptr(), d_state.data_ptr() if d_state is not None else None,
        g.dq.data_ptr(), g.dk.data_ptr(), g.dv.data_ptr(), g.da.data_ptr(), g.db.data_ptr(),
        g.dA_log.data_ptr(), g.ddt_bias.data_ptr(), g.d_state_pool.data_ptr(),
        T, H, HV, K, V, int(chunk_size), float(scale), ws_ptr, ws_bytes, sp)
    _lib.check(st, "gdn_chunkwise_backward")
    if check:
        _lib.check(L.gdn_get_device_status(ws_ptr, sp), "gdn_chunkwise_backward (device)")
    return g


class GatedDeltaNetChunkwise(torch.autograd.Function):
    """The chunkwise prefill as an autograd function: forward through gdn_extend_chunkwise, backward
    through gdn_chunkwise_backward.

    ``apply(q, k, v, a, b, A_log, dt_bias, initial_state, cu_seqlens, chunk_size=64, scale=1.0)`` with
    ``initial_state [B, HV, V, K]`` fp32 (one state per sequence) returns ``(out [T, HV, V],
    final_state [B, HV, V, K])``; gradients flow to q, k, v, a, b, A_log, dt_bias and initial_state
    (q, k, v get their gradients in their own dtype, the rest in fp32).
    """

    @staticmethod
    def forward(ctx, q, k, v, a, b, A_log, dt_bias, initial_state, cu_seqlens, chunk_size=64, scale=1.0):
        B = initial_state.shape[0]
        idx = torch.arange(B, dtype=torch.int64, device=q.device)
        pool = initial_state.detach().clone().contiguous()
        out = gdn_extend_chunkwise(q, k, v, a, b, A_log, dt_bias, pool, idx, cu_seqlens, chunk_size, scale=scale)
        ctx.save_for_backward(q, k, v, a, b, A_log, dt_bias, initial_state, cu_seqlens, idx)
        ctx.chunk_size, ctx.scale = chunk_size, scale
        return out, pool

    @staticmethod
    def backward(ctx, d_out, d_final):
        q, k, v, a, b, A_log, dt_bias, initial_state, cu_seqlens, idx = ctx.saved_tensors
        if d_out is None:
            d_out = torch.zeros(v.shape, dtype=v.dtype, device=v.device)
        d_state = None if d_final is None else d_final.float().contiguous()
        g = gdn_chunkwise_backward(q, k, v, a, b, A_log, dt_bias, initial_state.detach().contiguous(), idx,
                                   cu_seqlens, d_out.to(v.dtype).contiguous(), d_state, ctx.chunk_size,
                                   scale=ctx.scale)
        return (g.dq.to(q.dtype), g.dk.to(k.dtype), g.dv.to(v.dtype), g.da, g.db, g.dA_log, g.ddt_bias,
                g.d_state_pool, None, None, None)


def gdn_decode_step(q, k, v, a, b, A_log, dt_bias, state_pool, cache_indices, *, scale: float = 1.0,
                    out: torch.Tensor = None, check: bool = False, stream=None,
                    status: torch.Tensor = None) -> torch.Tensor:
    """One token per sequence against the state pool; returns ``out [B, HV, V]`` in v's dtype.

    The one-token case of :func:`gdn_extend_chunkwise` (``cu_seqlens = 0, 1, ..., B``), run by a
    dedicated kernel: q, k ``[B, H, K]``, v ``[B, HV, V]`` bf16 or fp16; a, b ``[B, HV]``, A_log,
    dt_bias ``[HV]`` fp32; state_pool ``[pool, HV, V, K]`` fp32 (updated in place); cache_indices
    ``[B]`` int64. ``check=True`` waits and raises on a bad or repeated cache index.
    ``status``: an int32 device tensor for the step's status word; by default one cached word
    per device, which steps issued concurrently on different streams would share.
    """
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("gdn_decode_step runs on a CUDA device; move the inputs there first")
    _req(q, "q", (torch.bfloat16, torch.float16), dev)
    _req(k, "k", q.dtype, dev)
    _req(v, "v", q.dtype, dev)
    for name, t in (("a", a), ("b", b), ("A_log", A_log), ("dt_bias", dt_bias), ("state_pool", state_pool)):
        _req(t, name, torch.float32, dev)
    _req(cache_indices, "cache_indices", torch.int64, dev)
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or v.shape[0] != q.shape[0]:
        raise ValueError(f"bad q/k/v shapes {tuple(q.shape)} {tuple(k.shape)} {tuple(v.shape)}")
    B, H, K = q.shape
    HV, V = v.shape[1], v.shape[2]
    if a.shape != (B, HV) or b.shape != (B, HV) or A_log.shape != (HV,) or dt_bias.shape != (HV,):
        raise ValueError("a, b must be [B, HV] and A_log, dt_bias [HV]")
    if state_pool.dim() != 4 or tuple(state_pool.shape[1:]) != (HV, V, K):
        raise ValueError(f"state_pool must be [pool, {HV}, {V}, {K}], got {tuple(state_pool.shape)}")
    if cache_indices.shape != (B,):
        raise ValueError("cache_indices must have one entry per sequence")
    if out is None:
        out = torch.empty((B, HV, V), dtype=v.dtype, device=dev)
    else:
        _req(out, "out", v.dtype, dev)
        if tuple(out.shape) != (B, HV, V):
            raise ValueError("out must be [B, HV, V]")
    if status is None:
        status = _status_cache.get(dev.index)
        if status is None:
            status = torch.zeros(64, dtype=torch.int32, device=dev)
            _status_cache[dev.index] = status
    else:
        _req(status, "status", torch.int32, dev)
        if status.numel() < 1:
            raise ValueError("status must hold at least one int32")
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    L = _lib.load()
    dtype_code = _lib.GDN_BF16 if q.dtype == torch.bfloat16 else _lib.GDN_FP16
    st = L.gdn_decode_step(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), dtype_code,
        a.data_ptr(), b.data_ptr(), A_log.data_ptr(), dt_bias.data_ptr(),
        state_pool.data_ptr(), state_pool.shape[0], cache_indices.data_ptr(), B, out.data_ptr(),
        H, HV, K, V, float(scale), status.data_ptr(), sp)
    _lib.check(st, "gdn_decode_step")
    if check:
        _lib.check(L.gdn_get_device_status(status.data_ptr(), sp), "gdn_decode_step (device)")
    return out


def gdn_get_device_status(device=None, stream=None) -> int:
    """Status recorded by the last call on (``device``, ``stream``) that used the cached workspace."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else torch.device(device).index)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    ws = _ws_cache.get((dev.index, stream.cuda_stream))
    if ws is None:
        return 0
    return int(_lib.load().gdn_get_device_status(_aligned_ptr(ws), stream.cuda_stream))


class KernelProfile:
    """Per-kernel device time of the library's launches between start() and stop().

    Each kernel is bracketed by CUDA events on the stream it is launched on.
    """

    def __init__(self, max_launches: int = 100000):
        self.max_launches = max_launches
        self.result = {}

    def start(self):
        _lib.check(_lib.load().gdn_profile_start(self.max_launches), "gdn_profile_start")
        return self

    def stop(self) -> dict:
        import ctypes
        L = _lib.load()
        n = 16
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int64 * n)()
        k = L.gdn_profile_stop(ms, cnt, n)
        if k < 0:
            raise GdnError(6, "gdn_profile_stop failed")
        self.result = {L.gdn_kernel_name(i).decode(): (ms[i], cnt[i]) for i in range(k)}
        return self.result


def launch_count() -> int:
    """Kernels launched by the library in this process so far."""
    return int(_lib.load().gdn_launch_count())
