"""Oracle for the Gated DeltaNet chunkwise prefill: fp64, CPU, plain.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package. The GPU
library (``gated_deltanet_chunkwise_gdn_gb300``) never imports it, and this
package never imports the GPU library: the two share no code.

* :func:`gdn_forward` — O1, the token-by-token recurrence in C (``gdn_recurrence.c``),
  threaded over (sequence, value head) chains.
* :func:`delta_rule` — the same recurrence with alpha, beta and normalised q/k given
  directly (for the hand-chosen pins).
* :mod:`oracle.chunkwise` — O2, numpy restatements of the chunkwise WY algebra.
* :mod:`oracle.backward` — O3, gradients of the recurrence (chain rule, fp64), with the final
  state's incoming gradient as an input.
* :mod:`oracle.chunkwise_grad` — O4, the chunkwise WY forward in fp64 PyTorch differentiated by
  autograd (a second route to O3's gradients, and per-chunk intermediate gradients).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_recurrence.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_gdn.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        vp = ctypes.c_void_p
        lib.oracle_softplus.argtypes = [ctypes.c_double]
        lib.oracle_softplus.restype = ctypes.c_double
        lib.oracle_log_alpha.argtypes = [ctypes.c_double] * 3
        lib.oracle_log_alpha.restype = ctypes.c_double
        lib.oracle_beta.argtypes = [ctypes.c_double]
        lib.oracle_beta.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_fp16_to_double.restype = ctypes.c_double
        lib.oracle_delta_rule.argtypes = [dp, dp, dp, dp, dp, ctypes.c_int64, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_double, dp, dp]
        lib.oracle_delta_rule.restype = ctypes.c_int
        lib.oracle_gdn_forward.argtypes = [
            vp, vp, vp, ctypes.c_int,            # q k v is_fp16
            vp, vp, vp, vp,                      # a b A_log dt_bias
            vp, ctypes.c_int64, vp, vp, ctypes.c_int,  # pool pool_size idx cu batch
            ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, vp, vp, ctypes.c_int, vp, vp, ctypes.c_int]
        lib.oracle_gdn_forward.restype = ctypes.c_int
        _lib = lib
        return lib


def softplus(x: float) -> float:
    return _load().oracle_softplus(float(x))


def log_alpha(a: float, A_log: float, dt_bias: float) -> float:
    return _load().oracle_log_alpha(float(a), float(A_log), float(dt_bias))


def beta(b: float) -> float:
    return _load().oracle_beta(float(b))


def bf16_bits_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits))


def fp16_bits_to_double(bits: int) -> float:
    return _load().oracle_fp16_to_double(int(bits))


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def delta_rule(qn, kn, v, alpha, beta_, S0, scale=1.0):
    """Recurrence with explicit alpha/beta and pre-normalised q/k (fp64).

    qn, kn: [T, K]; v: [T, V]; alpha, beta_: [T]; S0: [V, K]. Returns (out [T, V], S [V, K]).
    """
    qn = np.ascontiguousarray(qn, dtype=np.float64)
    kn = np.ascontiguousarray(kn, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    alpha = np.ascontiguousarray(alpha, dtype=np.float64).reshape(-1)
    beta_ = np.ascontiguousarray(beta_, dtype=np.float64).reshape(-1)
    S = np.array(S0, dtype=np.float64, copy=True, order="C")
    T, K = kn.shape
    V = v.shape[1]
    out = np.zeros((T, V), dtype=np.float64)
    rc = _load().oracle_delta_rule(_dptr(qn), _dptr(kn), _dptr(v), _dptr(alpha), _dptr(beta_),
                                   T, K, V, float(scale), _dptr(S), _dptr(out))
    if rc != 0:
        raise RuntimeError(f"oracle_delta_rule failed: {rc}")
    return out, S


class OracleResult:
    """Outputs of :func:`gdn_forward` for a list of (sequence, value head) chains."""

    def __init__(self, chains, lengths, starts, out, states, threads):
        self.chains = chains        # int32 [n, 2]: (seq, hv)
        self.lengths = lengths      # int64 [n]
        self.starts = starts        # int64 [n]: first output row of each chain in `out`
        self.out = out              # float64 [sum(lengths), V]
        self.states = states        # float64 [n, V, K]
        self.threads = threads

    def chain_output(self, i: int) -> np.ndarray:
        s = int(self.starts[i])
        return self.out[s:s + int(self.lengths[i])]


def _as_u16(x) -> np.ndarray:
    """bf16/fp16 torch tensor or uint16 array -> contiguous uint16 numpy view of the bits."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=np.uint16)


def _as_np(x, dtype) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=dtype)


def gdn_forward(q, k, v, a, b, A_log, dt_bias, state_pool, cache_indices, cu_seqlens,
                scale: float = 1.0, is_fp16: bool = False, chains=None,
                n_threads: int = 0) -> OracleResult:
    """O1: fp64 token recurrence for the given chains (default: every chain).

    q, k: [T, H, K] bf16 (or fp16 with is_fp16) as torch tensors or uint16 bit arrays;
    v: [T, HV, V]; a, b: [T, HV] fp32; A_log, dt_bias: [HV] fp32;
    state_pool: [pool, HV, V, K] fp32 (read only here); cache_indices: [B] int64;
    cu_seqlens: [B+1] int64; chains: optional [n, 2] (seq, hv) pairs.
    """
    qb, kb, vb = _as_u16(q), _as_u16(k), _as_u16(v)
    T, H, K = qb.shape
    HV, V = vb.shape[1], vb.shape[2]
    a_, b_ = _as_np(a, np.float32), _as_np(b, np.float32)
    Al, db = _as_np(A_log, np.float32), _as_np(dt_bias, np.float32)
    pool = _as_np(state_pool, np.float32)
    idx = _as_np(cache_indices, np.int64)
    cu = _as_np(cu_seqlens, np.int64)
    B = idx.shape[0]
    if chains is None:
        ch = np.stack(np.meshgrid(np.arange(B), np.arange(HV), indexing="ij"), -1).reshape(-1, 2)
    else:
        ch = np.asarray(chains).reshape(-1, 2)
    ch = np.ascontiguousarray(ch, dtype=np.int32)
    seq = np.ascontiguousarray(ch[:, 0])
    hv = np.ascontiguousarray(ch[:, 1])
    lengths = (cu[seq.astype(np.int64) + 1] - cu[seq.astype(np.int64)]).astype(np.int64)
    starts = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64) if len(ch) else np.zeros(0, np.int64)
    out = np.zeros((int(lengths.sum()), V), dtype=np.float64)
    states = np.zeros((len(ch), V, K), dtype=np.float64)
    vp = lambda arr: arr.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    rc = _load().oracle_gdn_forward(
        vp(qb), vp(kb), vp(vb), int(bool(is_fp16)), vp(a_), vp(b_), vp(Al), vp(db),
        vp(pool), pool.shape[0], vp(idx), vp(cu), B, T, H, HV, K, V, float(scale),
        vp(seq), vp(hv), len(ch), vp(out), vp(states), int(n_threads))
    if rc < 0:
        raise ValueError(f"oracle_gdn_forward rejected the inputs (code {-rc})")
    return OracleResult(ch, lengths, starts, out, states, rc)
