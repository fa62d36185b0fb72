"""Seeded synthetic inputs for chunkwise GDN prefill.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic, so both the GPU path and the oracle may consume what it
makes. Every tensor is generated on the CPU with ``torch.Generator`` (the same
bytes then go to the GPU and to the oracle).

Shapes follow the gdn_extend_chunkwise parameter list of the pymllm page
("pymllm.layers.attention.gdn_chunkwise", Parameters):
q, k ``[T, H, K]``, v ``[T, HV, V]`` (bf16), a, b ``[T, HV]`` fp32,
A_log, dt_bias ``[HV]`` fp32, state_pool ``[pool, HV, V, K]`` fp32,
cache_indices ``[B]`` int64, cu_seqlens ``[B+1]`` int64.

Gate distributions: a, b ~ N(mean, 1); A_log = log U[1, 16];
dt_bias = log(expm1(U[1e-3, 0.1])) (so softplus(dt_bias) is U[1e-3, 0.1]).
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import List, Optional, Sequence

import torch

_SLAB = 1 << 24  # elements drawn per randn call (keeps fp32 temporaries small)


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    lengths: Optional[Sequence[int]]  # None: drawn from the generator (varlen)
    H: int
    HV: int
    K: int
    V: int
    chunk_size: int
    pool_size: int
    state_std: float = 0.0            # 0: zero initial states, else N(0, state_std^2)
    index_rule: str = "arange"        # "arange" | "perm_subset" (randperm(pool)[:B])
    varlen_batch: int = 0             # number of sequences when lengths is None
    varlen_max: int = 0               # lengths ~ U{1..varlen_max}
    a_mean: float = 0.0
    b_mean: float = 0.0
    dtype: torch.dtype = torch.bfloat16
    note: str = ""

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five benchmark configurations, in order (seed = position).
CONFIGS: List[Workload] = [
    Workload("tiny", 0, [256], H=2, HV=2, K=64, V=64, chunk_size=64, pool_size=1,
             note="B=1, T=256, H=HV=2, K=V=64, C=64, zero state"),
    Workload("varlen", 1, None, H=16, HV=32, K=128, V=128, chunk_size=64, pool_size=64,
             state_std=0.1, index_rule="perm_subset", varlen_batch=8, varlen_max=4096,
             note="8 sequences, lengths U{1..4096}, H=16, HV=32, K=V=128, C=64, 64-slot pool"),
    Workload("long", 2, [65536], H=16, HV=16, K=128, V=128, chunk_size=64, pool_size=1,
             note="B=1, T=65536, H=HV=16, K=V=128, C=64, zero state"),
    Workload("throughput", 3, [8192] * 32, H=32, HV=32, K=128, V=128, chunk_size=64,
             pool_size=32, state_std=0.1, index_rule="perm_subset",
             note="B=32 x T=8192, H=HV=32, K=V=128, C=64, states N(0, 0.1^2)"),
    Workload("wide", 4, [16384] * 4, H=4, HV=4, K=256, V=256, chunk_size=128, pool_size=4,
             a_mean=-2.0, b_mean=1.0,
             note="B=4 x T=16384, H=HV=4, K=V=256, C=128, a ~ N(-2,1), b ~ N(1,1), zero state"),
]
# Single-token step (decode): one new token for each of 256 sequences against a 512-slot pool,
# the head shape of the varlen configuration. Every sequence has length 1, so cu_seqlens is
# 0, 1, ..., 256 and the same inputs serve the chunkwise call and the oracle.
DECODE = Workload("decode", 5, [1] * 256, H=16, HV=32, K=128, V=128, chunk_size=64, pool_size=512,
                  state_std=0.1, index_rule="perm_subset",
                  note="B=256 sequences x 1 token, H=16, HV=32, K=V=128, 512-slot pool, states N(0, 0.1^2)")
BY_NAME = {w.name: w for w in CONFIGS + [DECODE]}


def _randn_into(out: torch.Tensor, gen: torch.Generator, mean: float = 0.0, std: float = 1.0):
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, _SLAB):
        e = min(n, s + _SLAB)
        x = torch.randn(e - s, generator=gen, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        if mean != 0.0:
            x.add_(mean)
        flat[s:e].copy_(x)
    return out


def _uniform(n: int, lo: float, hi: float, gen: torch.Generator) -> torch.Tensor:
    return torch.rand(n, generator=gen, dtype=torch.float64) * (hi - lo) + lo


def sequence_lengths(w: Workload, gen: Optional[torch.Generator] = None) -> List[int]:
    if w.lengths is not None:
        return [int(x) for x in w.lengths]
    gen = gen if gen is not None else torch.Generator().manual_seed(w.seed)
    return [int(x) for x in torch.randint(1, w.varlen_max + 1, (w.varlen_batch,), generator=gen)]


def make_inputs(w: Workload) -> dict:
    """All inputs of one call, as CPU tensors, drawn in a fixed order from ``w.seed``."""
    gen = torch.Generator().manual_seed(w.seed)
    lengths = sequence_lengths(w, gen)
    B = len(lengths)
    T = sum(lengths)
    cu = torch.zeros(B + 1, dtype=torch.int64)
    if B:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0)
    q = _randn_into(torch.empty(T, w.H, w.K, dtype=w.dtype), gen)
    k = _randn_into(torch.empty(T, w.H, w.K, dtype=w.dtype), gen)
    v = _randn_into(torch.empty(T, w.HV, w.V, dtype=w.dtype), gen)
    a = _randn_into(torch.empty(T, w.HV, dtype=torch.float32), gen, mean=w.a_mean)
    b = _randn_into(torch.empty(T, w.HV, dtype=torch.float32), gen, mean=w.b_mean)
    A_log = torch.log(_uniform(w.HV, 1.0, 16.0, gen)).to(torch.float32)
    dt_bias = torch.log(torch.expm1(_uniform(w.HV, 1e-3, 0.1, gen))).to(torch.float32)
    pool = torch.zeros(w.pool_size, w.HV, w.V, w.K, dtype=torch.float32)
    if w.state_std > 0:
        _randn_into(pool, gen, std=w.state_std)
    if w.index_rule == "perm_subset":
        idx = torch.randperm(w.pool_size, generator=gen)[:B].to(torch.int64)
    else:
        idx = torch.arange(B, dtype=torch.int64)
    return dict(q=q, k=k, v=v, a=a, b=b, A_log=A_log, dt_bias=dt_bias, state_pool=pool,
                cache_indices=idx.contiguous(), cu_seqlens=cu, chunk_size=w.chunk_size)


def custom(name: str, lengths: Sequence[int], H: int, HV: int, K: int, V: int, chunk_size: int,
           seed: int, pool_size: Optional[int] = None, state_std: float = 0.1,
           index_rule: str = "perm_subset", a_mean: float = 0.0, b_mean: float = 0.0,
           dtype: torch.dtype = torch.bfloat16) -> Workload:
    """A parity-test workload of arbitrary shape, same distributions as the configs."""
    return Workload(name, seed, list(lengths), H=H, HV=HV, K=K, V=V, chunk_size=chunk_size,
                    pool_size=pool_size if pool_size is not None else max(1, 2 * len(lengths)),
                    state_std=state_std, index_rule=index_rule, a_mean=a_mean, b_mean=b_mean,
                    dtype=dtype)
