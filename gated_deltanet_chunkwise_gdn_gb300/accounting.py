"""Work and traffic accounting for one gdn_extend_chunkwise call.

Counting models used by the benchmark's roofline figures (TFLOP/s and GB/s are
algorithmic: what the method needs, not what a kernel happens to execute).
"""

from __future__ import annotations

from typing import Optional, Sequence


def flop_count(lengths: Sequence[int], H: int, HV: int, K: int, V: int, C: int) -> float:
    """Algorithmic FLOPs of one call (counting model stated in the design notes).

    Per chunk of true length L and value head: Gram products shared by the HV/H
    value heads of a q/k head, (H/HV) * (L(L-1) K + L(L+1) K); the triangular
    inverse L^3/3; W<- and U~: L(L+1)(K+V); intra output L(L+1) V; the three
    state products 6 L K V.
    """
    total = 0.0
    for n in lengths:
        for s in range(0, n, C):
            L = min(C, n - s)
            per_hv = ((H / HV) * (L * (L - 1) * K + L * (L + 1) * K) + L ** 3 / 3.0
                      + L * (L + 1) * (K + V) + L * (L + 1) * V + 6.0 * L * K * V)
            total += HV * per_hv
    return total


def min_hbm_bytes(lengths: Sequence[int], H: int, HV: int, K: int, V: int,
                  elem_bytes: int = 2, n_touched_states: Optional[int] = None) -> float:
    """Bytes a call must move at least: q, k, v, a, b read once, o written once,
    and each touched state read and written once (fp32)."""
    T = sum(lengths)
    B = len(lengths) if n_touched_states is None else n_touched_states
    return (T * (2 * H * K * elem_bytes + HV * V * elem_bytes * 2 + HV * 8)
            + B * HV * V * K * 4 * 2)
