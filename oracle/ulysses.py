"""Oracle for the Ulysses sequence-parallel layout.  TEST INFRASTRUCTURE ONLY.

"VeRL Backend Parallelism" (USP section; "do not mix the three Ulysses"):
verl's Ulysses sequence parallelism (``ulysses_sequence_parallel_size``) is a
real compute path -- a [dp, sp] mesh whose SP group splits the sequence --
and it is neither Megatron's sequence parallelism nor CP.  No algorithm is
printed; the plainest reading of Ulysses attention: activations are sharded
by sequence, an all-to-all over the SP group before attention gives every
rank the whole sequence for H / P of the heads, attention runs on those heads
locally, and the inverse all-to-all restores sequence sharding.

On one device the all-to-all is a layout transform of the packed [T, H, D]
array: ``to_head_groups`` gives [P, T, H/P, D] (group p = heads
[p H/P, (p+1) H/P)), ``from_head_groups`` inverts it.

Shares no code with the CUDA path and imports nothing from it.
"""

from __future__ import annotations

import numpy as np

from .attention import full_attention


def to_head_groups(x, P):
    """[T, H, ...] -> [P, T, H / P, ...]."""
    x = np.asarray(x)
    T, H = x.shape[0], x.shape[1]
    assert H % P == 0
    return np.ascontiguousarray(
        np.moveaxis(x.reshape((T, P, H // P) + x.shape[2:]), 1, 0))


def from_head_groups(y, P):
    """[P, T, H / P, ...] -> [T, H, ...]."""
    y = np.asarray(y)
    T, Hp = y.shape[1], y.shape[2]
    return np.ascontiguousarray(np.moveaxis(y, 0, 1).reshape((T, P * Hp) + y.shape[3:]))


def ulysses_attention(q, k, v, cu_seqlens, P, scale, causal=True):
    """Attention the Ulysses way: to head groups, attention of every group on
    the whole packed sequence, back to [T, H, D].  Returns ``(O, LSE)``."""
    qg, kg, vg = (to_head_groups(np.asarray(x, dtype=np.float64), P) for x in (q, k, v))
    outs, lses = [], []
    for p in range(P):
        o, l = full_attention(qg[p], kg[p], vg[p], cu_seqlens, scale, causal=causal)
        outs.append(o)
        lses.append(l)
    return from_head_groups(np.stack(outs), P), from_head_groups(np.stack(lses), P)
