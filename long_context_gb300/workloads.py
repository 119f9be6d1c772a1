"""Seeded synthetic inputs for the CP ring-attention hot path.

This module only draws inputs.  It holds none of the method's arithmetic, and
both the CUDA path's tests and the CPU oracle's tests are fed from it, so that
they see the same bytes.

Recipe (shared by tests and the benchmark):

* sample lengths come from ``numpy.random.default_rng(seed)``;
* Q, K and V come from a CPU ``torch.Generator().manual_seed(seed)``, drawn in
  that order as float32 standard normals, multiplied by ``std`` and rounded to
  bfloat16 (round to nearest even); for the largest inputs the same recipe
  runs on a seeded CUDA generator (``qkv_device``) and the rows the oracle
  needs are copied back, so both sides still see the same bytes;
* merge partials come from a CPU ``torch.Generator().manual_seed(seed)``:
  O_step ~ N(0, 1), then m_step ~ U[-5, 5], then l_step ~ U[1, 1024], float32.

Workloads (shapes of the dynamic-CP and ring-attention pages):

* ``tiny``       -- one causal sequence of 1024 tokens at CP=2, H=4, D=64.
* ``packed16k``  -- a THD micro-batch filling a 16,384-token budget with
  lognormal(7.5, 1.0) lengths clipped to [64, 16384]; world 4, per-rank limit
  4096, CP sizes from {1, 2, 4}; H=32, D=128.
* ``long128k``   -- one causal sequence of 131,072 tokens at CP=4 (32,768-token
  chunks), H=16, D=128, Q/K/V ~ N(0, 0.5^2).
* ``merge8``     -- CP=8 partials for T=32,768 tokens, H=32, D=128.
* ``sweep256``   -- 256 lengths uniform in [256, 32768], world 8, limit 4096,
  CP sizes from {1, 2, 4, 8}; H=32, D=128.
"""

from __future__ import annotations

import numpy as np
import torch

WORKLOADS = {
    "tiny": dict(lengths=[1024], cp=2, H=4, D=64, std=1.0, causal=True),
    "packed16k": dict(budget=16384, world=4, limit=4096, max_cp=4, H=32, D=128,
                      std=1.0, causal=True),
    "long128k": dict(lengths=[131072], cp=4, H=16, D=128, std=0.5, causal=True),
    "merge8": dict(S=8, T=32768, H=32, D=128),
    "sweep256": dict(n=256, lo=256, hi=32768, world=8, limit=4096, max_cp=8,
                     H=32, D=128, std=1.0, causal=True),
}


def packed_lengths(seed, budget=16384, mu=7.5, sigma=1.0, lo=64, hi=16384):
    """Lognormal lengths appended until ``budget`` tokens are used.

    Each draw is ``round(lognormal(mu, sigma))`` clipped to ``[lo, hi]``; the
    draw that would overflow the budget is cut to the remainder, so the lengths
    sum to ``budget`` exactly (the last one may fall below ``lo``).
    """
    rng = np.random.default_rng(seed)
    out = []
    used = 0
    while used < budget:
        L = int(np.clip(np.rint(rng.lognormal(mu, sigma)), lo, hi))
        L = min(L, budget - used)
        out.append(L)
        used += L
    return out


def uniform_lengths(seed, n=256, lo=256, hi=32768):
    """``n`` lengths uniform over the integers ``lo..hi`` inclusive."""
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


def cu_seqlens(lengths):
    """Prefix sums ``[0, L0, L0+L1, ...]`` as int32 (the THD boundary array)."""
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    if cu[-1] >= 2**31:
        raise ValueError("packed batch too large for int32 cu_seqlens")
    return cu.astype(np.int32)


def qkv(total_tokens, num_heads, head_dim, seed, std=1.0):
    """Q, K, V as CPU bfloat16 tensors ``[T, H, D]`` (drawn in that order)."""
    g = torch.Generator().manual_seed(int(seed))
    shape = (int(total_tokens), int(num_heads), int(head_dim))
    out = []
    for _ in range(3):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        out.append(x.to(torch.bfloat16))
    return tuple(out)


def qkv_device(total_tokens, num_heads, head_dim, seed, std=1.0, device="cuda"):
    """Q, K, V drawn on the GPU from a seeded CUDA generator (same recipe as
    :func:`qkv`, different stream of numbers); bfloat16 ``[T, H, D]``."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    shape = (int(total_tokens), int(num_heads), int(head_dim))
    out = []
    for _ in range(3):
        x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
        if std != 1.0:
            x.mul_(std)
        out.append(x.to(torch.bfloat16))
    return tuple(out)


def merge_partials(num_steps, total_tokens, num_heads, head_dim, seed):
    """Per-step partials for the merge stress case, float32 CPU tensors.

    ``o [S, T, H, D] ~ N(0, 1)``, ``m [S, T, H] ~ U[-5, 5]``,
    ``l [S, T, H] ~ U[1, 1024]``.
    """
    g = torch.Generator().manual_seed(int(seed))
    S, T, H, D = int(num_steps), int(total_tokens), int(num_heads), int(head_dim)
    o = torch.randn((S, T, H, D), generator=g, dtype=torch.float32)
    m = torch.rand((S, T, H), generator=g, dtype=torch.float32).mul_(10.0).sub_(5.0)
    l = torch.rand((S, T, H), generator=g, dtype=torch.float32).mul_(1023.0).add_(1.0)
    return o, m, l


def to_f64(t):
    """Exact upcast of a torch tensor to a float64 NumPy array."""
    return t.detach().to("cpu", torch.float64).numpy()
