"""Oracle dynamic-CP planner: plain Python.  TEST INFRASTRUCTURE ONLY.

[DCP] lets the engine pick a CP size per packed micro-batch with a
sequence-length-aware scheduler; every DPxCP rank sees the same mini-batch and
takes its own samples, and the per-rank packing limit is
``max_seqlen_per_dp_cp_rank`` (the static budget divided by the static CP size,
e.g. 16384 / 4 = 4096).  The DPxCP world size must be even and at least two;
CP groups are power-of-two subgroups plus, when needed, the full DPxCP group.
[MCore] section 4 packs dynamic batches by ``max_token_len_per_gpu * sp_size``,
i.e. W rank slots of ``limit`` tokens each.  The scheduler's internal algorithm
is not given on any page; this module is the plainest reading of those rules:

1. CP size of a sample of length L: the smallest candidate c with
   ``ceil(L / c) <= limit``.  Candidates are the powers of two below
   ``max_cp`` and ``max_cp`` itself (which may be the full, non-power-of-two
   DPxCP group when ``max_cp == world``).  No candidate fits -> infeasible.
2. Samples are taken longest first; equal lengths keep their original order.
3. A micro-batch has W rank slots of capacity ``limit``.  A sample with CP c
   occupies an aligned group of ranks ``[g*c, (g+1)*c)`` with
   ``g in 0 .. W//c - 1`` and adds ``ceil(L / c)`` tokens to each of them.
4. First fit: the first existing micro-batch (in creation order) and within it
   the first group where every rank stays within the limit; otherwise a new
   micro-batch is opened and the sample goes to its group 0.
"""

from __future__ import annotations

import itertools


class PlanInfeasible(ValueError):
    """A sample does not fit even at the largest allowed CP size."""


def _ceil_div(a, b):
    return -(-a // b)


def is_pow2(x):
    return x >= 1 and (x & (x - 1)) == 0


def check_args(world, limit, max_cp):
    """Argument rules taken from [DCP] and [MCore] section 1.

    The DPxCP world size is even and >= 2; the per-rank limit is required
    (positive); ``max_cp`` is a power of two no larger than the world size, or
    the world size itself (the full DPxCP group).
    """
    if world < 2 or world % 2 != 0:
        raise ValueError("DPxCP world size must be an even integer >= 2")
    if limit < 1:
        raise ValueError("max_seqlen_per_dp_cp_rank must be positive")
    if max_cp < 1 or max_cp > world or not (is_pow2(max_cp) or max_cp == world):
        raise ValueError("max_cp must be a power of two <= world, or world")


def cp_candidates(max_cp):
    """Allowed CP sizes in increasing order: powers of two below max_cp, then max_cp."""
    out = []
    c = 1
    while c < max_cp:
        out.append(c)
        c *= 2
    out.append(max_cp)
    return out


def cp_size_for_length(L, limit, max_cp):
    """Rule 1: smallest allowed c with ceil(L / c) <= limit, else None."""
    for c in cp_candidates(max_cp):
        if _ceil_div(L, c) <= limit:
            return c
    return None


def plan(seqlens, world, limit, max_cp):
    """Plan a mini-batch: rules 1-4 of the module docstring.

    Returns a dict with ``cp_size``, ``micro_batch``, ``first_rank`` (all
    indexed by original sample index), ``order`` (the processing order),
    ``num_micro_batches`` and ``rank_load`` (one list of W loads per
    micro-batch).
    """
    seqlens = [int(x) for x in seqlens]
    check_args(world, limit, max_cp)
    n = len(seqlens)
    if any(L < 0 for L in seqlens):
        raise ValueError("negative sequence length")
    cp = []
    for L in seqlens:
        c = cp_size_for_length(L, limit, max_cp)
        if c is None:
            raise PlanInfeasible("sample of length %d exceeds max_cp * limit" % L)
        cp.append(c)
    order = sorted(range(n), key=lambda b: (-seqlens[b], b))
    loads = []
    micro_batch = [0] * n
    first_rank = [0] * n
    for b in order:
        c = cp[b]
        need = _ceil_div(seqlens[b], c)
        placed = False
        for mb, load in enumerate(loads):
            for g in range(world // c):
                ranks = range(g * c, (g + 1) * c)
                if all(load[r] + need <= limit for r in ranks):
                    for r in ranks:
                        load[r] += need
                    micro_batch[b] = mb
                    first_rank[b] = g * c
                    placed = True
                    break
            if placed:
                break
        if not placed:
            load = [0] * world
            for r in range(c):
                load[r] += need
            loads.append(load)
            micro_batch[b] = len(loads) - 1
            first_rank[b] = 0
    return {
        "cp_size": cp,
        "micro_batch": micro_batch,
        "first_rank": first_rank,
        "order": order,
        "num_micro_batches": len(loads),
        "rank_load": loads,
    }


# ---------------------------------------------------------------------------
# Brute-force checkers (used by the oracle's own tests).
# ---------------------------------------------------------------------------

def brute_cp_size(L, limit, max_cp):
    """Rule 1 by enumeration: every allowed c that fits, take the minimum."""
    fits = [c for c in range(1, max_cp + 1)
            if (is_pow2(c) or c == max_cp) and c <= max_cp and L <= c * limit]
    return min(fits) if fits else None


def check_plan_invariants(seqlens, world, limit, result):
    """Structural rules every valid plan obeys; raises AssertionError if not."""
    n = len(seqlens)
    cp = result["cp_size"]
    mbs = result["micro_batch"]
    fr = result["first_rank"]
    nmb = result["num_micro_batches"]
    assert sorted(result["order"]) == list(range(n))
    loads = [[0] * world for _ in range(nmb)]
    for b in range(n):
        c = cp[b]
        assert 0 <= mbs[b] < nmb
        assert fr[b] % c == 0 and fr[b] + c <= world
        need = _ceil_div(seqlens[b], c)
        for r in range(fr[b], fr[b] + c):
            loads[mbs[b]][r] += need
    for load in loads:
        assert all(x <= limit for x in load)
    assert loads == result["rank_load"]
    return loads


def brute_min_micro_batches(seqlens, world, limit, cp):
    """Fewest micro-batches over every assignment of the given CP sizes.

    Exhaustive search, for instances of at most about eight samples.  Used only
    to report how far first fit is from optimal; first fit is not required to
    be optimal.
    """
    n = len(seqlens)
    need = [_ceil_div(seqlens[b], cp[b]) for b in range(n)]
    for k in range(1, n + 1):
        choices = []
        for b in range(n):
            choices.append([(mb, g) for mb in range(k) for g in range(world // cp[b])])
        for combo in itertools.product(*choices):
            loads = [[0] * world for _ in range(k)]
            ok = True
            for b, (mb, g) in enumerate(combo):
                for r in range(g * cp[b], (g + 1) * cp[b]):
                    loads[mb][r] += need[b]
                    if loads[mb][r] > limit:
                        ok = False
                        break
                if not ok:
                    break
            if ok:
                return k
    return n if n else 0
