"""Pins for the oracle's dynamic-CP planner (CPU only)."""

import json
import os

import numpy as np
import pytest

from oracle import attention as oa
from oracle import planner as op

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    return json.load(open(os.path.join(GOLDEN, "dcp_plans.json")))


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: c["name"])
def test_golden_plans(case):
    r = op.plan(case["seqlens"], case["world"], case["limit"], case["max_cp"])
    for key in ("cp_size", "micro_batch", "first_rank", "order",
                "num_micro_batches", "rank_load"):
        assert r[key] == case[key], key


def test_page_worked_example_limit():
    # 16,384-token static budget at CP4 -> per-rank limit 4096 (DCP page).
    budget, static_cp = 16384, 4
    limit = budget // static_cp
    assert limit == 4096
    assert op.cp_size_for_length(16384, limit, 4) == 4
    assert op.cp_size_for_length(4096, limit, 4) == 1
    assert op.cp_size_for_length(4097, limit, 4) == 2
    assert op.cp_size_for_length(8193, limit, 4) == 4
    assert op.cp_size_for_length(16385, limit, 4) is None


def test_infeasible():
    for case in _golden()["infeasible"]:
        with pytest.raises(op.PlanInfeasible):
            op.plan(case["seqlens"], case["world"], case["limit"], case["max_cp"])


@pytest.mark.parametrize("limit,max_cp", [(7, 1), (7, 2), (5, 4), (3, 8), (4, 6), (6, 2)])
def test_cp_size_brute_force(limit, max_cp):
    for L in range(0, limit * max_cp + 6):
        assert op.cp_size_for_length(L, limit, max_cp) == op.brute_cp_size(L, limit, max_cp)


def test_argument_rules():
    with pytest.raises(ValueError):
        op.plan([1], 3, 10, 1)        # odd world
    with pytest.raises(ValueError):
        op.plan([1], 0, 10, 1)        # world < 2
    with pytest.raises(ValueError):
        op.plan([1], 4, 0, 1)         # limit missing
    with pytest.raises(ValueError):
        op.plan([1], 4, 10, 3)        # not a power of two and not the world
    with pytest.raises(ValueError):
        op.plan([1], 4, 10, 8)        # larger than the world
    op.plan([1], 6, 10, 6)            # full non-power-of-two group is allowed
    op.plan([], 2, 10, 2)             # empty batch


def test_invariants_random_instances():
    rng = np.random.default_rng(0)
    for trial in range(300):
        world = int(rng.choice([2, 4, 6, 8]))
        cands = [c for c in (1, 2, 4, 8) if c <= world] + [world]
        max_cp = int(rng.choice(cands))
        limit = int(rng.integers(1, 50))
        n = int(rng.integers(0, 30))
        lens = [int(x) for x in rng.integers(0, limit * max_cp + 1, n)]
        r = op.plan(lens, world, limit, max_cp)
        op.check_plan_invariants(lens, world, limit, r)
        assert r["order"] == sorted(range(n), key=lambda b: (-lens[b], b))
        for b in range(n):
            assert r["cp_size"][b] == op.brute_cp_size(lens[b], limit, max_cp)


def test_first_fit_vs_brute_force_minimum():
    """First fit never beats the optimum; the gap is only reported."""
    rng = np.random.default_rng(1)
    gaps = []
    for trial in range(40):
        world, limit, max_cp = 4, 10, 4
        n = int(rng.integers(1, 6))
        lens = [int(x) for x in rng.integers(1, 41, n)]
        r = op.plan(lens, world, limit, max_cp)
        best = op.brute_min_micro_batches(lens, world, limit, r["cp_size"])
        assert r["num_micro_batches"] >= best
        gaps.append(r["num_micro_batches"] - best)
    print("first-fit gap histogram:", np.bincount(gaps))


def test_cp_invariance_dynamic_vs_static():
    """Only the CP assignment changes between static and dynamic CP, so the
    attention outputs agree (DCP comparison method; 1/2/4-rank checklist)."""
    rng = np.random.default_rng(2)
    lens = [3, 17, 9, 30, 1, 12]
    limit, world, max_cp = 8, 4, 4
    r = op.plan(lens, world, limit, max_cp)
    T = sum(lens)
    q = rng.standard_normal((T, 2, 8))
    k = rng.standard_normal((T, 2, 8))
    v = rng.standard_normal((T, 2, 8))
    cu = np.concatenate([[0], np.cumsum(lens)])
    dyn = oa.ring_attention(q, k, v, cu, r["cp_size"], 0.3)
    for c in (1, 2, 4):
        stat = oa.ring_attention(q, k, v, cu, [c] * len(lens), 0.3)
        np.testing.assert_allclose(dyn[0], stat[0], atol=1e-12)
        np.testing.assert_allclose(dyn[1], stat[1], atol=1e-12)
