"""Pins of the DCP data-movement oracle (oracle/dcp.py), CPU only."""

import numpy as np

from oracle import attention as oa
from oracle import dcp as od
from oracle import planner as op


def _batch(lengths, H, D, seed):
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    q, k, v = (rng.normal(0.0, 1.0, (T, H, D)) for _ in range(3))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return q, k, v, cu


def test_select_layout_and_round_trip():
    lengths = [5, 0, 3, 9, 1]
    x = np.arange(sum(lengths) * 2).reshape(-1, 2)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    ids = [3, 0, 4]
    y, ycu = od.select(x, cu, ids)
    assert list(ycu) == [0, 9, 14, 15]
    # By hand: sample 3 is rows 8..16, sample 0 rows 0..4, sample 4 row 17.
    want = np.concatenate([x[8:17], x[0:5], x[17:18]])
    assert np.array_equal(y, want)
    out = np.full_like(x, -1)
    od.restore(y, ids, cu, out)
    for b in ids:
        assert np.array_equal(out[cu[b]:cu[b + 1]], x[cu[b]:cu[b + 1]])
    assert (out[cu[2]:cu[3]] == -1).all()        # not selected: untouched
    y0, _ = od.select(x, cu, [])
    assert y0.shape == (0, 2)


def test_micro_batches_partition_the_batch():
    rng = np.random.default_rng(4)
    lengths = [int(x) for x in rng.integers(1, 9000, 40)]
    plan = op.plan(lengths, 8, 4096, 8)
    x = np.arange(sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    seen = []
    out = np.full_like(x, -1)
    for m in range(plan["num_micro_batches"]):
        ids = od.micro_batch_samples(plan, m)
        # planner order: non-increasing length within the micro-batch
        assert all(lengths[a] >= lengths[b] for a, b in zip(ids, ids[1:]))
        seen += ids
        y, _ = od.select(x, cu, ids)
        od.restore(y, ids, cu, out)
    assert sorted(seen) == list(range(len(lengths)))
    assert np.array_equal(out, x)


def test_dcp_forward_equals_full_attention():
    """Splitting into micro-batches and restoring changes nothing: every
    sample's attention is computed whole, with or without the ring."""
    lengths = [37, 5, 120, 64, 1, 90]
    q, k, v, cu = _batch(lengths, 2, 8, seed=9)
    plan = op.plan(lengths, 4, 48, 4)
    assert plan["num_micro_batches"] > 1
    ref_o, ref_l = oa.full_attention(q, k, v, cu, 0.3)
    for ring in (False, True):
        o, l = od.dcp_forward(q, k, v, cu, plan, 0.3, ring=ring)
        assert np.max(np.abs(o - ref_o)) < 1e-12 and np.max(np.abs(l - ref_l)) < 1e-12
