"""GPU parity of cpattn_merge against the oracle's step-by-step fold.

The merge is fp32 throughout, so O / l is held to MERGE_RTOL relative to its
row's largest magnitude (helpers.check_merge_o), l to MERGE_L_RTOL relative,
and m exactly up to fp32 rounding of the maximum."""

import numpy as np
import pytest
import torch

from helpers import MERGE_L_RTOL, check_merge_o
from long_context_gb300 import workloads
from oracle import attention as oa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_gb300 import build as lib_build
    lib_build.build()
    from long_context_gb300 import cpattn
    return cpattn


def _check(cp, o, m, l, rows=None):
    go, gm, gl = cp.merge(o.cuda(), m.cuda(), l.cuda())
    go, gm, gl = (x.cpu().numpy().astype(np.float64) for x in (go, gm, gl))
    S, T, H, D = o.shape
    if rows is None:
        ro, rm, rl = oa.merge_partials(o.numpy(), m.numpy(), l.numpy())
        go_, gm_, gl_ = go, gm, gl
    else:
        t_idx, h_idx = rows
        ro, rm, rl = oa.merge_partials(o[:, t_idx, h_idx].numpy(), m[:, t_idx, h_idx].numpy(),
                                       l[:, t_idx, h_idx].numpy())
        go_, gm_, gl_ = go[t_idx, h_idx], gm[t_idx, h_idx], gl[t_idx, h_idx]
    worst = check_merge_o(go_, ro, "merge S=%d T=%d H=%d D=%d" % (S, T, H, D))
    print("merge S=%d T=%d H=%d D=%d: max |dO| / row max |O| = %.3g" % (S, T, H, D, worst))
    fin = np.isfinite(rm)
    assert np.array_equal(np.isfinite(gm_), fin)
    assert np.max(np.abs(gm_[fin] - rm[fin]), initial=0) <= 1e-6
    assert np.all(gl_[~fin] == 0)
    assert np.max(np.abs(gl_ - rl) / np.maximum(rl, 1e-30) * (rl > 0), initial=0) <= MERGE_L_RTOL
    return go, gm, gl


@pytest.mark.parametrize("S,T,H,D", [(1, 37, 3, 128), (3, 100, 2, 64), (8, 257, 4, 128),
                                     (9, 65, 2, 128), (17, 33, 1, 64)])
def test_merge_small_full_compare(cp, S, T, H, D):
    o, m, l = workloads.merge_partials(S, T, H, D, seed=S * 100 + T)
    # Empty steps (the partial of a step that saw nothing) and empty rows.
    m[0, :5] = float("-inf")
    l[0, :5] = 0.0
    o[0, :5] = 0.0
    m[:, 7] = float("-inf")
    l[:, 7] = 0.0
    o[:, 7] = 0.0
    go, gm, gl = _check(cp, o, m, l)
    assert np.all(go[7] == 0) and np.all(np.isneginf(gm[7])) and np.all(gl[7] == 0)


def test_merge_stress_workload(cp):
    """CP=8 partials for T=32,768 tokens, H=32, D=128 (full size, sampled rows)."""
    w = workloads.WORKLOADS["merge8"]
    o, m, l = workloads.merge_partials(w["S"], w["T"], w["H"], w["D"], seed=0)
    rng = np.random.default_rng(0)
    t_idx = np.concatenate([[0, 1, w["T"] - 1], rng.integers(0, w["T"], 4096)])
    h_idx = np.concatenate([[0, w["H"] - 1, w["H"] - 1], rng.integers(0, w["H"], 4096)])
    go, gm, gl = _check(cp, o, m, l, rows=(t_idx, h_idx))
    # Properties at every row: m = max_s m_s exactly.
    assert np.array_equal(gm.astype(np.float32), m.max(dim=0).values.numpy())
