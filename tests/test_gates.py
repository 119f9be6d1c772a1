"""The parity gates themselves have teeth (CPU, no GPU needed).

The merge gate (helpers.check_merge_o) must tell an fp32 merge from one whose
O path was rounded to bf16 anywhere: the oracle's own merge, rounded to fp32,
passes; the same result rounded to bf16 fails.  With O_step ~ N(0, 1) and
l_step in [1, 1024] (the CP=8 merge workload's distributions) the median row's
largest |O / l| is about 4e-3, where a plain 1e-5 absolute bound would accept
the bf16 result -- which is why the gate is relative to each row's largest
magnitude.
"""

import numpy as np
import pytest
import torch

from helpers import check_merge_o, MERGE_RTOL
from long_context_gb300 import workloads
from oracle import attention as oa


def _merged(seed):
    o, m, l = workloads.merge_partials(8, 64, 4, 128, seed=seed)
    ro, rm, rl = oa.merge_partials(o.numpy(), m.numpy(), l.numpy())
    return ro


@pytest.mark.parametrize("seed", [0, 1])
def test_merge_gate_accepts_fp32_rounding(seed):
    ro = _merged(seed)
    got = ro.astype(np.float32).astype(np.float64)
    assert check_merge_o(got, ro) <= MERGE_RTOL


@pytest.mark.parametrize("seed", [0, 1])
def test_merge_gate_rejects_bf16_rounding(seed):
    ro = _merged(seed)
    got = torch.from_numpy(ro).to(torch.bfloat16).to(torch.float64).numpy()
    with pytest.raises(AssertionError):
        check_merge_o(got, ro)
    # On the typical rows (max |O / l| below 2.5e-3) an absolute 1e-5 bound
    # would not have noticed the bf16 rounding; the relative gate does.
    typical = np.max(np.abs(ro), axis=-1) < 2.5e-3
    assert typical.sum() >= 16
    assert np.max(np.abs(got[typical] - ro[typical])) < 1e-5
    with pytest.raises(AssertionError):
        check_merge_o(got[typical], ro[typical])


def test_merge_gate_rejects_nonzero_empty_rows():
    ro = _merged(2)
    ro[3] = 0.0
    got = ro.copy()
    got[3, 0, 5] = 1e-30
    with pytest.raises(AssertionError):
        check_merge_o(got, ro)
