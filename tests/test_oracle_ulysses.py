"""Pins of the Ulysses layout oracle (oracle/ulysses.py), CPU only."""

import numpy as np

from oracle import attention as oa
from oracle import ulysses as ou


def test_layout_by_hand_and_round_trip():
    T, H, D, P = 3, 4, 2, 2
    x = np.arange(T * H * D).reshape(T, H, D)
    y = ou.to_head_groups(x, P)
    assert y.shape == (P, T, H // P, D)
    # Group 1, token 2, local head 0 is global head 2 of token 2.
    assert np.array_equal(y[1, 2, 0], x[2, 2])
    assert np.array_equal(y[0, 1, 1], x[1, 1])
    assert np.array_equal(ou.from_head_groups(y, P), x)
    lse = np.arange(T * H).reshape(T, H)
    assert np.array_equal(ou.from_head_groups(ou.to_head_groups(lse, 4), 4), lse)


def test_ulysses_attention_equals_full_attention():
    rng = np.random.default_rng(3)
    lengths, H, D = [9, 30, 1], 4, 8
    T = sum(lengths)
    q, k, v = (rng.normal(size=(T, H, D)) for _ in range(3))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    ref_o, ref_l = oa.full_attention(q, k, v, cu, 0.4)
    for P in (1, 2, 4):
        o, l = ou.ulysses_attention(q, k, v, cu, P, 0.4)
        assert np.max(np.abs(o - ref_o)) < 1e-13 and np.max(np.abs(l - ref_l)) < 1e-13
