"""Pins of the backward oracle (oracle/backward.py), CPU only.

The backward is the derivative of the forward's definition.  It is pinned
against things other than its own formulas: central finite differences of the
forward oracle, the chunk-by-chunk ring sum, and identities that follow from
the softmax (each row of P sums to 1, so every row of dS sums to 0).
"""

import numpy as np
import pytest

from oracle import attention as oa
from oracle import backward as ob


def _batch(lengths, H, D, seed, std=1.0):
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    q, k, v, do = (rng.normal(0.0, std, (T, H, D)) for _ in range(4))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return q, k, v, do, cu


@pytest.mark.parametrize("causal", [True, False])
def test_matches_finite_differences_of_the_forward(causal):
    """Loss = sum(dO * O); every gradient entry against a central difference of
    the forward oracle (step 1e-6, float64)."""
    lengths, H, D = [5, 3, 1], 2, 4
    q, k, v, do, cu = _batch(lengths, H, D, seed=1)
    scale = 0.7
    g = ob.full_attention_backward(q, k, v, do, cu, scale, causal=causal)

    def loss(q_, k_, v_):
        o, _ = oa.full_attention(q_, k_, v_, cu, scale, causal=causal)
        return float((o * do).sum())

    eps = 1e-6
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args = {"dq": (xp, k, v), "dk": (q, xp, v), "dv": (q, k, xp)}[name]
            argm = {"dq": (xm, k, v), "dk": (q, xm, v), "dv": (q, k, xm)}[name]
            num[idx] = (loss(*args) - loss(*argm)) / (2 * eps)
        assert np.max(np.abs(num - g[name])) < 1e-7, name


@pytest.mark.parametrize("causal", [True, False])
def test_ring_blocks_sum_to_the_full_backward(causal):
    lengths, H, D = [1, 2, 7, 13, 40, 3], 2, 8
    q, k, v, do, cu = _batch(lengths, H, D, seed=2)
    full = ob.full_attention_backward(q, k, v, do, cu, 0.35, causal=causal)
    for c in (1, 2, 3, 4, 8):
        ring = ob.ring_attention_backward(q, k, v, do, cu, [c] * len(lengths), 0.35,
                                          causal=causal)
        for name in ("dq", "dk", "dv"):
            assert np.max(np.abs(ring[name] - full[name])) < 1e-12, (c, name)
        assert np.max(np.abs(ring["delta"] - full["delta"])) < 1e-12


def test_softmax_identities():
    """Rows of P sum to 1 and rows of dS to 0, so per sample and head
    sum_j dV_j = sum_i dO_i and sum_j dK_j = 0; and D_i = <dO_i, O_i>."""
    lengths, H, D = [9, 30, 4], 3, 8
    q, k, v, do, cu = _batch(lengths, H, D, seed=3)
    for causal in (True, False):
        g = ob.full_attention_backward(q, k, v, do, cu, 0.5, causal=causal)
        for b in range(len(lengths)):
            s0, s1 = cu[b], cu[b + 1]
            assert np.allclose(g["dv"][s0:s1].sum(0), do[s0:s1].sum(0), atol=1e-12)
            assert np.max(np.abs(g["dk"][s0:s1].sum(0))) < 1e-12
        assert np.allclose(g["delta"], (do * g["out"]).sum(2), atol=1e-12)
        o, lse = oa.full_attention(q, k, v, cu, 0.5, causal=causal)
        assert np.allclose(g["out"], o, atol=1e-13) and np.allclose(g["lse"], lse, atol=1e-13)


def test_length_one_and_constant_values():
    """A length-1 sample: P = 1, so dV = dO and dQ = dK = 0.  Equal value rows:
    dP_ij = <dO_i, v> for every j, so dS = 0 and dQ = dK = 0 while dV = P^T dO."""
    q, k, v, do, cu = _batch([1], 2, 4, seed=4)
    g = ob.full_attention_backward(q, k, v, do, cu, 0.5)
    assert np.allclose(g["dv"], do) and np.abs(g["dq"]).max() == 0 and np.abs(g["dk"]).max() == 0
    q, k, v, do, cu = _batch([6], 2, 4, seed=5)
    v[:] = v[0]
    g = ob.full_attention_backward(q, k, v, do, cu, 0.5)
    assert np.abs(g["dq"]).max() < 1e-13 and np.abs(g["dk"]).max() < 1e-13
    assert np.abs(g["dv"]).max() > 0.1


def test_rows_match_the_full_backward():
    lengths, H, D = [17, 5, 33], 2, 8
    q, k, v, do, cu = _batch(lengths, H, D, seed=6)
    g = ob.full_attention_backward(q, k, v, do, cu, 0.4)
    toks = [0, 1, 16, 17, 21, 22, 40, 54]
    dq, lse, delta = ob.backward_rows(q, k, v, do, cu, 0.4, toks)
    assert np.max(np.abs(dq - g["dq"][toks])) < 1e-12
    assert np.max(np.abs(lse - g["lse"][toks])) < 1e-12
    assert np.max(np.abs(delta - g["delta"][toks])) < 1e-12
