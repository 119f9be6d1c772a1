"""Pins of the decode-time CP oracle (oracle/decode.py), CPU only."""

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import attention as oa
from oracle import decode as odc


def _cache(lengths, H, D, seed):
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    k, v = (rng.normal(0.0, 1.0, (T, H, D)) for _ in range(2))
    q = rng.normal(0.0, 1.0, (len(lengths), H, D))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return q, k, v, cu


def test_decode_matches_textbook_softmax():
    """Each (sequence, head): scipy's softmax of the score row times V."""
    lengths, H, D = [7, 1, 30], 2, 8
    q, k, v, cu = _cache(lengths, H, D, seed=1)
    o, lse = odc.decode_attention(q, k, v, cu, 0.4)
    for b in range(len(lengths)):
        for h in range(H):
            s = 0.4 * k[cu[b]:cu[b + 1], h] @ q[b, h]
            assert np.allclose(o[b, h], softmax(s) @ v[cu[b]:cu[b + 1], h], atol=1e-13)
            assert abs(lse[b, h] - logsumexp(s)) < 1e-13


def test_decode_is_the_last_row_of_causal_attention():
    """The new token as the last query of its sequence (its K, V in the cache)
    is the last row of the forward's causal attention."""
    lengths, H, D = [5, 12], 2, 4
    q, k, v, cu = _cache(lengths, H, D, seed=2)
    qfull = np.zeros_like(k)
    for b in range(len(lengths)):
        qfull[cu[b + 1] - 1] = q[b]
    o_full, l_full = oa.full_attention(qfull, k, v, cu, 0.5)
    o, lse = odc.decode_attention(q, k, v, cu, 0.5)
    for b in range(len(lengths)):
        assert np.allclose(o[b], o_full[cu[b + 1] - 1], atol=1e-13)
        assert np.allclose(lse[b], l_full[cu[b + 1] - 1], atol=1e-13)


@pytest.mark.parametrize("c", [1, 2, 3, 4, 8])
def test_shards_merge_to_the_whole(c):
    lengths, H, D = [1, 2, 9, 40, 17], 2, 8
    q, k, v, cu = _cache(lengths, H, D, seed=3)
    o, lse = odc.decode_attention(q, k, v, cu, 0.3)
    o_s, l_s = odc.shard_partials(q, k, v, cu, c, 0.3)
    o_m, l_m = odc.merge_lse(o_s, l_s)
    assert np.max(np.abs(o_m - o)) < 1e-12 and np.max(np.abs(l_m - lse)) < 1e-12


def test_special_cases():
    """q = 0: O is the mean of V and LSE = ln L; an all-empty set of shards
    merges to (0, -inf)."""
    lengths, H, D = [6, 1], 2, 4
    q, k, v, cu = _cache(lengths, H, D, seed=4)
    q[:] = 0
    o, lse = odc.decode_attention(q, k, v, cu, 0.7)
    assert np.allclose(o[0], v[0:6].mean(0)) and np.allclose(lse[0], np.log(6))
    assert np.allclose(o[1], v[6]) and np.allclose(lse[1], 0.0)
    o_m, l_m = odc.merge_lse(np.zeros((3, 1, 1, 4)), np.full((3, 1, 1), -np.inf))
    assert np.all(o_m == 0) and np.all(np.isneginf(l_m))
