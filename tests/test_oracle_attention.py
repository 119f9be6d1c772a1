"""Pins for the oracle's attention, ring loop and merge (CPU only).

Each test ties the oracle to something other than itself: hand-derived closed
forms (tests/golden), special cases that reduce to a mean or an identity,
SciPy's softmax/logsumexp, and the ring == full-attention identity of the
ring-attention section of the Megatron 6D guide (section 六).
"""

import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _num(x):
    if isinstance(x, (int, float)):
        return float(x)
    table = {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4),
             "ln5": math.log(5), "2ln2": 2 * math.log(2), "2ln3": 2 * math.log(3),
             "8/5": 8 / 5, "10/3": 10 / 3, "14/5": 14 / 5}
    return table[x]


def _arr(nested):
    if isinstance(nested, list):
        return np.array([_arr(x) for x in nested], dtype=np.float64)
    return _num(nested)


def _rand_batch(rng, lengths, H, D, scale_inputs=1.0):
    T = int(sum(lengths))
    q = rng.standard_normal((T, H, D)) * scale_inputs
    k = rng.standard_normal((T, H, D)) * scale_inputs
    v = rng.standard_normal((T, H, D))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return q, k, v, cu


# --------------------------------------------------------------------------
# Closed forms.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
def test_golden_closed_form(causal):
    g = json.load(open(os.path.join(GOLDEN, "attention_closed_form.json")))
    q, k, v = _arr(g["q"]), _arr(g["k"]), _arr(g["v"])
    cu = g["cu_seqlens"]
    exp = g["causal" if causal else "noncausal"]
    want_o, want_lse = _arr(exp["out"]), _arr(exp["lse"])
    out, lse = oa.full_attention(q, k, v, cu, g["scale"], causal=causal)
    np.testing.assert_allclose(out, want_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-12)
    # The literal ring reaches the same closed form at every CP size.
    for c in (1, 2, 3, 4):
        out_r, lse_r = oa.ring_attention(q, k, v, cu, [c, c], g["scale"], causal=causal)
        np.testing.assert_allclose(out_r, want_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse_r, want_lse, rtol=0, atol=1e-12)
    # Row-sampled evaluation agrees too.
    out_s, lse_s = oa.attention_rows(q, k, v, cu, g["scale"], range(5), causal=causal)
    np.testing.assert_allclose(out_s, want_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_s, want_lse, rtol=0, atol=1e-12)


def test_all_equal_scores_give_prefix_mean():
    """q = 0: every score is 0, so o_p is the mean of the visible v rows and
    LSE_p = ln(number visible); sample boundaries must not leak."""
    rng = np.random.default_rng(1)
    lengths = [5, 1, 17, 64, 3]
    q, k, v, cu = _rand_batch(rng, lengths, 3, 8)
    q[:] = 0.0
    for causal in (True, False):
        out, lse = oa.full_attention(q, k, v, cu, 0.3, causal=causal)
        for b, L in enumerate(lengths):
            s0 = cu[b]
            for p in range(L):
                n = p + 1 if causal else L
                np.testing.assert_allclose(out[s0 + p], v[s0:s0 + n].mean(axis=0),
                                           atol=1e-12)
                np.testing.assert_allclose(lse[s0 + p], math.log(n), atol=1e-12)
        for c in (2, 4, 8):
            out_r, lse_r = oa.ring_attention(q, k, v, cu, [c] * len(lengths), 0.3,
                                             causal=causal)
            np.testing.assert_allclose(out_r, out, atol=1e-12)
            np.testing.assert_allclose(lse_r, lse, atol=1e-12)


def test_length_one_sequence_returns_own_value():
    rng = np.random.default_rng(2)
    q, k, v, cu = _rand_batch(rng, [1, 1, 1], 4, 16)
    scale = 0.125
    out, lse = oa.full_attention(q, k, v, cu, scale)
    np.testing.assert_allclose(out, v, atol=1e-15)
    np.testing.assert_allclose(lse, scale * np.einsum("thd,thd->th", q, k), atol=1e-13)
    for c in (1, 2, 4):
        out_r, lse_r = oa.ring_attention(q, k, v, cu, [c] * 3, scale)
        np.testing.assert_allclose(out_r, v, atol=1e-15)
        np.testing.assert_allclose(lse_r, lse, atol=1e-13)


def test_noncausal_single_block_matches_scipy_softmax():
    rng = np.random.default_rng(3)
    L, H, D = 37, 2, 8
    q, k, v, cu = _rand_batch(rng, [L], H, D)
    scale = 0.37
    out, lse = oa.full_attention(q, k, v, cu, scale, causal=False)
    for h in range(H):
        s = scale * q[:, h, :] @ k[:, h, :].T
        np.testing.assert_allclose(out[:, h], softmax(s, axis=1) @ v[:, h], atol=1e-12)
        np.testing.assert_allclose(lse[:, h], logsumexp(s, axis=1), atol=1e-12)


def test_causal_matches_scipy_per_row():
    rng = np.random.default_rng(4)
    L, H, D = 29, 2, 8
    q, k, v, cu = _rand_batch(rng, [L], H, D)
    out, lse = oa.full_attention(q, k, v, cu, 0.5, causal=True, row_block=7)
    for h in range(H):
        for p in range(L):
            s = 0.5 * k[:p + 1, h, :] @ q[p, h, :]
            np.testing.assert_allclose(out[p, h], softmax(s) @ v[:p + 1, h], atol=1e-12)
            np.testing.assert_allclose(lse[p, h], logsumexp(s), atol=1e-12)


def test_key_permutation_invariance_noncausal():
    rng = np.random.default_rng(5)
    q, k, v, cu = _rand_batch(rng, [23], 2, 8)
    perm = rng.permutation(23)
    out, lse = oa.full_attention(q, k, v, cu, 0.4, causal=False)
    # Permuting keys and values together leaves every query's output alone.
    out_p, lse_p = oa.full_attention(q, k[perm], v[perm], cu, 0.4, causal=False)
    np.testing.assert_allclose(out_p, out, atol=1e-12)
    np.testing.assert_allclose(lse_p, lse, atol=1e-12)


# --------------------------------------------------------------------------
# Ring == full attention (the identity the listing relies on).
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
def test_ring_equals_full_attention_tiny(causal):
    rng = np.random.default_rng(6)
    for L in list(range(1, 41)):
        q, k, v, cu = _rand_batch(rng, [L], 2, 8)
        ref_o, ref_l = oa.full_attention(q, k, v, cu, 0.35, causal=causal)
        for c in (1, 2, 3, 4, 8):
            o, lse = oa.ring_attention(q, k, v, cu, [c], 0.35, causal=causal)
            assert np.max(np.abs(o - ref_o)) <= 1e-12
            assert np.max(np.abs(lse - ref_l)) <= 1e-12


def test_ring_equals_full_attention_mixed_batch():
    rng = np.random.default_rng(7)
    lengths = [1, 2, 7, 33, 64, 65, 100, 5]
    cps = [1, 2, 4, 8, 2, 4, 8, 8]
    q, k, v, cu = _rand_batch(rng, lengths, 3, 16, scale_inputs=2.0)
    ref_o, ref_l = oa.full_attention(q, k, v, cu, 0.25)
    o, lse = oa.ring_attention(q, k, v, cu, cps, 0.25)
    assert np.max(np.abs(o - ref_o)) <= 1e-12
    assert np.max(np.abs(lse - ref_l)) <= 1e-12


def test_tiny_workload_ring_cp2_matches_full():
    """The 1024-token, CP=2, H=4, D=64 case of the workload list."""
    rng = np.random.default_rng(8)
    q, k, v, cu = _rand_batch(rng, [1024], 4, 64)
    scale = 1.0 / 8.0
    ref_o, ref_l = oa.full_attention(q, k, v, cu, scale)
    o, lse = oa.ring_attention(q, k, v, cu, [2], scale)
    assert np.max(np.abs(o - ref_o)) <= 1e-12
    assert np.max(np.abs(lse - ref_l)) <= 1e-12


def test_ring_partials_merge_back_to_ring_output():
    rng = np.random.default_rng(9)
    lengths = [9, 40, 3]
    cps = [4, 2, 8]
    q, k, v, cu = _rand_batch(rng, lengths, 2, 8)
    o, lse, (os_, ms_, ls_) = oa.ring_attention(q, k, v, cu, cps, 0.3, num_steps=8)
    mo, mm, ml = oa.merge_partials(os_, ms_, ls_)
    np.testing.assert_allclose(mo, o, atol=1e-12)
    np.testing.assert_allclose(mm + np.log(ml), lse, atol=1e-12)
    # Steps that do not exist, or see nothing, hold the empty partial.
    b = 2  # L=3 at CP=8: chunks of 1 token, ranks 3..7 are empty
    assert np.all(np.isneginf(ms_[3:, cu[b]:cu[b + 1]]) | (ls_[3:, cu[b]:cu[b + 1]] > 0))
    # Token 0 of sample 0 (rank 0, CP 4) sees only its own chunk at step 0.
    assert np.all(np.isneginf(ms_[1:4, 0])) and np.all(ls_[1:4, 0] == 0)
    # Ring direction: sample 0 (L=9, CP 4, chunks of 3) rank 2 holds chunk 1
    # at step 1 and chunk 3 (empty) at step 3; KV arrives from the previous rank.
    assert np.all(np.isfinite(ms_[1, 6:9])) and np.all(np.isfinite(ms_[2, 6:9]))
    assert np.all(np.isneginf(ms_[3, 6:9]))


def test_chunk_bounds():
    assert oa.chunk_bounds(10, 4) == [(0, 3), (3, 6), (6, 9), (9, 10)]
    assert oa.chunk_bounds(3, 8) == [(0, 1), (1, 2), (2, 3)] + [(3, 3)] * 5
    assert oa.chunk_bounds(131072, 4) == [(0, 32768), (32768, 65536),
                                          (65536, 98304), (98304, 131072)]
    assert oa.chunk_bounds(0, 2) == [(0, 0), (0, 0)]


# --------------------------------------------------------------------------
# Merge.
# --------------------------------------------------------------------------

def test_merge_single_step_is_identity_up_to_normalisation():
    rng = np.random.default_rng(10)
    o = rng.standard_normal((1, 50, 4, 8))
    m = rng.uniform(-5, 5, (1, 50, 4))
    l = rng.uniform(1, 1024, (1, 50, 4))
    mo, mm, ml = oa.merge_partials(o, m, l)
    np.testing.assert_allclose(mo, o[0] / l[0][..., None], rtol=1e-15)
    np.testing.assert_array_equal(mm, m[0])
    np.testing.assert_allclose(ml, l[0], rtol=1e-15)


def test_merge_of_split_row_equals_unsplit_softmax():
    """Split one score row into S random parts; each part's (O, m, l) built
    from its own max; the fold must equal the softmax over the whole row."""
    rng = np.random.default_rng(11)
    for trial in range(20):
        n, d, S = int(rng.integers(5, 60)), 6, int(rng.integers(1, 9))
        s = rng.normal(0, 3, n)
        vv = rng.standard_normal((n, d))
        part = rng.integers(0, S, n)
        o_st = np.zeros((S, d))
        m_st = np.full(S, -np.inf)
        l_st = np.zeros(S)
        for p in range(S):
            idx = np.nonzero(part == p)[0]
            if len(idx) == 0:
                continue
            m_st[p] = s[idx].max()
            w = np.exp(s[idx] - m_st[p])
            l_st[p] = w.sum()
            o_st[p] = w @ vv[idx]
        mo, mm, ml = oa.merge_partials(o_st, m_st, l_st)
        np.testing.assert_allclose(mo, softmax(s) @ vv, atol=1e-12)
        np.testing.assert_allclose(mm + np.log(ml), logsumexp(s), atol=1e-12)
        assert mm == s.max()


def test_merge_step_order_does_not_matter():
    rng = np.random.default_rng(12)
    S = 8
    o = rng.standard_normal((S, 40, 3, 8))
    m = rng.uniform(-5, 5, (S, 40, 3))
    l = rng.uniform(1, 1024, (S, 40, 3))
    m[2, :5] = -np.inf
    l[2, :5] = 0.0
    o[2, :5] = 0.0
    base = oa.merge_partials(o, m, l)
    for _ in range(5):
        perm = rng.permutation(S)
        other = oa.merge_partials(o[perm], m[perm], l[perm])
        for a, b in zip(base, other):
            np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)


def test_merge_empty_steps():
    o = np.zeros((3, 2, 4))
    m = np.full((3, 2), -np.inf)
    l = np.zeros((3, 2))
    mo, mm, ml = oa.merge_partials(o, m, l)
    assert np.all(mo == 0) and np.all(np.isneginf(mm)) and np.all(ml == 0)
    o[1, 0] = [1, 2, 3, 4]
    m[1, 0] = 2.0
    l[1, 0] = 4.0
    mo, mm, ml = oa.merge_partials(o, m, l)
    np.testing.assert_allclose(mo[0], [0.25, 0.5, 0.75, 1.0])
    assert mm[0] == 2.0 and ml[0] == 4.0
    assert np.all(mo[1] == 0) and np.isneginf(mm[1])


def test_merge_alpha_beta_by_hand():
    """Two steps with maxima 0 and ln 2: alpha = 1/2, beta = 1."""
    o = np.array([[[2.0]], [[6.0]]])
    m = np.array([[0.0], [math.log(2)]])
    l = np.array([[1.0], [3.0]])
    mo, mm, ml = oa.merge_partials(o, m, l)
    # l = 0.5 * 1 + 3 = 3.5, O = 0.5 * 2 + 6 = 7 -> O / l = 2
    np.testing.assert_allclose(ml, [3.5], rtol=1e-15)
    np.testing.assert_allclose(mo, [[2.0]], rtol=1e-15)
    np.testing.assert_allclose(mm, [math.log(2)], rtol=0)


def test_attention_rows_matches_full():
    rng = np.random.default_rng(13)
    lengths = [70, 1, 130]
    q, k, v, cu = _rand_batch(rng, lengths, 2, 8)
    ref_o, ref_l = oa.full_attention(q, k, v, cu, 0.3, row_block=16)
    toks = [0, 69, 70, 71, 140, 200]
    o, lse = oa.attention_rows(q, k, v, cu, 0.3, toks)
    np.testing.assert_allclose(o, ref_o[toks], atol=1e-12)
    np.testing.assert_allclose(lse, ref_l[toks], atol=1e-12)
