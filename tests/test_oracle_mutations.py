"""Planted mistakes in the oracle must fail its pins (CPU only).

Each case replaces one oracle function with a copy that carries one
plausible mistake (a dropped scale, a causal off-by-one, a leaking sample
boundary, swapped operands, a wrong log base, a missing rescale in the merge,
a floor instead of a ceiling in the chunking, a wrong CP rule, a dropped
term or transposed operand in the backward, a wrong weight in the LSE-form
merge, a strided head grouping, a reordered sample selection), runs the pin
tests that cover that function, and requires at least one of them to fail.
The oracle itself is untouched: the copies live in this file and are patched
in for the duration of one case.  A control case runs the same pins on the
unpatched oracle and requires all of them to pass.
"""

import numpy as np
import pytest

import test_oracle_attention as attn_pins
import test_oracle_backward as bwd_pins
import test_oracle_dcp as dcp_pins
import test_oracle_decode as dec_pins
import test_oracle_planner as plan_pins
import test_oracle_ulysses as uly_pins
from oracle import attention as oa
from oracle import backward as ob
from oracle import dcp as od
from oracle import decode as odc
from oracle import planner as op
from oracle import ulysses as ou


# ------------------------------------------------------- full attention --

def _full_attention_with(mistake):
    """Full attention per sample, head and query row, with one mistake."""

    def full_attention(q, k, v, cu_seqlens, scale, causal=True, row_block=1024):
        q = np.asarray(q, dtype=np.float64)
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        cu = [int(x) for x in cu_seqlens]
        T, H, D = q.shape
        out = np.zeros((T, H, D))
        lse = np.full((T, H), -np.inf)
        sc = 1.0 if mistake == "no_scale" else scale
        for b in range(len(cu) - 1):
            s0, s1 = cu[b], cu[b + 1]
            for p in range(s1 - s0):
                k_lo = 0 if mistake == "boundary_leak" else s0
                if causal:
                    last = s0 + p
                    if mistake == "causal_plus1":
                        last += 1
                    if mistake == "causal_minus1":
                        last -= 1
                    k_hi = min(last + 1, s1)
                else:
                    k_hi = s1
                if k_hi <= k_lo:
                    continue
                for h in range(H):
                    a, keys = q[s0 + p, h], k[k_lo:k_hi, h]
                    if mistake == "qk_swap":
                        a, keys = k[s0 + p, h], q[k_lo:k_hi, h]
                    s = sc * (keys @ a)
                    mx = s.max()
                    row_lse = mx + np.log(np.exp(s - mx).sum())
                    vals = k[k_lo:k_hi, h] if mistake == "kv_swap" else v[k_lo:k_hi, h]
                    out[s0 + p, h] = np.exp(s - row_lse) @ vals
                    lse[s0 + p, h] = row_lse / np.log(2.0) if mistake == "lse_log2" else row_lse
        return out, lse

    return full_attention


# ---------------------------------------------------- ring and merge parts --

_ORIG_BLOCK = oa.block_attention


def _merge_step_with(mistake):
    def merge_step(o, m, l, o_step, m_step, l_step):
        m_new = np.maximum(m, m_step)
        alpha = oa._exp_diff(m, m_new)
        beta = oa._exp_diff(m_step, m_new)
        if mistake == "beta_from_running_max":
            beta = oa._exp_diff(m, m_new)
        if mistake == "l_not_rescaled":
            l_new = l + beta * l_step
        else:
            l_new = alpha * l + beta * l_step
        if mistake == "o_not_rescaled":
            o_new = o + beta[..., None] * o_step
        else:
            o_new = alpha[..., None] * o + beta[..., None] * o_step
        return o_new, m_new, l_new

    return merge_step


def _block_attention_normalised(q_blk, k_blk, v_blk, q_pos, k_pos, scale, causal=True):
    """O_step divided by l_step while l_step is still merged (the reading the
    finalize step O / l rules out)."""
    o_step, m_step, l_step = _ORIG_BLOCK(q_blk, k_blk, v_blk, q_pos, k_pos, scale, causal)
    safe = np.where(l_step > 0, l_step, 1.0)
    return o_step / safe[..., None], m_step, l_step


def _chunk_bounds_floor(L, c):
    """floor(L / c) per chunk instead of the ceiling (the tail goes missing)."""
    chunk = L // c if c > 0 else 0
    return [(min(r * chunk, L), min((r + 1) * chunk, L)) for r in range(c)]


# ------------------------------------------------------------ backward --

def _sample_backward_with(mistake):
    """The per-sample backward (matrix form) with one mistake."""

    def sample_backward(qb, kb, vb, dob, scale, causal):
        H, L, _ = qb.shape
        kt = np.transpose(kb, (0, 2, 1))
        s = scale * np.matmul(qb, kt)
        if causal:
            vis = np.arange(L)[None, :] <= np.arange(L)[:, None]
            s = np.where(vis[None], s, -np.inf)
        mx = s.max(axis=2, keepdims=True)
        lse = mx + np.log(np.exp(s - mx).sum(axis=2, keepdims=True))
        p = np.exp(s - lse)
        o = np.matmul(p, vb)
        pt = p if mistake == "p_not_transposed_in_dv" else np.transpose(p, (0, 2, 1))
        dv = np.matmul(pt, dob)
        dp = np.matmul(dob, np.transpose(vb, (0, 2, 1)))
        delta = (p * dp).sum(axis=2, keepdims=True)
        ds = p * dp if mistake == "drop_delta" else p * (dp - delta)
        dq = np.matmul(ds, kb) * (1.0 if mistake == "dq_unscaled" else scale)
        dst = ds if mistake == "ds_not_transposed_in_dk" else np.transpose(ds, (0, 2, 1))
        dk = np.matmul(dst, qb) * (1.0 if mistake == "dk_unscaled" else scale)
        return dq, dk, dv, lse[:, :, 0], delta[:, :, 0], o

    return sample_backward


# ------------------------------------------- LSE merge, Ulysses, DCP --

def _merge_lse_with(mistake):
    def merge_lse(o_s, lse_s):
        o_s = np.asarray(o_s, dtype=np.float64)
        lse_s = np.asarray(lse_s, dtype=np.float64)
        mx = lse_s.max(axis=0)
        ref = np.where(np.isfinite(mx), mx, 0.0)
        w = np.where(np.isfinite(lse_s), np.exp(lse_s - ref[None]), 0.0)
        if mistake == "unweighted":
            w = np.where(np.isfinite(lse_s), 1.0, 0.0)
        tot = w.sum(axis=0)
        lse = np.where(tot > 0, ref + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
        if mistake == "lse_is_max":
            lse = mx
        o = (w[..., None] * o_s).sum(axis=0)
        if mistake != "not_renormalised":
            o = o / np.where(tot > 0, tot, 1.0)[..., None]
        return o, lse

    return merge_lse


def _to_groups_strided(x, P):
    """Head h to group h mod P (instead of h // (H / P))."""
    x = np.asarray(x)
    T, H = x.shape[0], x.shape[1]
    return np.ascontiguousarray(np.moveaxis(x.reshape((T, H // P, P) + x.shape[2:]), 2, 0))


def _from_groups_strided(y, P):
    y = np.asarray(y)
    T, Hp = y.shape[1], y.shape[2]
    return np.ascontiguousarray(np.moveaxis(y, 0, 2).reshape((T, P * Hp) + y.shape[3:]))


_ORIG_SELECT = od.select


def _select_sorted(x, cu_seqlens, ids):
    """The samples in index order instead of the order asked for."""
    return _ORIG_SELECT(x, cu_seqlens, sorted(ids))


# ------------------------------------------------------------- planner --

def _cp_size_with(mistake):
    def cp_size_for_length(L, limit, max_cp):
        cands = op.cp_candidates(max_cp)
        if mistake == "largest_fitting":
            fits = [c for c in cands if -(-L // c) <= limit]
            return fits[-1] if fits else None
        if mistake == "strict_limit":
            for c in cands:
                if -(-L // c) < limit:
                    return c
            return None
        if mistake == "floor_division":
            for c in cands:
                if L // c <= limit:
                    return c
            return None
        raise ValueError(mistake)

    return cp_size_for_length


# --------------------------------------------------------------- runner --

# Pins that call the full-attention definition, pins of the ring loop and
# the merge, and pins of the planner's CP rule.
ATTENTION_PINS = [
    attn_pins.test_golden_closed_form,
    attn_pins.test_all_equal_scores_give_prefix_mean,
    attn_pins.test_length_one_sequence_returns_own_value,
    attn_pins.test_noncausal_single_block_matches_scipy_softmax,
    attn_pins.test_causal_matches_scipy_per_row,
    attn_pins.test_ring_equals_full_attention_tiny,
    attn_pins.test_ring_equals_full_attention_mixed_batch,
]
RING_PINS = [
    attn_pins.test_golden_closed_form,
    attn_pins.test_ring_equals_full_attention_tiny,
    attn_pins.test_ring_equals_full_attention_mixed_batch,
    attn_pins.test_chunk_bounds,
    attn_pins.test_merge_of_split_row_equals_unsplit_softmax,
    attn_pins.test_merge_alpha_beta_by_hand,
]
BACKWARD_PINS = [
    bwd_pins.test_matches_finite_differences_of_the_forward,
    bwd_pins.test_ring_blocks_sum_to_the_full_backward,
    bwd_pins.test_softmax_identities,
    bwd_pins.test_length_one_and_constant_values,
    bwd_pins.test_rows_match_the_full_backward,
]
DECODE_PINS = [
    dec_pins.test_decode_matches_textbook_softmax,
    dec_pins.test_decode_is_the_last_row_of_causal_attention,
    dec_pins.test_shards_merge_to_the_whole,
    dec_pins.test_special_cases,
]
ULYSSES_PINS = [uly_pins.test_layout_by_hand_and_round_trip,
                uly_pins.test_ulysses_attention_equals_full_attention]
DCP_PINS = [dcp_pins.test_select_layout_and_round_trip,
            dcp_pins.test_micro_batches_partition_the_batch,
            dcp_pins.test_dcp_forward_equals_full_attention]
PLANNER_PINS = [
    plan_pins.test_golden_plans,
    plan_pins.test_page_worked_example_limit,
    plan_pins.test_cp_size_brute_force,
]


def _calls(fn):
    """One call per combination of the pin's parametrize marks."""
    combos = [{}]
    for mark in getattr(fn, "pytestmark", []):
        if mark.name != "parametrize":
            continue
        names = mark.args[0]
        names = [n.strip() for n in names.split(",")] if isinstance(names, str) else list(names)
        combos = [dict(c, **dict(zip(names, val if len(names) > 1 else (val,))))
                  for c in combos for val in mark.args[1]]
    return [(fn, kw) for kw in combos]


def _failures(pins):
    failed = 0
    for fn in pins:
        for f, kw in _calls(fn):
            try:
                f(**kw)
            except Exception:  # an assertion, or a mistake that breaks the arithmetic
                failed += 1
    return failed


def test_control_every_pin_passes_on_the_oracle():
    assert _failures(ATTENTION_PINS + RING_PINS + BACKWARD_PINS + DECODE_PINS + ULYSSES_PINS
                     + DCP_PINS + PLANNER_PINS) == 0


@pytest.mark.parametrize("mistake", ["no_scale", "causal_plus1", "causal_minus1",
                                     "boundary_leak", "qk_swap", "kv_swap", "lse_log2"])
def test_full_attention_mistake_fails_a_pin(monkeypatch, mistake):
    monkeypatch.setattr(oa, "full_attention", _full_attention_with(mistake))
    assert _failures(ATTENTION_PINS) > 0


def test_correct_copy_passes_the_pins(monkeypatch):
    """The planted copies differ from the oracle only by their mistake: with
    none, the copy passes every attention pin."""
    monkeypatch.setattr(oa, "full_attention", _full_attention_with(None))
    assert _failures(ATTENTION_PINS) == 0


@pytest.mark.parametrize("mistake", ["beta_from_running_max", "l_not_rescaled",
                                     "o_not_rescaled"])
def test_merge_mistake_fails_a_pin(monkeypatch, mistake):
    monkeypatch.setattr(oa, "merge_step", _merge_step_with(mistake))
    assert _failures(RING_PINS) > 0


def test_normalised_step_output_fails_a_pin(monkeypatch):
    monkeypatch.setattr(oa, "block_attention", _block_attention_normalised)
    assert _failures(RING_PINS) > 0


def test_floor_chunking_fails_a_pin(monkeypatch):
    monkeypatch.setattr(oa, "chunk_bounds", _chunk_bounds_floor)
    assert _failures(RING_PINS) > 0


@pytest.mark.parametrize("mistake", ["largest_fitting", "strict_limit", "floor_division"])
def test_cp_rule_mistake_fails_a_pin(monkeypatch, mistake):
    monkeypatch.setattr(op, "cp_size_for_length", _cp_size_with(mistake))
    assert _failures(PLANNER_PINS) > 0


def test_correct_backward_copy_passes_the_pins(monkeypatch):
    monkeypatch.setattr(ob, "_sample_backward", _sample_backward_with(None))
    assert _failures(BACKWARD_PINS) == 0


@pytest.mark.parametrize("mistake", ["drop_delta", "p_not_transposed_in_dv",
                                     "ds_not_transposed_in_dk", "dq_unscaled", "dk_unscaled"])
def test_backward_mistake_fails_a_pin(monkeypatch, mistake):
    monkeypatch.setattr(ob, "_sample_backward", _sample_backward_with(mistake))
    assert _failures(BACKWARD_PINS) > 0


@pytest.mark.parametrize("mistake", ["unweighted", "lse_is_max", "not_renormalised"])
def test_lse_merge_mistake_fails_a_pin(monkeypatch, mistake):
    monkeypatch.setattr(odc, "merge_lse", _merge_lse_with(mistake))
    assert _failures(DECODE_PINS) > 0


def test_strided_head_groups_fail_a_pin(monkeypatch):
    # A consistent pair: round trips still pass, the hand-built layout does not.
    monkeypatch.setattr(ou, "to_head_groups", _to_groups_strided)
    monkeypatch.setattr(ou, "from_head_groups", _from_groups_strided)
    assert _failures(ULYSSES_PINS) > 0


def test_reordered_selection_fails_a_pin(monkeypatch):
    monkeypatch.setattr(od, "select", _select_sorted)
    assert _failures(DCP_PINS) > 0
