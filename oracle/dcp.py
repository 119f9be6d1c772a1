"""Oracle for the data movement around attention under dynamic CP.
TEST INFRASTRUCTURE ONLY.

[DCP] (the verl page, "Dynamic Context Parallelism (DCP)"): every DPxCP rank
receives the same mini-batch and selects its assigned samples from that local
batch, with no input all-to-all; the Megatron THD forward gathers each dynamic
CP group's output; verl records the original sample IDs and restores their
order after the pipeline schedule.

On one device the mini-batch is one packed THD array in the original sample
order.  Reading of the pages' steps, written out plainly:

* the samples of micro-batch m are those the planner put in it, taken in the
  planner's order (longest first);
* selecting them builds a packed THD array of just those samples, in that
  order, with its own cu_seqlens (the prefix sum of their lengths);
* the CP group's output for a sample is the attention of that whole sample
  (the ring gathers the chunks back), so after attention on the selected
  array each sample's rows go back to the sample's original rows.

Shares no code with the CUDA path and imports nothing from it.
"""

from __future__ import annotations

import numpy as np

from .attention import full_attention, ring_attention


def micro_batch_samples(plan, m):
    """Sample ids of micro-batch ``m`` in the planner's order (``plan`` as
    returned by :func:`oracle.planner.plan`)."""
    return [b for b in plan["order"] if plan["micro_batch"][b] == m]


def select(x, cu_seqlens, ids):
    """Packed rows of samples ``ids`` (in that order) and their cu_seqlens.
    ``x`` is any array indexed by token first ([T, ...])."""
    cu = [int(c) for c in cu_seqlens]
    parts = [x[cu[b]:cu[b + 1]] for b in ids]
    lens = [cu[b + 1] - cu[b] for b in ids]
    out_cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64) if ids else np.zeros(1, np.int64)
    if parts:
        out = np.concatenate(parts, axis=0)
    else:
        out = np.zeros((0,) + tuple(x.shape[1:]), dtype=x.dtype)
    return out, out_cu


def restore(y, ids, cu_seqlens, out):
    """Writes the rows of packed samples ``ids`` (``y``, packed in that order)
    back to their original rows of ``out`` (original ``cu_seqlens``)."""
    cu = [int(c) for c in cu_seqlens]
    pos = 0
    for b in ids:
        L = cu[b + 1] - cu[b]
        out[cu[b]:cu[b + 1]] = y[pos:pos + L]
        pos += L
    return out


def dcp_forward(q, k, v, cu_seqlens, plan, scale, causal=True, ring=False):
    """Attention of a packed batch run the DCP way: for every micro-batch,
    select its samples, run attention on them (each at its CP size through
    the ring when ``ring`` is set, else the plain definition), and restore
    the outputs to the original sample order.  Returns ``(O, LSE)``."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    T, H, D = q.shape
    out = np.zeros((T, H, D))
    lse = np.full((T, H), -np.inf)
    for m in range(int(plan["num_micro_batches"])):
        ids = micro_batch_samples(plan, m)
        qs, cu_s = select(q, cu_seqlens, ids)
        ks, _ = select(k, cu_seqlens, ids)
        vs, _ = select(v, cu_seqlens, ids)
        if ring:
            cps = [int(plan["cp_size"][b]) for b in ids]
            o_s, l_s = ring_attention(qs, ks, vs, cu_s, cps, scale, causal=causal)
        else:
            o_s, l_s = full_attention(qs, ks, vs, cu_s, scale, causal=causal)
        restore(o_s, ids, cu_seqlens, out)
        restore(l_s, ids, cu_seqlens, lse)
    return out, lse
