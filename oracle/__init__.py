"""Oracle for the context-parallel (CP) ring-attention hot path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, float64 CPU
restatement of what the hot path computes.  It exists so that the CUDA path can
be checked against something written directly from the source pages.  Only the
test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import it; the library under ``long_context_gb300`` never does, and this package
imports nothing from that library (the two share no code).

Sources (cited by title and section throughout):

* [6D-CP]  "Megatron 架构与 6D 并行完整指南" (Megatron architecture and 6D
  parallelism guide), section 六 "上下文并行（CP）深入" (context parallelism in
  depth): the ``ring_attention`` listing -- the per-step block attention, the
  online-softmax merge of (O, m, l), the ring hand-off of KV and the final
  division by l.  Section 6.1 "Dynamic CP".
* [DCP]    "Dynamic Context Parallelism (DCP)", verl 0.9.0 documentation page
  ``docs/advance/dynamic_context_parallel``: per-micro-batch CP size,
  power-of-two subgroups plus a full DPxCP group, the even DPxCP world size of
  at least two, the per-rank limit ``max_seqlen_per_dp_cp_rank`` and its worked
  example (a 16,384-token budget at CP4 gives a limit of 4096).
* [MCore]  "20-Megatron-MCore-TP-PP-EP如何支撑MoE", section 1 (DCP requires
  ``max_seqlen_per_dp_cp_rank``) and section 4 (dynamic batches by
  ``max_token_len_per_gpu * sp_size``; dynamic CP split of remove-padding data).
* [VBP]    "VeRL Backend Parallelism", section 验证清单 (verification
  checklist): results at 1, 2 and 4 parallel ranks must match one card.

Modules:

* :mod:`oracle.attention` -- full softmax attention (the plain definition the
  ring reaches), the literal ring loop with the page's merge, the merge of
  stored per-step partials, and row-sampled attention for large inputs.
* :mod:`oracle.planner`   -- the dynamic-CP planner (CP size per sample and
  aligned-group first-fit packing into micro-batches) plus brute-force checkers.
* :mod:`oracle.backward`  -- the attention backward (dQ, dK, dV): the exact
  derivative of the forward's definition, in full and over the ring's blocks.
* :mod:`oracle.dcp`       -- selecting a micro-batch's samples into a packed
  array and restoring outputs to the original sample order ([DCP]).
* :mod:`oracle.decode`    -- decode-time CP: one new token per sequence
  against its sharded KV cache, with the LSE-form merge of the shards.
* :mod:`oracle.ulysses`   -- the Ulysses all-to-all as a head-group layout
  transform, and attention run per head group.
"""

from . import attention, backward, dcp, decode, planner, ulysses  # noqa: F401
