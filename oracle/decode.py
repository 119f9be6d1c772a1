"""Oracle for decode-time context parallelism.  TEST INFRASTRUCTURE ONLY.

"VeRL Backend Parallelism" (backend matrix and the vLLM inference section):
for the vLLM rollout and teacher engines, CP means only decode context
parallelism, ``decode_context_parallel_size`` -- the KV cache of a sequence
split over ranks that reuse the TP group -- and it is not training CP.  The
page gives no algorithm; the plainest reading, consistent with the training
ring ([6D-CP], section 六):

* each sequence b has a cache of L_b keys and values (packed THD rows
  ``cu_seqlens[b] .. cu_seqlens[b+1]``) and one new query token q_b per head,
  which attends to every cached key (the new token's own K, V are already in
  the cache);
* with decode CP size c the cache is cut into c contiguous shards of
  ``ceil(L_b / c)`` keys (the last shorter, possibly empty); shard s yields
  the normalised partial ``O_s = softmax(s_s) V_s`` and ``lse_s = ln sum
  exp(s_s)`` (an empty shard: ``O_s = 0``, ``lse_s = -inf``);
* the partials are merged in the LSE form: ``LSE = ln sum_s exp(lse_s)``,
  ``O = sum_s exp(lse_s - LSE) O_s`` -- the [6D-CP] merge with l_s = 1 and
  m_s = lse_s for normalised partials.

Shares no code with the CUDA path and imports nothing from it.
"""

from __future__ import annotations

import numpy as np

from .attention import NEG_INF, chunk_bounds


def decode_attention(q, k, v, cu_seqlens, scale):
    """The plain definition: ``q [B, H, D]`` against every cached key of its
    sequence.  Returns ``(O [B, H, D], LSE [B, H])``."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    cu = [int(x) for x in cu_seqlens]
    B, H, D = q.shape
    out = np.zeros((B, H, D))
    lse = np.full((B, H), NEG_INF)
    for b in range(B):
        s0, s1 = cu[b], cu[b + 1]
        if s1 <= s0:
            continue
        kb = np.transpose(k[s0:s1], (1, 0, 2))                      # [H, L, D]
        vb = np.transpose(v[s0:s1], (1, 0, 2))
        s = scale * np.matmul(kb, q[b][:, :, None])[:, :, 0]        # [H, L]
        mx = s.max(axis=1, keepdims=True)
        row = mx + np.log(np.exp(s - mx).sum(axis=1, keepdims=True))
        p = np.exp(s - row)
        out[b] = np.matmul(p[:, None, :], vb)[:, 0, :]
        lse[b] = row[:, 0]
    return out, lse


def shard_partials(q, k, v, cu_seqlens, c, scale):
    """Per-shard normalised partials: ``(O_s [c, B, H, D], lse_s [c, B, H])``."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    cu = [int(x) for x in cu_seqlens]
    B, H, D = q.shape
    o_s = np.zeros((c, B, H, D))
    l_s = np.full((c, B, H), NEG_INF)
    for b in range(B):
        s0 = cu[b]
        L = cu[b + 1] - s0
        for s, (a, z) in enumerate(chunk_bounds(L, c)):
            if z <= a:
                continue
            sub = [0, z - a]
            o, l = decode_attention(q[b:b + 1], k[s0 + a:s0 + z], v[s0 + a:s0 + z], sub, scale)
            o_s[s, b] = o[0]
            l_s[s, b] = l[0]
    return o_s, l_s


def merge_lse(o_s, lse_s):
    """The LSE-form merge over the leading (step) axis:
    ``LSE = ln sum_s exp(lse_s)``, ``O = sum_s exp(lse_s - LSE) O_s``
    (steps with lse = -inf get weight 0; all -inf gives O = 0, LSE = -inf)."""
    o_s = np.asarray(o_s, dtype=np.float64)
    lse_s = np.asarray(lse_s, dtype=np.float64)
    mx = lse_s.max(axis=0)
    finite = np.isfinite(mx)
    ref = np.where(finite, mx, 0.0)
    w = np.where(np.isfinite(lse_s), np.exp(lse_s - ref[None]), 0.0)
    tot = w.sum(axis=0)
    lse = np.where(tot > 0, ref + np.log(np.where(tot > 0, tot, 1.0)), NEG_INF)
    o = (w[..., None] * o_s).sum(axis=0) / np.where(tot > 0, tot, 1.0)[..., None]
    return o, lse
