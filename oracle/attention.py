"""Oracle attention: float64, CPU, NumPy.  TEST INFRASTRUCTURE ONLY.

Everything here follows [6D-CP] (see ``oracle/__init__.py`` for the source
keys).  Arrays use the packed THD layout: ``q, k, v`` are ``[T, H, D]`` float64
arrays holding every sample's tokens back to back, and ``cu_seqlens`` is the
``[B + 1]`` prefix sum of the sample lengths.  Positions are 0-based within a
sample.  Causal attention lets query position ``p`` see key positions ``0..p``
of its own sample; non-causal attention lets it see the whole sample.

Conventions where the page is silent (each is also listed in the design notes):

* ``O_step`` returned by a block is *unnormalised* (sum of ``exp(s - m_step) v``);
  only that reading makes the listing's final ``O / l`` correct.
* ``exp(-inf - (-inf))`` is taken as 0: alpha = 0 when the running max is
  -inf, beta = 0 when the step max is -inf.  An empty state stays (0, -inf, 0);
  finalising l = 0 gives O = 0 and LSE = -inf.
* LSE is the natural log of the row's exponential sum in the scaled-score
  domain: ``LSE = m + ln(l)``.
* A sample of length L split over c CP ranks uses contiguous chunks of
  ``ceil(L / c)`` tokens; the last chunk is shorter and may be empty.
* At ring step s, rank i holds the KV chunk of rank ``(i - s) mod c``: KV moves
  to the next rank and arrives from the previous one each step.
"""

from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


# ---------------------------------------------------------------------------
# (c1) Full softmax attention: the plain definition.
# ---------------------------------------------------------------------------

def full_attention(q, k, v, cu_seqlens, scale, causal=True, row_block=1024):
    """Full softmax attention per sample and head, float64.

    For each query row p the scores are ``s_j = scale * <q_p, k_j>`` over the
    visible keys j; ``LSE_p = ln sum_j exp(s_j)`` and
    ``o_p = sum_j exp(s_j - LSE_p) v_j``.  [6D-CP] states this as the problem:
    every query has to interact with every (visible) key and value.

    Query rows are evaluated ``row_block`` at a time only to bound memory;
    each row's arithmetic is the definition above, unchanged.

    Returns ``(out [T, H, D], lse [T, H])``.  Rows of empty samples do not exist.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    cu = [int(x) for x in cu_seqlens]
    T, H, D = q.shape
    out = np.zeros((T, H, D))
    lse = np.full((T, H), NEG_INF)
    for b in range(len(cu) - 1):
        s0, s1 = cu[b], cu[b + 1]
        L = s1 - s0
        if L <= 0:
            continue
        kb = np.transpose(k[s0:s1], (1, 0, 2))  # [H, L, D]
        vb = np.transpose(v[s0:s1], (1, 0, 2))
        for r0 in range(0, L, row_block):
            r1 = min(L, r0 + row_block)
            kend = r1 if causal else L
            qb = np.transpose(q[s0 + r0:s0 + r1], (1, 0, 2))  # [H, R, D]
            s = scale * np.matmul(qb, np.transpose(kb[:, :kend], (0, 2, 1)))
            if causal:
                rows = np.arange(r0, r1)[:, None]
                cols = np.arange(kend)[None, :]
                s = np.where(cols <= rows, s, NEG_INF)
            mx = s.max(axis=2, keepdims=True)
            row_lse = mx + np.log(np.exp(s - mx).sum(axis=2, keepdims=True))
            p = np.exp(s - row_lse)
            o = np.matmul(p, vb[:, :kend])  # [H, R, D]
            out[s0 + r0:s0 + r1] = np.transpose(o, (1, 0, 2))
            lse[s0 + r0:s0 + r1] = np.transpose(row_lse[:, :, 0], (1, 0))
    return out, lse


def attention_rows(q, k, v, cu_seqlens, scale, tokens, causal=True):
    """The same definition as :func:`full_attention`, for selected query tokens.

    ``tokens`` lists packed token indices; every head of each listed token is
    computed.  Used to check outputs at sizes where the whole result would
    take the CPU too long.  ``q, k, v`` may be any arrays convertible to
    float64 (for example bf16 torch tensors; they are upcast exactly, one
    sample at a time).  Returns ``(out [n, H, D], lse [n, H])`` in the order of
    ``tokens``.
    """
    cu = np.asarray([int(x) for x in cu_seqlens], dtype=np.int64)
    H, D = q.shape[1], q.shape[2]
    tokens = [int(t) for t in tokens]
    out = np.zeros((len(tokens), H, D))
    lse = np.zeros((len(tokens), H))
    by_sample = {}
    for n, t in enumerate(tokens):
        b = int(np.searchsorted(cu, t, side="right") - 1)
        by_sample.setdefault(b, []).append(n)
    for b, idx in by_sample.items():
        s0, s1 = int(cu[b]), int(cu[b + 1])
        kend_max = max(tokens[n] for n in idx) + 1 if causal else s1
        # [H, n_k, D] float64 copies of this sample's visible keys and values.
        kt = np.ascontiguousarray(np.transpose(_f64(k[s0:kend_max]), (1, 0, 2)))
        vt = np.ascontiguousarray(np.transpose(_f64(v[s0:kend_max]), (1, 0, 2)))
        for n in idx:
            t = tokens[n]
            nk = (t - s0 + 1) if causal else (s1 - s0)
            qt = _f64(q[t])                                          # [H, D]
            s = scale * np.matmul(kt[:, :nk], qt[:, :, None])[:, :, 0]  # [H, nk]
            mx = s.max(axis=1, keepdims=True)
            row_lse = mx + np.log(np.exp(s - mx).sum(axis=1, keepdims=True))
            p_ = np.exp(s - row_lse)
            out[n] = np.matmul(p_[:, None, :], vt[:, :nk])[:, 0, :]
            lse[n] = row_lse[:, 0]
    return out, lse


def _f64(x):
    """Exact float64 copy of a NumPy array or a (CPU) torch tensor."""
    if hasattr(x, "detach"):
        import torch  # only when handed torch tensors
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# (c2) The literal ring loop of [6D-CP].
# ---------------------------------------------------------------------------

def chunk_bounds(L, c):
    """Contiguous CP chunks of a length-L sample split over c ranks.

    Chunk r holds positions ``[r * ceil(L/c), min((r + 1) * ceil(L/c), L))``,
    clamped to L; the last chunks may be short or empty.  The page's example
    (128K tokens at CP=4 -> 32K per GPU) divides evenly; the split of a length
    that does not divide is not stated, and this is the plainest reading.
    """
    chunk = -(-L // c) if c > 0 else 0
    return [(min(r * chunk, L), min((r + 1) * chunk, L)) for r in range(c)]


def block_attention(q_blk, k_blk, v_blk, q_pos, k_pos, scale, causal=True):
    """One ring step's block attention, the listing's ``flash_attention`` call.

    ``q_blk [H, Lq, D]`` at sample positions ``q_pos [Lq]`` attends to
    ``k_blk, v_blk [H, Lk, D]`` at positions ``k_pos [Lk]``.  Returns the step's
    partial result ``(O_step [H, Lq, D], m_step [H, Lq], l_step [H, Lq])``:
    ``m_step`` is the row max of the visible scaled scores (-inf when no key is
    visible), ``l_step = sum exp(s - m_step)`` and ``O_step`` is the
    unnormalised ``sum exp(s - m_step) v``.
    """
    Hh, Lq, Dd = q_blk.shape
    if Lq == 0:
        return np.zeros((Hh, 0, Dd)), np.zeros((Hh, 0)), np.zeros((Hh, 0))
    if k_blk.shape[1] == 0:
        return (np.zeros((Hh, Lq, Dd)), np.full((Hh, Lq), NEG_INF),
                np.zeros((Hh, Lq)))
    s = scale * np.matmul(q_blk, np.transpose(k_blk, (0, 2, 1)))  # [H, Lq, Lk]
    if causal:
        visible = k_pos[None, :] <= q_pos[:, None]
    else:
        visible = np.ones((Lq, k_pos.shape[0]), dtype=bool)
    s = np.where(visible[None], s, NEG_INF)
    m_step = s.max(axis=2)
    has_any = np.isfinite(m_step)
    ref = np.where(has_any, m_step, 0.0)
    p = np.where(visible[None], np.exp(s - ref[:, :, None]), 0.0)
    l_step = p.sum(axis=2)
    o_step = np.matmul(p, v_blk)
    return o_step, m_step, l_step


def _exp_diff(a, b):
    """exp(a - b) with the convention exp(-inf - x) = 0 (also for x = -inf)."""
    safe = np.isfinite(a)
    return np.where(safe, np.exp(np.where(safe, a, 0.0) - np.where(safe, b, 0.0)), 0.0)


def merge_step(o, m, l, o_step, m_step, l_step):
    """Fold one step's partial into the running state, as in [6D-CP].

    m_new = max(m, m_step); alpha = exp(m - m_new); beta = exp(m_step - m_new);
    l = alpha * l + beta * l_step; O = alpha * O + beta * O_step; m = m_new.
    (The extracted listing lost its multiplication signs; they are restored.)
    ``o`` has one more trailing axis (D) than ``m`` and ``l``.
    """
    m_new = np.maximum(m, m_step)
    alpha = _exp_diff(m, m_new)
    beta = _exp_diff(m_step, m_new)
    l_new = alpha * l + beta * l_step
    o_new = alpha[..., None] * o + beta[..., None] * o_step
    return o_new, m_new, l_new


def finalize(o, m, l):
    """``O / l`` (the listing's return value) and ``LSE = m + ln l``.

    l = 0 (nothing visible) gives O = 0 and LSE = -inf.
    """
    pos = l > 0
    safe_l = np.where(pos, l, 1.0)
    out = np.where(pos[..., None], o / safe_l[..., None], 0.0)
    lse = np.where(pos, m + np.log(safe_l), NEG_INF)
    return out, lse


def ring_attention(q, k, v, cu_seqlens, cp_sizes, scale, causal=True,
                   num_steps=None):
    """The ring loop of [6D-CP], literally, for every sample of a THD batch.

    Sample b is split into ``cp_sizes[b]`` chunks (:func:`chunk_bounds`); rank
    i holds Q chunk i.  It starts from O = 0, m = -inf, l = 0 and for
    ``step = 0 .. c-1`` attends to the KV chunk it holds at that step,
    ``j = (i - step) mod c``, folding each block into (O, m, l) with
    :func:`merge_step`.  Positions are global within the sample, so the causal
    mask hides whole chunks j > i and half of the diagonal chunk.

    Returns ``(out [T, H, D], lse [T, H])``; when ``num_steps`` is given it
    also returns the per-step partials ``(o_steps [S, T, H, D],
    m_steps [S, T, H], l_steps [S, T, H])`` with ``S = num_steps >= max c``.
    Slot s of token t holds the step-s partial of t's rank; steps that do not
    exist for a sample (s >= c) hold the empty partial (0, -inf, 0).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    cu = [int(x) for x in cu_seqlens]
    T, H, D = q.shape
    out = np.zeros((T, H, D))
    lse = np.full((T, H), NEG_INF)
    if num_steps is not None:
        S = int(num_steps)
        o_steps = np.zeros((S, T, H, D))
        m_steps = np.full((S, T, H), NEG_INF)
        l_steps = np.zeros((S, T, H))
    for b in range(len(cu) - 1):
        s0 = cu[b]
        L = cu[b + 1] - s0
        c = int(cp_sizes[b])
        if num_steps is not None and c > S:
            raise ValueError("num_steps smaller than a sample's CP size")
        bounds = chunk_bounds(L, c)
        for i in range(c):
            qa, qb_ = bounds[i]
            if qb_ <= qa:
                continue
            q_pos = np.arange(qa, qb_)
            q_i = np.transpose(q[s0 + qa:s0 + qb_], (1, 0, 2))
            o_run = np.zeros((H, qb_ - qa, D))
            m_run = np.full((H, qb_ - qa), NEG_INF)
            l_run = np.zeros((H, qb_ - qa))
            for step in range(c):
                j = (i - step) % c
                ka, kb_ = bounds[j]
                k_pos = np.arange(ka, kb_)
                k_j = np.transpose(k[s0 + ka:s0 + kb_], (1, 0, 2))
                v_j = np.transpose(v[s0 + ka:s0 + kb_], (1, 0, 2))
                o_s, m_s, l_s = block_attention(q_i, k_j, v_j, q_pos, k_pos,
                                                scale, causal)
                if num_steps is not None:
                    o_steps[step, s0 + qa:s0 + qb_] = np.transpose(o_s, (1, 0, 2))
                    m_steps[step, s0 + qa:s0 + qb_] = m_s.T
                    l_steps[step, s0 + qa:s0 + qb_] = l_s.T
                o_run, m_run, l_run = merge_step(o_run, m_run, l_run,
                                                 o_s, m_s, l_s)
            o_fin, lse_fin = finalize(o_run, m_run, l_run)
            out[s0 + qa:s0 + qb_] = np.transpose(o_fin, (1, 0, 2))
            lse[s0 + qa:s0 + qb_] = lse_fin.T
    if num_steps is not None:
        return out, lse, (o_steps, m_steps, l_steps)
    return out, lse


# ---------------------------------------------------------------------------
# (c3) Merge of stored partials (the unfused path).
# ---------------------------------------------------------------------------

def merge_partials(o_steps, m_steps, l_steps):
    """Fold S stored partials in step order 0..S-1 with the [6D-CP] merge.

    ``o_steps [S, ..., D]``, ``m_steps`` and ``l_steps [S, ...]``.  Returns the
    merged ``(O / l, m, l)``; O / l is 0 where l = 0.
    """
    o_steps = np.asarray(o_steps, dtype=np.float64)
    m_steps = np.asarray(m_steps, dtype=np.float64)
    l_steps = np.asarray(l_steps, dtype=np.float64)
    o = np.zeros(o_steps.shape[1:])
    m = np.full(m_steps.shape[1:], NEG_INF)
    l = np.zeros(l_steps.shape[1:])
    for s in range(o_steps.shape[0]):
        o, m, l = merge_step(o, m, l, o_steps[s], m_steps[s], l_steps[s])
    pos = l > 0
    out = np.where(pos[..., None], o / np.where(pos, l, 1.0)[..., None], 0.0)
    return out, m, l
