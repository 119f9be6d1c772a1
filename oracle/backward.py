"""Oracle attention backward: float64, CPU, NumPy.  TEST INFRASTRUCTURE ONLY.

The pages name the backward pass as the step that follows the forward in
training ("20-Megatron-MCore-TP-PP-EP如何支撑MoE", section 4: an update runs
``forward_backward_batch`` per micro-batch; "VeRL Backend Parallelism",
MindSpeed-MM recipe section: ``loss.backward()``) but print no formula for it.
The plainest reading is therefore the exact derivative of the forward's own
definition ([6D-CP], section 六: every query attends to every visible key):

    s_ij = scale * <q_i, k_j>        (visible pairs only)
    P_ij = exp(s_ij - LSE_i)         (the row softmax)
    o_i  = sum_j P_ij v_j

For an upstream gradient dO (the gradient of the loss with respect to O),
calculus gives, per sample and head:

    dV_j  = sum_i P_ij dO_i
    dP_ij = <dO_i, v_j>
    D_i   = sum_j P_ij dP_ij  (= <dO_i, o_i>)
    dS_ij = P_ij (dP_ij - D_i)
    dQ_i  = scale * sum_j dS_ij k_j
    dK_j  = scale * sum_i dS_ij q_i

Masked pairs have P = 0 and contribute nothing.  The functions below write
this out in matrix form (a library matmul is the only primitive) and, for
the ring, as the sum over the same (Q chunk, KV chunk) blocks the forward
visits: the gradient of a sum of blocks is the sum of the blocks' gradients,
each block using the row statistics (LSE, D) of the whole row.

Shares no code with the CUDA path and imports nothing from it.
"""

from __future__ import annotations

import numpy as np

from .attention import NEG_INF, chunk_bounds, full_attention


def _sample_backward(qb, kb, vb, dob, scale, causal):
    """One sample, all heads at once.  ``qb, kb, vb, dob`` are ``[H, L, D]``
    float64.  Returns ``(dq, dk, dv, lse, delta)`` with ``[H, L, D]`` and
    ``[H, L]`` shapes."""
    H, L, _ = qb.shape
    s = scale * np.matmul(qb, np.transpose(kb, (0, 2, 1)))          # [H, L, L]
    if causal:
        vis = np.arange(L)[None, :] <= np.arange(L)[:, None]
        s = np.where(vis[None], s, NEG_INF)
    mx = s.max(axis=2, keepdims=True)
    lse = mx + np.log(np.exp(s - mx).sum(axis=2, keepdims=True))     # [H, L, 1]
    p = np.exp(s - lse)                                              # masked -> 0
    o = np.matmul(p, vb)
    dv = np.matmul(np.transpose(p, (0, 2, 1)), dob)
    dp = np.matmul(dob, np.transpose(vb, (0, 2, 1)))
    delta = (p * dp).sum(axis=2, keepdims=True)                      # [H, L, 1]
    ds = p * (dp - delta)
    dq = scale * np.matmul(ds, kb)
    dk = scale * np.matmul(np.transpose(ds, (0, 2, 1)), qb)
    return dq, dk, dv, lse[:, :, 0], delta[:, :, 0], o


def full_attention_backward(q, k, v, do, cu_seqlens, scale, causal=True):
    """Gradients of the full attention of every sample of a THD batch.

    ``q, k, v, do`` are ``[T, H, D]`` (anything convertible to float64).
    Returns ``dict(dq, dk, dv, lse, delta, out)``: the three gradients
    ``[T, H, D]``, the forward's ``LSE`` and ``D = rowsum(P * dP)`` (``[T, H]``),
    and the forward output ``O``.  Memory is ``H * L^2`` per sample: meant for
    the sizes the tests use.
    """
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    cu = [int(x) for x in cu_seqlens]
    T, H, D = q.shape
    res = {n: np.zeros((T, H, D)) for n in ("dq", "dk", "dv", "out")}
    res["lse"] = np.full((T, H), NEG_INF)
    res["delta"] = np.zeros((T, H))
    tr = lambda a: np.ascontiguousarray(np.transpose(a, (1, 0, 2)))  # noqa: E731
    for b in range(len(cu) - 1):
        s0, s1 = cu[b], cu[b + 1]
        if s1 <= s0:
            continue
        dq, dk, dv, lse, delta, o = _sample_backward(
            tr(q[s0:s1]), tr(k[s0:s1]), tr(v[s0:s1]), tr(do[s0:s1]), scale, causal)
        res["dq"][s0:s1] = tr(dq)
        res["dk"][s0:s1] = tr(dk)
        res["dv"][s0:s1] = tr(dv)
        res["out"][s0:s1] = tr(o)
        res["lse"][s0:s1] = lse.T
        res["delta"][s0:s1] = delta.T
    return res


def ring_attention_backward(q, k, v, do, cu_seqlens, cp_sizes, scale, causal=True):
    """The backward over the ring's blocks, literally.

    For every sample split into ``c`` chunks, rank i holds Q chunk i and at
    ring step s the KV chunk ``j = (i - s) mod c`` (as in the forward).  The
    row statistics ``LSE`` and ``D`` of each query row are those of the whole
    row (from the forward of the full row); with them each block's
    contribution is

        P  = exp(scale * Q_i K_j^T - LSE_i)     (visible pairs; else 0)
        dS = P * (dO_i V_j^T - D_i)
        dQ_i += scale * dS K_j,  dK_j += scale * dS^T Q_i,  dV_j += P^T dO_i

    and the gradients are the sums over all blocks, accumulated in ring order.
    """
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    cu = [int(x) for x in cu_seqlens]
    T, H, D = q.shape
    fwd, lse_all = full_attention(q, k, v, cu, scale, causal=causal)
    delta_all = (do * fwd).sum(axis=2)                               # [T, H]
    dq = np.zeros((T, H, D))
    dk = np.zeros((T, H, D))
    dv = np.zeros((T, H, D))
    for b in range(len(cu) - 1):
        s0, s1 = cu[b], cu[b + 1]
        L = s1 - s0
        if L <= 0:
            continue
        c = int(cp_sizes[b])
        bounds = chunk_bounds(L, c)
        for i in range(c):
            qa, qz = bounds[i]
            if qz <= qa:
                continue
            for step in range(c):
                j = (i - step) % c
                ka, kz = bounds[j]
                if kz <= ka:
                    continue
                qp = np.arange(qa, qz)
                kp = np.arange(ka, kz)
                for h in range(H):
                    qi = q[s0 + qa:s0 + qz, h]
                    kj = k[s0 + ka:s0 + kz, h]
                    vj = v[s0 + ka:s0 + kz, h]
                    doi = do[s0 + qa:s0 + qz, h]
                    s = scale * qi @ kj.T
                    if causal:
                        s = np.where(kp[None, :] <= qp[:, None], s, NEG_INF)
                    p = np.exp(s - lse_all[s0 + qa:s0 + qz, h][:, None])
                    ds = p * (doi @ vj.T - delta_all[s0 + qa:s0 + qz, h][:, None])
                    dq[s0 + qa:s0 + qz, h] += scale * ds @ kj
                    dk[s0 + ka:s0 + kz, h] += scale * ds.T @ qi
                    dv[s0 + ka:s0 + kz, h] += p.T @ doi
    return dict(dq=dq, dk=dk, dv=dv, lse=lse_all, delta=delta_all)


def backward_rows(q, k, v, do, cu_seqlens, scale, tokens, causal=True):
    """dQ and the row statistics for selected query tokens (every head), by the
    same definition.  Each row needs only its own visible keys, so this is
    usable at sizes where the full backward is out of reach.  Returns
    ``(dq [n, H, D], lse [n, H], delta [n, H])`` in the order of ``tokens``."""
    cu = np.asarray([int(x) for x in cu_seqlens], dtype=np.int64)
    H, D = q.shape[1], q.shape[2]
    tokens = [int(t) for t in tokens]
    dq = np.zeros((len(tokens), H, D))
    lse = np.zeros((len(tokens), H))
    delta = np.zeros((len(tokens), H))
    for n, t in enumerate(tokens):
        b = int(np.searchsorted(cu, t, side="right") - 1)
        s0, s1 = int(cu[b]), int(cu[b + 1])
        kend = t + 1 if causal else s1
        kt = np.transpose(_f64(k[s0:kend]), (1, 0, 2))               # [H, n, D]
        vt = np.transpose(_f64(v[s0:kend]), (1, 0, 2))
        qt = _f64(q[t])                                              # [H, D]
        dot = _f64(do[t])
        s = scale * np.matmul(kt, qt[:, :, None])[:, :, 0]           # [H, n]
        mx = s.max(axis=1, keepdims=True)
        row_lse = mx + np.log(np.exp(s - mx).sum(axis=1, keepdims=True))
        p = np.exp(s - row_lse)
        dp = np.matmul(vt, dot[:, :, None])[:, :, 0]                  # [H, n]
        dlt = (p * dp).sum(axis=1, keepdims=True)
        ds = p * (dp - dlt)
        dq[n] = scale * np.matmul(ds[:, None, :], kt)[:, 0, :]
        lse[n] = row_lse[:, 0]
        delta[n] = dlt[:, 0]
    return dq, lse, delta


def _f64(x):
    """Exact float64 copy of a NumPy array or a (CPU) torch tensor."""
    if hasattr(x, "detach"):
        import torch  # only when handed torch tensors
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)
