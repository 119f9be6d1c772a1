"""Shared helpers for the GPU parity tests (tolerances, batch construction)."""

import math

import numpy as np
import torch

from long_context_gb300 import workloads

# Tolerances for bf16 inputs with fp32 accumulation, against the float64 oracle.
O_ATOL = 2e-2          # attention output, max abs
LSE_RTOL = 1e-3        # |dLSE| <= 1e-3 * max(1, |LSE|)
MERGE_RTOL = 1e-5      # fp32 merge output O / l, relative to its row's max |O / l|
MERGE_L_RTOL = 1e-5    # fp32 merge output l, relative


def check_merge_o(got, ref, what=""):
    """Assert the fp32 merge gate on O / l; returns the largest error relative
    to its row's max |O / l|.

    A row is one (token, head) vector of D values.  The merge runs in fp32, so
    every element must agree with the oracle to within MERGE_RTOL of the
    largest magnitude in its row (fp32 rounding of the fold, a few ulp, is
    ~1e-7 of it); an O path that went through bf16 anywhere (relative
    rounding up to 2^-9) misses this by two orders of magnitude.  Rows whose
    reference is all zero (nothing visible) must be exactly zero."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, what
    assert np.all(np.isfinite(got)), "%s: non-finite merge output" % what
    if ref.size == 0:
        return 0.0
    d = ref.shape[-1]
    g2 = got.reshape(-1, d)
    r2 = ref.reshape(-1, d)
    row_max = np.max(np.abs(r2), axis=1)
    zero = row_max == 0
    assert np.all(g2[zero] == 0), "%s: rows with nothing visible must be zero" % what
    rel = np.abs(g2[~zero] - r2[~zero]) / row_max[~zero][:, None]
    worst = float(np.max(rel)) if rel.size else 0.0
    assert worst <= MERGE_RTOL, "%s: max |dO| / row max |O| = %g" % (what, worst)
    return worst


def check_attention(out, lse, ref_o, ref_lse, what=""):
    """Assert the attention tolerances; returns (max |dO|, max scaled |dLSE|)."""
    out = np.asarray(out, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert np.all(np.isfinite(out)), "%s: non-finite output" % what
    do = float(np.max(np.abs(out - ref_o))) if out.size else 0.0
    dl = float(np.max(np.abs(lse - ref_lse) / np.maximum(1.0, np.abs(ref_lse)))) if lse.size else 0.0
    assert do <= O_ATOL, "%s: max |dO| = %g" % (what, do)
    assert dl <= LSE_RTOL, "%s: max rel |dLSE| = %g" % (what, dl)
    return do, dl


# Gradients (bf16 outputs of cpattn_bwd) against the float64 oracle.  Rounding
# points of the GPU path: P and dS are rounded to bf16 (relative 2^-9) before
# their products, O (bf16) enters D = rowsum(dO * O), and each gradient is
# rounded to bf16 (relative 2^-9).  A rounding error of relative size 2^-9 on
# each of the N terms of a gradient sum adds up like a random walk to about
# 2^-9 * sqrt(sum of squared terms) -- a fraction of a percent of the RMS of
# the gradient -- so:
#   * RMS(error) <= GRAD_RMS_RTOL * RMS(gradient) over each tensor (a dropped
#     or wrongly scaled term gives errors of the order of the gradient itself);
#   * every element: |error| <= GRAD_RTOL * |g| + GRAD_ATOL_RMS * RMS(gradient)
#     (the first term bounds the output rounding with 8x margin, the second the
#     tail of the summed rounding errors over ~1e5-1e6 elements; a wrong mask
#     on a row gives errors of the order of RMS(gradient) there).
GRAD_RMS_RTOL = 1e-2
GRAD_RTOL = 2 ** -6
GRAD_ATOL_RMS = 0.15


def check_grad(got, ref, what=""):
    """Assert the gradient tolerances; returns (RMS err / RMS ref, worst ratio)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), "%s: non-finite gradient" % what
    if ref.size == 0:
        return 0.0, 0.0
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    rel_rms = float(np.sqrt(np.mean(err ** 2))) / max(rms, 1e-30)
    worst = float(np.max(err / (GRAD_RTOL * np.abs(ref) + GRAD_ATOL_RMS * rms + 1e-30)))
    assert rel_rms <= GRAD_RMS_RTOL, "%s: RMS error / RMS = %g" % (what, rel_rms)
    assert worst <= 1.0, "%s: worst elementwise error ratio %g" % (what, worst)
    return rel_rms, worst


def make_batch(lengths, H, D, seed, std=1.0, device="cuda"):
    """Seeded THD batch: CPU bf16 q/k/v, int32 cu_seqlens, and GPU copies."""
    T = int(sum(lengths))
    q, k, v = workloads.qkv(T, H, D, seed, std)
    cu = workloads.cu_seqlens(lengths)
    g = dict(q=q.to(device), k=k.to(device), v=v.to(device),
             cu=torch.from_numpy(cu).to(device))
    return (q, k, v, cu), g


def sample_tokens(cu, n_random, seed, extra=()):
    """Token indices to check at full size: the first, second, last and last-but-
    one token of every sample, tile and chunk edges near them, plus random ones."""
    rng = np.random.default_rng(seed)
    cu = [int(x) for x in cu]
    T = cu[-1]
    toks = set(int(t) for t in extra if 0 <= t < T)
    for b in range(len(cu) - 1):
        s0, s1 = cu[b], cu[b + 1]
        for t in (s0, s0 + 1, s0 + 127, s0 + 128, s1 - 2, s1 - 1):
            if s0 <= t < s1:
                toks.add(t)
    if T > 0:
        toks.update(int(t) for t in rng.integers(0, T, n_random))
    return sorted(toks)


def chunk_edge_tokens(cu, cps):
    """Token indices at the ring-chunk edges of every sample with CP > 1: for
    each boundary between chunk j-1 and chunk j (chunks of ceil(L / c)
    tokens), the rows around it and one and two 128-row tiles past it."""
    cu = [int(x) for x in cu]
    toks = set()
    for b, c in enumerate(cps):
        c = int(c)
        s0, s1 = cu[b], cu[b + 1]
        L = s1 - s0
        if c <= 1 or L == 0:
            continue
        chunk = -(-L // c)
        for j in range(1, c + 1):
            e = min(j * chunk, L)
            for d in (-129, -128, -1, 0, 1, 127, 128, 255):
                if 0 <= e + d < L:
                    toks.add(s0 + e + d)
    return sorted(toks)


def default_scale(D):
    return 1.0 / math.sqrt(D)
