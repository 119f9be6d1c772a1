"""GPU parity of cpattn_fwd / cpattn_fwd_partials against the float64 oracle.

Every call goes through the C ABI (libcpattn.so via the ctypes binding).
Small cases compare every output element; the full-size workloads compare
sampled rows that the oracle computes one by one.
"""

import numpy as np
import pytest
import torch

from helpers import (O_ATOL, check_attention, check_merge_o, chunk_edge_tokens,
                     default_scale, make_batch, sample_tokens)
from long_context_gb300 import workloads
from oracle import attention as oa
from oracle import planner as op

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_gb300 import build as lib_build
    lib_build.build()
    from long_context_gb300 import cpattn
    return cpattn


def _run(cp, g, lengths, cps, H, D, causal, mode, scale):
    cps_t = None if cps is None else torch.tensor(cps, dtype=torch.int32, device="cuda")
    max_cp = 1 if cps is None else max(cps) if len(cps) else 1
    T = int(sum(lengths))
    # Guard bands around the outputs catch stray writes.
    guard = 64
    out_buf = torch.full((T + 2 * guard, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse_buf = torch.full((T + 2 * guard, H), float("nan"), dtype=torch.float32, device="cuda")
    out = out_buf[guard:guard + T]
    lse = lse_buf[guard:guard + T]
    ws = cp.alloc_workspace(T, len(lengths), H, D, max_cp, mode)
    cp.fwd(g["q"], g["k"], g["v"], g["cu"], cps_t, max_seqlen=max(max(lengths), 1),
           max_cp=max_cp, softmax_scale=scale, causal=causal, mode=mode, out=out, lse=lse,
           workspace=ws)
    assert cp.poll_error(ws) == cp.OK
    assert torch.isnan(out_buf[:guard].float()).all() and torch.isnan(out_buf[guard + T:].float()).all()
    assert torch.isnan(lse_buf[:guard]).all() and torch.isnan(lse_buf[guard + T:]).all()
    return out.float().cpu().numpy(), lse.cpu().numpy()


# ----------------------------------------------------------------- small --

@pytest.mark.parametrize("mode", [0, 1])
def test_tiny_ring_cp2(cp, mode):
    """One causal 1024-token sequence at CP=2, H=4, D=64 (full comparison)."""
    w = workloads.WORKLOADS["tiny"]
    (q, k, v, cu), g = make_batch(w["lengths"], w["H"], w["D"], seed=0)
    scale = default_scale(w["D"])
    out, lse = _run(cp, g, w["lengths"], [w["cp"]], w["H"], w["D"], True, mode, scale)
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    ref_o, ref_lse = oa.ring_attention(qf, kf, vf, cu, [w["cp"]], scale)
    full_o, full_lse = oa.full_attention(qf, kf, vf, cu, scale)
    assert np.max(np.abs(ref_o - full_o)) < 1e-12
    check_attention(out, lse, ref_o, ref_lse, "tiny mode %d" % mode)


RAGGED = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 511, 513]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("mode", [0, 1])
def test_ragged_lengths_all_cp(cp, D, causal, mode):
    lengths = RAGGED
    cps = [[1, 2, 4, 8][i % 4] for i in range(len(lengths))]
    H = 3
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=11)
    scale = default_scale(D)
    out, lse = _run(cp, g, lengths, cps, H, D, causal, mode, scale)
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    ref_o, ref_lse = oa.full_attention(qf, kf, vf, cu, scale, causal=causal)
    check_attention(out, lse, ref_o, ref_lse, "ragged D=%d causal=%s mode=%d" % (D, causal, mode))


@pytest.mark.parametrize("mode", [0, 1])
def test_empty_samples(cp, mode):
    lengths = [0, 5, 0, 130, 0, 1]
    cps = [2, 4, 1, 2, 8, 2]
    H, D = 2, 128
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=3)
    out, lse = _run(cp, g, lengths, cps, H, D, True, mode, 0.2)
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    ref_o, ref_lse = oa.full_attention(qf, kf, vf, cu, 0.2)
    check_attention(out, lse, ref_o, ref_lse, "empty samples")


@pytest.mark.parametrize("n_seqs", [2048, 2500])
def test_many_samples(cp, n_seqs):
    """Thousands of short samples (empty ones included) at CP sizes 1-8 in
    one batch: the schedule kernel's sort and table fill over many samples,
    every output element against the oracle."""
    rng = np.random.default_rng(n_seqs)
    lengths = [int(x) for x in rng.integers(0, 40, n_seqs)]
    cps = [int(x) for x in rng.choice([1, 2, 4, 8], n_seqs)]
    H, D = 2, 64
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=n_seqs)
    scale = default_scale(D)
    out, lse = _run(cp, g, lengths, cps, H, D, True, 0, scale)
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    ref_o, ref_lse = oa.full_attention(qf, kf, vf, cu, scale)
    check_attention(out, lse, ref_o, ref_lse, "%d samples" % n_seqs)


def test_zero_tokens(cp):
    H, D = 2, 64
    q = torch.empty((0, H, D), dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    out, lse = cp.fwd(q, q, q, cu, None, max_seqlen=1, max_cp=1)
    assert out.shape == (0, H, D)


def test_large_scores_and_rescale(cp):
    """Scores spread over many powers of two exercise the running-max update.
    The spread comes from the softmax scale (as if Q and K had std 2.5); V
    stays N(0, 1), the distribution the output tolerance is stated for."""
    lengths = [700, 1500]
    H, D = 2, 128
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=5)
    scale = 6.25 * default_scale(D)
    out, lse = _run(cp, g, lengths, [2, 4], H, D, True, 0, scale)
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    ref_o, ref_lse = oa.full_attention(qf, kf, vf, cu, scale)
    check_attention(out, lse, ref_o, ref_lse, "large scores")


@pytest.mark.parametrize("causal", [True, False])
def test_late_dominant_keys(cp, causal):
    """Keys from token 512 on have 6x larger components, so for every row that
    sees them the scores jump by many powers of two after the first KV tiles:
    the running max found on the early tiles is far too low for the late ones
    and those tiles must be taken again with their own max."""
    lengths = [1000, 900]
    H, D = 2, 128
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=21)
    k = k.clone()
    for b in range(len(lengths)):
        k[int(cu[b]) + 512:int(cu[b + 1])] *= 6
    g["k"] = k.to("cuda")
    scale = default_scale(D)
    out, lse = _run(cp, g, lengths, [1, 2], H, D, causal, 0, scale)
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    ref_o, ref_lse = oa.full_attention(qf, kf, vf, cu, scale, causal=causal)
    check_attention(out, lse, ref_o, ref_lse, "late dominant keys")


def test_cp_invariance(cp):
    """Only the CP assignment changes: static CP 1/2/4/8 and the dynamic plan
    all agree with the oracle (and the dynamic plan matches the oracle's)."""
    lengths = [300, 1000, 77, 2048, 513]
    H, D = 2, 128
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=8)
    scale = default_scale(D)
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    ref_o, ref_lse = oa.full_attention(qf, kf, vf, cu, scale)
    plan_c = cp.plan(lengths, 4, 600, 4)
    plan_o = op.plan(lengths, 4, 600, 4)
    assert list(plan_c["cp_size"]) == plan_o["cp_size"]
    outs = []
    for cps in ([1] * 5, [2] * 5, [4] * 5, [8] * 5, [int(x) for x in plan_c["cp_size"]]):
        out, lse = _run(cp, g, lengths, cps, H, D, True, 0, scale)
        check_attention(out, lse, ref_o, ref_lse, "cp %s" % cps)
        outs.append(out)
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= 2 * O_ATOL


def test_deterministic(cp):
    lengths = [1000, 333]
    H, D = 4, 128
    (_, _, _, _), g = make_batch(lengths, H, D, seed=9)
    cps = torch.tensor([4, 2], dtype=torch.int32, device="cuda")
    a, la = cp.fwd(g["q"], g["k"], g["v"], g["cu"], cps, max_seqlen=1000, max_cp=4)
    b, lb = cp.fwd(g["q"], g["k"], g["v"], g["cu"], cps, max_seqlen=1000, max_cp=4)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_device_side_validation(cp):
    """Bad cu_seqlens or CP sizes are caught by the kernels: the error word is
    set and no output is written."""
    H, D = 2, 64
    (_, _, _, _), g = make_batch([100, 50], H, D, seed=1)
    out = torch.full((150, H, D), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((150, H), 7.0, dtype=torch.float32, device="cuda")
    ws = cp.alloc_workspace(150, 2, H, D, 2)
    bad_cu = torch.tensor([0, 120, 100], dtype=torch.int32, device="cuda")
    cp.fwd(g["q"], g["k"], g["v"], bad_cu, None, max_seqlen=200, max_cp=2, out=out, lse=lse,
           workspace=ws)
    assert cp.poll_error(ws) == cp.ERR_INVALID_ARG
    bad_cp = torch.tensor([4, 1], dtype=torch.int32, device="cuda")
    cp.fwd(g["q"], g["k"], g["v"], g["cu"], bad_cp, max_seqlen=200, max_cp=2, out=out, lse=lse,
           workspace=ws)
    assert cp.poll_error(ws) == cp.ERR_INVALID_ARG
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())
    # The same workspace is usable again afterwards.
    cp.fwd(g["q"], g["k"], g["v"], g["cu"], None, max_seqlen=200, max_cp=2, out=out, lse=lse,
           workspace=ws)
    assert cp.poll_error(ws) == cp.OK


# -------------------------------------------------------------- partials --

@pytest.mark.parametrize("causal", [True, False])
def test_partials_match_oracle_ring_steps(cp, causal):
    lengths = [9, 300, 3, 1000]
    cps = [4, 2, 8, 4]
    S = 8
    H, D = 2, 128
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=4)
    scale = 0.09
    cps_t = torch.tensor(cps, dtype=torch.int32, device="cuda")
    o, m, l = cp.fwd_partials(g["q"], g["k"], g["v"], g["cu"], cps_t, max_seqlen=1000, max_cp=8,
                              num_steps=S, softmax_scale=scale, causal=causal)
    o, m, l = (x.cpu().numpy().astype(np.float64) for x in (o, m, l))
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    _, _, (ro, rm, rl) = oa.ring_attention(qf, kf, vf, cu, cps, scale, causal=causal, num_steps=S)
    empty = rl == 0
    # Steps that see nothing are exactly the empty partial.
    assert np.array_equal(l == 0, empty)
    assert np.all(np.isneginf(m[empty])) and np.all(o[empty] == 0)
    # Elsewhere compare what does not depend on the reference value chosen
    # for m_step: O_step / l_step and m_step + ln l_step.
    nz = ~empty
    on = o[nz] / l[nz][:, None]
    ron = ro[nz] / rl[nz][:, None]
    assert np.max(np.abs(on - ron)) <= O_ATOL
    lse_s = m[nz] + np.log(l[nz])
    rlse_s = rm[nz] + np.log(rl[nz])
    assert np.max(np.abs(lse_s - rlse_s) / np.maximum(1, np.abs(rlse_s))) <= 1e-3
    # Folding them with the library's merge gives the attention result; the
    # fold itself is fp32 and is held to the fp32 merge gate against the
    # oracle's fold of the same partials.
    mo, mm, ml = cp.merge(*(torch.from_numpy(x.astype(np.float32)).cuda() for x in (o, m, l)))
    fo, _, _ = oa.merge_partials(o.astype(np.float32), m.astype(np.float32),
                                 l.astype(np.float32))
    check_merge_o(mo.cpu().numpy(), fo, "partials fold")
    ref_o, ref_lse = oa.full_attention(qf, kf, vf, cu, scale, causal=causal)
    check_attention(mo.cpu().numpy(), (mm + torch.log(ml)).cpu().numpy(), ref_o, ref_lse,
                    "partials merged")


# ------------------------------------------------------------ full sizes --

# Seed 0 plans every sample at CP 1; seed 1 has two samples at CP 2 (4112
# and 4471 tokens) and seed 2 one at CP 4 (10935 tokens), so the ring steps
# run at the full size of the workload too.
PACKED16K_CPS = {0: [1, 1, 1, 1, 1, 1, 1], 1: [1, 2, 1, 1, 2, 1], 2: [1, 1, 1, 1, 4, 1]}


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("mode", [0, 1])
def test_packed16k_workload(cp, mode, seed):
    """16,384-token packed THD batch at world 4, limit 4096, dynamic CP."""
    w = workloads.WORKLOADS["packed16k"]
    lengths = workloads.packed_lengths(seed, w["budget"])
    plan_c = cp.plan(lengths, w["world"], w["limit"], w["max_cp"])
    plan_o = op.plan(lengths, w["world"], w["limit"], w["max_cp"])
    assert list(plan_c["cp_size"]) == plan_o["cp_size"]
    cps = [int(x) for x in plan_c["cp_size"]]
    assert cps == PACKED16K_CPS[seed]
    H, D = w["H"], w["D"]
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=seed)
    scale = default_scale(D)
    out, lse = _run(cp, g, lengths, cps, H, D, True, mode, scale)
    toks = sample_tokens(cu, 48, seed=seed, extra=chunk_edge_tokens(cu, cps))
    ref_o, ref_lse = oa.attention_rows(q, k, v, cu, scale, toks)
    check_attention(out[toks], lse[toks], ref_o, ref_lse,
                    "packed16k seed %d mode %d" % (seed, mode))


@pytest.mark.parametrize("mode", [0, 1])
def test_long128k_workload(cp, mode):
    """One causal 131,072-token sequence at CP=4 (32K chunks), H=16, D=128."""
    w = workloads.WORKLOADS["long128k"]
    H, D = w["H"], w["D"]
    (q, k, v, cu), g = make_batch(w["lengths"], H, D, seed=0, std=w["std"])
    scale = default_scale(D)
    out, lse = _run(cp, g, w["lengths"], [w["cp"]], H, D, True, mode, scale)
    chunk = 32768
    edges = [j * chunk + d for j in range(4) for d in (-129, -128, -1, 0, 1, 127, 128, 255)]
    toks = sample_tokens(cu, 24, seed=1, extra=edges)
    ref_o, ref_lse = oa.attention_rows(q, k, v, cu, scale, toks)
    check_attention(out[toks], lse[toks], ref_o, ref_lse, "long128k mode %d" % mode)


def test_sweep256_workload(cp):
    """256 samples (256..32768 tokens), world 8, limit 4096: the planner's
    micro-batches run one after another as THD batches."""
    w = workloads.WORKLOADS["sweep256"]
    lengths = workloads.uniform_lengths(0, w["n"], w["lo"], w["hi"])
    plan_c = cp.plan(lengths, w["world"], w["limit"], w["max_cp"])
    plan_o = op.plan(lengths, w["world"], w["limit"], w["max_cp"])
    for key in ("cp_size", "micro_batch", "first_rank", "order"):
        assert list(plan_c[key]) == plan_o[key]
    H, D = w["H"], w["D"]
    scale = default_scale(D)
    rng = np.random.default_rng(0)
    n_mb = plan_c["num_micro_batches"]
    rows = 0
    for mb in range(n_mb):
        members = [b for b in range(len(lengths)) if plan_c["micro_batch"][b] == mb]
        lens = [lengths[b] for b in members]
        cps = [int(plan_c["cp_size"][b]) for b in members]
        # Each micro-batch draws its own tensors on the GPU (seed = 1000 + id);
        # the oracle reads back only the rows it checks.
        q, k, v = workloads.qkv_device(sum(lens), H, D, seed=1000 + mb)
        cu = workloads.cu_seqlens(lens)
        cu_t = torch.from_numpy(cu).cuda()
        cps_t = torch.tensor(cps, dtype=torch.int32, device="cuda")
        out, lse = cp.fwd(q, k, v, cu_t, cps_t, max_seqlen=max(lens),
                          max_cp=w["max_cp"], softmax_scale=scale)
        # Every micro-batch: the first and last row of each sample, the rows
        # around one chunk edge of each CP > 1 sample, and random rows, at
        # least 16 in all.
        edge = {}
        for b in range(len(lens)):
            s0, s1 = int(cu[b]), int(cu[b + 1])
            edge[s0] = edge[s1 - 1] = True
            if cps[b] > 1:
                chunk = -(-lens[b] // cps[b])
                j = int(rng.integers(1, cps[b]))
                for d in (-1, 0, 128):
                    t = s0 + min(j * chunk, lens[b]) + d
                    if s0 <= t < s1:
                        edge[t] = True
        toks = set(edge) | set(int(t) for t in rng.integers(0, int(cu[-1]), 8))
        while len(toks) < 16:
            toks.add(int(rng.integers(0, int(cu[-1]))))
        toks = sorted(toks)
        ref_o, ref_lse = oa.attention_rows(q, k, v, cu, scale, toks)
        check_attention(out[toks].float().cpu().numpy(), lse[toks].cpu().numpy(),
                        ref_o, ref_lse, "sweep256 mb %d" % mb)
        rows += len(toks)
    assert rows >= 16 * n_mb
