"""GPU parity of cpattn_bwd (dQ, dK, dV) against the float64 backward oracle.

The GPU backward takes the GPU forward's O and LSE (the product path: forward
then backward); the oracle computes everything from Q, K, V and dO alone.
Small cases and the full-size packed 16K batch compare every element; the
131,072-token sequence compares sampled dQ rows (computed one by one) and the
identities that hold at any size: per sample and head, sum_j dV_j = sum_i dO_i
and sum_j dK_j = 0.
"""

import numpy as np
import pytest
import torch

from helpers import check_grad, default_scale
from long_context_gb300 import workloads
from oracle import backward as ob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_gb300 import build as lib_build
    lib_build.build()
    from long_context_gb300 import cpattn
    return cpattn


def _inputs(lengths, H, D, seed):
    T = int(sum(lengths))
    q, k, v = workloads.qkv(T, H, D, seed)
    g = torch.Generator().manual_seed(seed + 1000)
    do = torch.randn((T, H, D), generator=g).to(torch.bfloat16)
    cu = workloads.cu_seqlens(lengths)
    return q, k, v, do, cu


def _fwd_bwd(cp, q, k, v, do, cu, cps, causal, scale, guard=64):
    dev = "cuda"
    T, H, D = q.shape
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    cud = torch.from_numpy(cu).to(dev)
    cpd = None if cps is None else torch.tensor(cps, dtype=torch.int32, device=dev)
    lengths = np.diff(cu)
    max_seqlen = int(max(lengths.max() if len(lengths) else 1, 1))
    max_cp = 1 if cps is None else max(cps)
    out, lse = cp.fwd(qd, kd, vd, cud, cpd, max_seqlen=max_seqlen, max_cp=max_cp,
                      softmax_scale=scale, causal=causal)
    # Guard bands around the gradients catch stray writes.
    bufs = [torch.full((T + 2 * guard, H, D), float("nan"), dtype=torch.bfloat16, device=dev)
            for _ in range(3)]
    grads = [b[guard:guard + T] for b in bufs]
    ws = cp.alloc_bwd_workspace(T, len(cu) - 1, H, D, max_cp, dev)
    cp.bwd(qd, kd, vd, out, dod, lse, cud, cpd, max_seqlen=max_seqlen, max_cp=max_cp,
           softmax_scale=scale, causal=causal, dq=grads[0], dk=grads[1], dv=grads[2],
           workspace=ws)
    assert cp.poll_error(ws) == cp.OK
    for b in bufs:
        assert torch.isnan(b[:guard].float()).all() and torch.isnan(b[guard + T:].float()).all()
    return [g.float().cpu().numpy() for g in grads]


CASES = [
    # lengths, H, D, causal, cp sizes
    ([300], 2, 128, True, [1]),
    ([1000, 300, 77, 513], 2, 128, True, [1, 2, 4, 1]),
    ([700, 129], 2, 128, False, [2, 1]),
    ([640, 64, 1], 2, 64, True, [2, 1, 1]),
    ([1, 127, 128, 129, 255, 256, 257], 2, 128, True, [1, 1, 2, 1, 2, 4, 2]),
    ([3, 5, 200], 3, 64, False, [4, 8, 2]),
]


@pytest.mark.parametrize("lengths,H,D,causal,cps", CASES)
def test_backward_matches_oracle(cp, lengths, H, D, causal, cps):
    q, k, v, do, cu = _inputs(lengths, H, D, seed=sum(lengths) % 97)
    scale = default_scale(D)
    dq, dk, dv = _fwd_bwd(cp, q, k, v, do, cu, cps, causal, scale)
    ref = ob.full_attention_backward(*(workloads.to_f64(x) for x in (q, k, v, do)), cu, scale,
                                     causal=causal)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_grad(got, ref[name], "%s %s" % (name, lengths))


def test_backward_cp_invariance_and_determinism(cp):
    """Only the CP split changes: every split agrees with the oracle; the same
    call twice gives the same bits."""
    lengths, H, D = [900, 260, 33], 2, 128
    q, k, v, do, cu = _inputs(lengths, H, D, seed=3)
    scale = default_scale(D)
    ref = ob.full_attention_backward(*(workloads.to_f64(x) for x in (q, k, v, do)), cu, scale)
    for cps in ([1, 1, 1], [2, 2, 2], [4, 4, 4], [8, 8, 8], [4, 2, 1]):
        grads = _fwd_bwd(cp, q, k, v, do, cu, cps, True, scale)
        for name, got in zip(("dq", "dk", "dv"), grads):
            check_grad(got, ref[name], "%s cp %s" % (name, cps))
    a = _fwd_bwd(cp, q, k, v, do, cu, [2, 1, 1], True, scale)
    b = _fwd_bwd(cp, q, k, v, do, cu, [2, 1, 1], True, scale)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_backward_empty_batch(cp):
    dev = "cuda"
    H, D = 2, 128
    z = torch.zeros((0, H, D), dtype=torch.bfloat16, device=dev)
    cu = torch.zeros(1, dtype=torch.int32, device=dev)
    lse = torch.zeros((0, H), dtype=torch.float32, device=dev)
    ws = cp.alloc_bwd_workspace(0, 0, H, D, 1, dev)
    dq, dk, dv = cp.bwd(z, z, z, z, z, lse, cu, None, max_seqlen=1, max_cp=1, workspace=ws)
    assert cp.poll_error(ws) == cp.OK and dq.numel() == 0


@pytest.mark.parametrize("seed,heads", [(0, None), (1, (0, 13, 31))])
def test_backward_packed16k_every_element(cp, seed, heads):
    """The packed 16K batch (H=32, D=128, CP from the plan: all 1 for seed 0,
    two samples at CP 2 for seed 1) at full size: every element of dQ, dK and
    dV against the oracle's full backward, taken one head at a time (the
    oracle holds L^2 scores per head; every head for seed 0, three for seed 1,
    whose heads differ only in their data), and per (sample, head)
    sum_j dV_j = sum_i dO_i, sum_j dK_j = 0."""
    w = workloads.WORKLOADS["packed16k"]
    H, D = w["H"], w["D"]
    lengths = workloads.packed_lengths(seed, w["budget"])
    plan = cp.plan(lengths, w["world"], w["limit"], w["max_cp"])
    cps = [int(c) for c in plan["cp_size"]]
    q, k, v, do, cu = _inputs(lengths, H, D, seed=seed)
    scale = default_scale(D)
    dq, dk, dv = _fwd_bwd(cp, q, k, v, do, cu, cps, True, scale)
    qf, kf, vf, dof = (workloads.to_f64(x) for x in (q, k, v, do))
    for h in (range(H) if heads is None else heads):
        sl = slice(h, h + 1)
        ref = ob.full_attention_backward(qf[:, sl], kf[:, sl], vf[:, sl], dof[:, sl], cu, scale)
        for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
            check_grad(got[:, sl], ref[name], "seed %d head %d %s" % (seed, h, name))
    for b in range(len(lengths)):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        sum_dv = dv[s0:s1].astype(np.float64).sum(0)
        want = dof[s0:s1].sum(0)
        scale_dv = np.sqrt((dv[s0:s1].astype(np.float64) ** 2).sum(0)) + 1e-30
        assert np.max(np.abs(sum_dv - want) / scale_dv) < 0.05, b
        sum_dk = dk[s0:s1].astype(np.float64).sum(0)
        scale_dk = np.sqrt((dk[s0:s1].astype(np.float64) ** 2).sum(0)) + 1e-30
        assert np.max(np.abs(sum_dk) / scale_dk) < 0.05, b


def test_backward_long128k_rows_and_identities(cp):
    """The 131,072-token sequence at CP 4 (H=16, D=128, N(0, 0.5^2)): the
    size and launch configuration the benchmark times.  dQ rows at the chunk
    edges and at random positions against the oracle (each row computed on
    its own), and per head sum_j dV_j = sum_i dO_i, sum_j dK_j = 0."""
    w = workloads.WORKLOADS["long128k"]
    H, D, L, c = w["H"], w["D"], w["lengths"][0], w["cp"]
    q, k, v = workloads.qkv(L, H, D, 0, std=w["std"])
    g = torch.Generator().manual_seed(1000)
    do = torch.randn((L, H, D), generator=g).to(torch.bfloat16)
    cu = workloads.cu_seqlens([L])
    scale = default_scale(D)
    dq, dk, dv = _fwd_bwd(cp, q, k, v, do, cu, [c], True, scale)
    chunk = L // c
    toks = [0, 1, 127, 128] + [j * chunk + d for j in range(1, c) for d in (-1, 0)] + [L - 1]
    toks += [int(t) for t in np.random.default_rng(7).integers(0, L, 3)]
    ref_dq, _, _ = ob.backward_rows(q, k, v, do, cu, scale, toks)
    check_grad(dq[toks], ref_dq, "long128k dq rows")
    dof = do.float().numpy().astype(np.float64)
    sum_dv = dv.astype(np.float64).sum(0)
    scale_dv = np.sqrt((dv.astype(np.float64) ** 2).sum(0)) + 1e-30
    assert np.max(np.abs(sum_dv - dof.sum(0)) / scale_dv) < 0.05
    sum_dk = dk.astype(np.float64).sum(0)
    scale_dk = np.sqrt((dk.astype(np.float64) ** 2).sum(0)) + 1e-30
    assert np.max(np.abs(sum_dk) / scale_dk) < 0.05
