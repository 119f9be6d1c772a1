"""Seeded random sweep of the forward and backward against the float64 oracle.

Each case draws a small packed batch: 1-6 samples whose lengths mix empty
samples, lengths at the 128-row tile edges and arbitrary ones; CP sizes that
include non-powers of two (a chunk of ceil(L / c) rows, possibly empty);
H in {1, 2, 3}, D in {64, 128}, causal or not, a softmax scale and an input
spread drawn per case.  The forward runs in both kernel modes (merge folded
in, and per-step partials plus the merge kernel) and is compared element by
element with the oracle's full attention (the ring's result equals it, up to
rounding); the backward is compared element by element with the oracle's
full backward.  Guard bands around every output catch stray writes.  The
output is compared in units of the inputs' spread (the absolute bound on O
is set for unit spread); LSE and the gradients have relative bounds.
"""

import numpy as np
import pytest
import torch

from helpers import check_attention, check_grad, make_batch
from long_context_gb300 import workloads
from oracle import attention as oa
from oracle import backward as ob

pytestmark = pytest.mark.gpu

N_CASES = 16
EDGES = (1, 2, 127, 128, 129, 255, 256, 257, 383, 384, 385)


@pytest.fixture(scope="module")
def cp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_gb300 import build as lib_build
    lib_build.build()
    from long_context_gb300 import cpattn
    return cpattn


def _case(i):
    rng = np.random.default_rng(7000 + i)
    B = int(rng.integers(1, 7))
    lengths = []
    for _ in range(B):
        u = rng.random()
        if u < 0.15:
            lengths.append(0)
        elif u < 0.5:
            lengths.append(int(rng.choice(EDGES)))
        else:
            lengths.append(int(rng.integers(1, 600)))
    if sum(lengths) == 0:
        lengths[0] = int(rng.integers(1, 300))
    cps = [int(rng.choice([1, 2, 3, 4, 5, 8])) for _ in range(B)]
    H = int(rng.choice([1, 2, 3]))
    D = int(rng.choice([64, 128]))
    causal = bool(rng.random() < 0.7)
    scale = float(rng.uniform(0.04, 0.2))
    std = float(rng.choice([0.5, 1.0, 2.0]))
    return lengths, cps, H, D, causal, scale, std


def _guarded(shape, dtype, guard=64):
    buf = torch.full((shape[0] + 2 * guard,) + tuple(shape[1:]), float("nan"), dtype=dtype,
                     device="cuda")
    return buf, buf[guard:guard + shape[0]]


def _guard_intact(buf, T, guard=64):
    return bool(torch.isnan(buf[:guard].float()).all() and
                torch.isnan(buf[guard + T:].float()).all())


@pytest.mark.parametrize("i", range(N_CASES))
def test_fuzz_forward_and_backward(cp, i):
    lengths, cps, H, D, causal, scale, std = _case(i)
    what = "case %d: lengths %s cp %s H %d D %d causal %s" % (i, lengths, cps, H, D, causal)
    T = int(sum(lengths))
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=100 + i, std=std)
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    ref_o, ref_lse = oa.full_attention(qf, kf, vf, cu, scale, causal=causal)
    cps_t = torch.tensor(cps, dtype=torch.int32, device="cuda")
    max_seqlen, max_cp = max(max(lengths), 1), max(cps)

    outs = {}
    for mode in (cp.MODE_FUSED, cp.MODE_UNFUSED):
        out_buf, out = _guarded((T, H, D), torch.bfloat16)
        lse_buf, lse = _guarded((T, H), torch.float32)
        ws = cp.alloc_workspace(T, len(lengths), H, D, max_cp, mode)
        cp.fwd(g["q"], g["k"], g["v"], g["cu"], cps_t, max_seqlen=max_seqlen, max_cp=max_cp,
               softmax_scale=scale, causal=causal, mode=mode, out=out, lse=lse, workspace=ws)
        assert cp.poll_error(ws) == cp.OK, what
        assert _guard_intact(out_buf, T) and _guard_intact(lse_buf, T), what
        # O is a convex combination of V rows and every error term (bf16
        # rounding of P and of O) scales with them, so O is compared in units
        # of the inputs' spread: the absolute bound holds for unit spread.
        check_attention(out.float().cpu().numpy() / std, lse.cpu().numpy(), ref_o / std, ref_lse,
                        "%s mode %d" % (what, mode))
        outs[mode] = (out, lse)

    # Backward from the fused forward's O and LSE.
    gen = torch.Generator().manual_seed(200 + i)
    do = torch.randn((T, H, D), generator=gen).to(torch.bfloat16)
    out, lse = outs[cp.MODE_FUSED]
    bufs = [_guarded((T, H, D), torch.bfloat16) for _ in range(3)]
    ws = cp.alloc_bwd_workspace(T, len(lengths), H, D, max_cp, "cuda")
    cp.bwd(g["q"], g["k"], g["v"], out, do.to("cuda"), lse, g["cu"], cps_t,
           max_seqlen=max_seqlen, max_cp=max_cp, softmax_scale=scale, causal=causal,
           dq=bufs[0][1], dk=bufs[1][1], dv=bufs[2][1], workspace=ws)
    assert cp.poll_error(ws) == cp.OK, what
    for b, _ in bufs:
        assert _guard_intact(b, T), what
    ref = ob.full_attention_backward(qf, kf, vf, workloads.to_f64(do), cu, scale, causal=causal)
    for name, (_, got) in zip(("dq", "dk", "dv"), bufs):
        check_grad(got.float().cpu().numpy(), ref[name], "%s %s" % (name, what))
