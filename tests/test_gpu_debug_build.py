"""The debug build of the library (-DCPATTN_DEBUG) on the GPU.

In the debug build the schedule, forward and backward kernels check every
global index and TMA coordinate they derive against the tensors' bounds, and
a failed check is reported as CPATTN_ERR_DEVICE_BOUNDS in the workspace error
word (the access is skipped; nothing traps).  Run over the ragged lengths at
every CP size, head dim, causal flag and mode, the checks must stay silent
(status OK) and the results must match the float64 oracle: no kernel reaches
outside its tensors on these shapes.
"""

import ctypes

import numpy as np
import pytest
import torch

from helpers import check_attention, check_grad, default_scale, make_batch
from long_context_gb300 import workloads
from oracle import attention as oa
from oracle import backward as ob

pytestmark = pytest.mark.gpu

RAGGED = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 511, 513]


@pytest.fixture(scope="module")
def dbg():
    """The binding with its library swapped for libcpattn_debug.so."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_gb300 import build as lib_build
    path = lib_build.build_debug()
    from long_context_gb300 import cpattn
    lib = ctypes.CDLL(path)
    for name in dir(cpattn._lib):
        if name.startswith("cpattn_"):
            f, g = getattr(cpattn._lib, name), getattr(lib, name)
            g.argtypes, g.restype = f.argtypes, f.restype
    regular = cpattn._lib
    cpattn._lib = lib
    yield cpattn
    cpattn._lib = regular


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("mode", [0, 1])
def test_debug_build_forward_ragged(dbg, D, causal, mode):
    cp = dbg
    lengths = RAGGED
    cps = [[1, 2, 4, 8][i % 4] for i in range(len(lengths))]
    H = 3
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=11)
    T = sum(lengths)
    scale = default_scale(D)
    ws = cp.alloc_workspace(T, len(lengths), H, D, 8, mode)
    cps_t = torch.tensor(cps, dtype=torch.int32, device="cuda")
    out, lse = cp.fwd(g["q"], g["k"], g["v"], g["cu"], cps_t, max_seqlen=max(lengths),
                      max_cp=8, softmax_scale=scale, causal=causal, mode=mode, workspace=ws)
    assert cp.poll_error(ws) == cp.OK
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    ref_o, ref_lse = oa.full_attention(qf, kf, vf, cu, scale, causal=causal)
    check_attention(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_lse,
                    "debug build D=%d causal=%s mode=%d" % (D, causal, mode))


@pytest.mark.parametrize("D", [64, 128])
def test_debug_build_backward_ragged(dbg, D):
    cp = dbg
    lengths = [1, 127, 128, 129, 255, 256, 257, 513]
    cps = [1, 1, 2, 1, 2, 4, 2, 8]
    H = 2
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=12)
    T = sum(lengths)
    scale = default_scale(D)
    gen = torch.Generator().manual_seed(99)
    do = torch.randn((T, H, D), generator=gen).to(torch.bfloat16)
    cps_t = torch.tensor(cps, dtype=torch.int32, device="cuda")
    out, lse = cp.fwd(g["q"], g["k"], g["v"], g["cu"], cps_t, max_seqlen=max(lengths),
                      max_cp=8, softmax_scale=scale)
    ws = cp.alloc_bwd_workspace(T, len(lengths), H, D, 8)
    dq, dk, dv = cp.bwd(g["q"], g["k"], g["v"], out, do.cuda(), lse, g["cu"], cps_t,
                        max_seqlen=max(lengths), max_cp=8, softmax_scale=scale, workspace=ws)
    assert cp.poll_error(ws) == cp.OK
    ref = ob.full_attention_backward(*(workloads.to_f64(x) for x in (q, k, v, do)), cu, scale)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_grad(got.float().cpu().numpy(), ref[name], "debug build %s D=%d" % (name, D))
