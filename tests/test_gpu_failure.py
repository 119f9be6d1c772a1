"""Failure detection on the GPU without a GPU fault.

A test-only build of the library (``CPATTN_FAULT_INJECT_DROP_P``) makes the
first CTA of the forward kernel skip one hand-off from its softmax warps to
its MMA warp, and the first CTA of the backward's dK/dV kernel wait for its
first S^T on a barrier that completes only after its last MMA.  Every such
wait is bounded (2 s), so the kernels must end by themselves, report
CPATTN_ERR_DEVICE_TIMEOUT through the workspace error word, and leave the
CUDA context usable: the regular library then runs the same problem
correctly on the same device.
"""

import ctypes
import time

import numpy as np
import pytest
import torch

from helpers import check_attention, default_scale, make_batch
from long_context_gb300 import workloads
from oracle import attention as oa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_gb300 import build as lib_build
    path = lib_build.build_fault_injection()
    from long_context_gb300 import cpattn
    fault = ctypes.CDLL(path)
    fault.cpattn_fwd.argtypes = cpattn._lib.cpattn_fwd.argtypes
    fault.cpattn_fwd.restype = ctypes.c_int
    fault.cpattn_poll_error.argtypes = cpattn._lib.cpattn_poll_error.argtypes
    fault.cpattn_poll_error.restype = ctypes.c_int
    fault.cpattn_bwd.argtypes = cpattn._lib.cpattn_bwd.argtypes
    fault.cpattn_bwd.restype = ctypes.c_int
    return cpattn, fault


def test_bounded_wait_times_out_and_context_survives(libs):
    cp, fault = libs
    lengths, H, D = [700, 300], 2, 128
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=17)
    T = sum(lengths)
    out = torch.zeros((T, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    ws = cp.alloc_workspace(T, 2, H, D, 1)
    stream = torch.cuda.current_stream()
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    torch.cuda.synchronize()
    t0 = time.time()
    st = fault.cpattn_fwd(p(g["q"]), p(g["k"]), p(g["v"]), p(g["cu"]), None, 2, T, 700, 1, H, D,
                          default_scale(D), 1, 0, p(out), p(lse), p(ws), ws.numel(),
                          ctypes.c_void_p(stream.cuda_stream))
    assert st == cp.OK  # the launch itself is fine
    status = fault.cpattn_poll_error(p(ws), ctypes.c_void_p(stream.cuda_stream))
    elapsed = time.time() - t0
    assert status == cp.ERR_DEVICE_TIMEOUT
    assert elapsed < 30.0
    # The context is still usable: the regular library gets the right answer.
    out2, lse2 = cp.fwd(g["q"], g["k"], g["v"], g["cu"], None, max_seqlen=700, max_cp=1,
                        workspace=ws)
    assert cp.poll_error(ws) == cp.OK
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    ref_o, ref_lse = oa.full_attention(qf, kf, vf, cu, default_scale(D))
    check_attention(out2.float().cpu().numpy(), lse2.cpu().numpy(), ref_o, ref_lse,
                    "after timeout")


def test_backward_bounded_wait_times_out_and_context_survives(libs):
    """The dK/dV kernel's compute warp whose wait ran out keeps taking part in
    the named-barrier hand-offs (bar.sync), so the MMA warp and the kernel
    finish; the status is a timeout, then the regular backward is right."""
    from helpers import check_grad
    from oracle import backward as ob
    cp, fault = libs
    lengths, H, D = [700, 300], 2, 128
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=19)
    T = sum(lengths)
    gen = torch.Generator().manual_seed(23)
    dout = torch.randn((T, H, D), generator=gen).to(torch.bfloat16)
    dout_d = dout.cuda()
    out, lse = cp.fwd(g["q"], g["k"], g["v"], g["cu"], None, max_seqlen=700, max_cp=1)
    ws = cp.alloc_bwd_workspace(T, 2, H, D, 1, torch.device("cuda"))
    dq, dk, dv = (torch.zeros_like(g["q"]) for _ in range(3))
    stream = torch.cuda.current_stream()
    p = lambda t_: ctypes.c_void_p(t_.data_ptr())  # noqa: E731
    torch.cuda.synchronize()
    t0 = time.time()
    st = fault.cpattn_bwd(p(g["q"]), p(g["k"]), p(g["v"]), p(out), p(dout_d), p(lse), p(g["cu"]),
                          None, 2, T, 700, 1, H, D, default_scale(D), 1, p(dq), p(dk), p(dv),
                          p(ws), ws.numel(), ctypes.c_void_p(stream.cuda_stream))
    assert st == cp.OK
    status = fault.cpattn_poll_error(p(ws), ctypes.c_void_p(stream.cuda_stream))
    elapsed = time.time() - t0
    assert status == cp.ERR_DEVICE_TIMEOUT
    assert elapsed < 30.0
    dq2, dk2, dv2 = cp.bwd(g["q"], g["k"], g["v"], out, dout_d, lse, g["cu"], None,
                           max_seqlen=700, max_cp=1, workspace=ws)
    assert cp.poll_error(ws) == cp.OK
    ref = ob.full_attention_backward(*(workloads.to_f64(x) for x in (q, k, v, dout)), cu,
                                     default_scale(D))
    for name, got in (("dq", dq2), ("dk", dk2), ("dv", dv2)):
        check_grad(got.float().cpu().numpy(), ref[name], name + " after timeout")
