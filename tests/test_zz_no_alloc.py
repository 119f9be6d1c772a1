"""cpattn_fwd_noalloc against cpattn_fwd and the float64 oracle.

cpattn_fwd_noalloc serves callers that cannot allocate device memory (for
example code running inside a host program whose memory pool owns the whole
device budget, or latency-critical code that must not call cudaMalloc because
it can synchronise the device).  Instead of a workspace argument it uses a
fixed scratch array inside the library, shared by every call.  These tests go
through the C ABI: two calls in a row, on different batches, must each match
cpattn_fwd and the oracle within the parity tolerance; a problem too large for
the fixed scratch must be refused before anything is enqueued; and an error
the kernels detect on the device must reach the status word, with the next
good call on the shared scratch clean again.
"""

import ctypes

import numpy as np
import pytest
import torch

from helpers import LSE_RTOL, O_ATOL, check_attention, default_scale, make_batch
from long_context_gb300 import workloads
from oracle import attention as oa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_gb300 import build as lib_build
    lib_build.build()
    from long_context_gb300 import cpattn
    return cpattn


CASES = [
    # lengths, cp sizes, H, D, seed
    ([300, 1000, 77, 2048], [1, 2, 4, 4], 4, 128, 21),
    ([1024, 513, 1], [2, 1, 8], 3, 64, 22),
]


def _noalloc(cp, g, lengths, cps_t, max_cp, like_out, like_lse):
    out = torch.full_like(like_out, float("nan"))
    lse = torch.full_like(like_lse, float("nan"))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    cp.fwd_noalloc(g["q"], g["k"], g["v"], g["cu"], cps_t, max_seqlen=max(lengths),
                   max_cp=max_cp, out=out, lse=lse, status=status)
    torch.cuda.synchronize()
    return out, lse, int(status.item())


def test_noalloc_matches_fwd_and_oracle_on_two_calls_in_a_row(cp):
    for lengths, cps, H, D, seed in CASES:
        (q, k, v, cu), g = make_batch(lengths, H, D, seed=seed)
        cps_t = torch.tensor(cps, dtype=torch.int32, device="cuda")
        ref_out, ref_lse = cp.fwd(g["q"], g["k"], g["v"], g["cu"], cps_t,
                                  max_seqlen=max(lengths), max_cp=max(cps))
        out, lse, st = _noalloc(cp, g, lengths, cps_t, max(cps), ref_out, ref_lse)
        assert st == cp.OK
        do = (out.float() - ref_out.float()).abs().max().item()
        dl = ((lse - ref_lse).abs() / ref_lse.abs().clamp(min=1.0)).max().item()
        assert do <= O_ATOL, do
        assert dl <= LSE_RTOL, dl
        # Every element against the float64 oracle as well.
        qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
        want_o, want_lse = oa.full_attention(qf, kf, vf, cu, default_scale(D))
        check_attention(out.float().cpu().numpy(), lse.cpu().numpy(), want_o, want_lse,
                        "noalloc %s" % lengths)


def test_noalloc_reports_device_errors_and_recovers(cp):
    lengths, H, D = [100, 50], 2, 64
    (q, k, v, cu), g = make_batch(lengths, H, D, seed=4)
    # cu_seqlens ends short of the 150 tokens passed: only the schedule kernel
    # can see that; it sets the error word and no attention work runs.
    bad = dict(g, cu=torch.tensor([0, 100, 140], dtype=torch.int32, device="cuda"))
    like_out = torch.empty_like(g["q"])
    like_lse = torch.empty((150, H), dtype=torch.float32, device="cuda")
    out, lse, st = _noalloc(cp, bad, lengths, None, 1, like_out, like_lse)
    assert st == cp.ERR_INVALID_ARG
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()
    # The next valid call on the same shared scratch starts clean.
    out, lse, st = _noalloc(cp, g, lengths, None, 1, like_out, like_lse)
    assert st == cp.OK
    ref_out, ref_lse = cp.fwd(g["q"], g["k"], g["v"], g["cu"], None, max_seqlen=100, max_cp=1)
    assert (out.float() - ref_out.float()).abs().max().item() <= O_ATOL
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    want_o, want_lse = oa.full_attention(qf, kf, vf, cu, default_scale(D))
    check_attention(out.float().cpu().numpy(), lse.cpu().numpy(), want_o, want_lse,
                    "noalloc after an error")


def test_noalloc_refuses_problems_beyond_its_scratch(cp):
    q = torch.zeros((16, 1, 128), dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 16], dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(q.data_ptr())
    # 2^30 tokens need a 33 MB work list, beyond the fixed 1 MiB scratch; the
    # call is refused on the host, so the small buffers are never read.
    st = cp._lib.cpattn_fwd_noalloc(p, p, p, ctypes.c_void_p(cu.data_ptr()), None, 1, 2**30,
                                    2**30, 1, 1, 128, 0.1, 1, p, None, None, None)
    assert st == cp.ERR_WORKSPACE_TOO_SMALL
