"""cpattn_fwd_noalloc against cpattn_fwd.

cpattn_fwd_noalloc serves callers that cannot allocate device memory (for
example code running inside a host program whose memory pool owns the whole
device budget, or latency-critical code that must not call cudaMalloc because
it can synchronise the device).  Instead of a workspace argument it uses a
fixed scratch array inside the library, shared by every call.  These tests go
through the C ABI: two calls in a row, on different batches, must each match
cpattn_fwd within the parity tolerance, and a problem too large for the fixed
scratch must be refused before anything is enqueued.
"""

import ctypes

import pytest
import torch

from helpers import LSE_RTOL, O_ATOL, make_batch

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


def test_noalloc_matches_fwd_on_two_calls_in_a_row(cp):
    for lengths, cps, H, D, seed in CASES:
        (_, _, _, _), g = make_batch(lengths, H, D, seed=seed)
        cps_t = torch.tensor(cps, dtype=torch.int32, device="cuda")
        ref_out, ref_lse = cp.fwd(g["q"], g["k"], g["v"], g["cu"], cps_t,
                                  max_seqlen=max(lengths), max_cp=max(cps))
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        cp.fwd_noalloc(g["q"], g["k"], g["v"], g["cu"], cps_t, max_seqlen=max(lengths),
                       max_cp=max(cps), out=out, lse=lse, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == cp.OK
        do = (out.float() - ref_out.float()).abs().max().item()
        dl = ((lse - ref_lse).abs() / ref_lse.abs().clamp(min=1.0)).max().item()
        assert do <= O_ATOL, do
        assert dl <= LSE_RTOL, dl


def test_noalloc_refuses_problems_beyond_its_scratch(cp):
    q = torch.zeros((16, 1, 128), dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 16], dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(q.data_ptr())
    # 2^30 tokens need a 33 MB work list, beyond the fixed 1 MiB scratch; the
    # call is refused on the host, so the small buffers are never read.
    st = cp._lib.cpattn_fwd_noalloc(p, p, p, ctypes.c_void_p(cu.data_ptr()), None, 1, 2**30,
                                    2**30, 1, 1, 128, 0.1, 1, p, None, None, None)
    assert st == cp.ERR_WORKSPACE_TOO_SMALL
