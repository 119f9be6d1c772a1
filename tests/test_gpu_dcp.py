"""GPU parity of the dynamic-CP data movement (cpattn_select_cu,
cpattn_permute_samples) against the oracle in oracle/dcp.py: bit-exact on
bytes and indices; and the DCP forward (select, attention at the planned CP
sizes, restore) against the oracle's attention."""

import numpy as np
import pytest
import torch

from helpers import check_attention, default_scale
from long_context_gb300 import workloads
from oracle import attention as oa
from oracle import dcp as od
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


@pytest.mark.parametrize("H,dtype", [(2, torch.float32), (4, torch.float32), (3, torch.bfloat16),
                                     (32, torch.bfloat16)])
def test_select_and_restore_bit_exact(cp, H, dtype):
    lengths = [5, 0, 300, 129, 1, 0, 77, 4096, 2]
    T = sum(lengths)
    cu = workloads.cu_seqlens(lengths)
    g = torch.Generator().manual_seed(H)
    shape = (T, H) if dtype == torch.float32 else (T, H, 8)
    x = torch.randn(shape, generator=g).to(dtype)
    ids = [7, 2, 0, 8, 1, 6]
    want, want_cu = od.select(x.numpy() if dtype == torch.float32 else x.view(torch.int16).numpy(),
                              cu, ids)
    dcu = torch.from_numpy(cu).cuda()
    dids = torch.tensor(ids, dtype=torch.int32, device="cuda")
    pack_cu, status = cp.select_cu(dcu, dids)
    assert int(status.item()) == 0
    assert np.array_equal(pack_cu.cpu().numpy(), want_cu)
    xd = x.cuda()
    packed = torch.full((int(want_cu[-1]),) + tuple(shape[1:]), float("nan"), dtype=dtype,
                        device="cuda")
    cp.permute_samples(xd, dcu, pack_cu, dids, status, gather=True, dst=packed)
    got = packed.cpu()
    got = got.numpy() if dtype == torch.float32 else got.view(torch.int16).numpy()
    assert np.array_equal(got, want)
    # Restore into a NaN-filled array: the selected samples come back bit for
    # bit, everything else stays untouched.
    back = torch.full_like(xd, float("nan"))
    cp.permute_samples(packed, dcu, pack_cu, dids, status, gather=False, dst=back)
    b = back.cpu()
    for s in ids:
        assert torch.equal(b[cu[s]:cu[s + 1]].view(torch.int16 if dtype != torch.float32 else torch.int32),
                           x[cu[s]:cu[s + 1]].view(torch.int16 if dtype != torch.float32 else torch.int32))
    for s in set(range(len(lengths))) - set(ids):
        assert torch.isnan(b[cu[s]:cu[s + 1]].float()).all()


def test_invalid_ids_copy_nothing(cp):
    cu = torch.from_numpy(workloads.cu_seqlens([3, 4])).cuda()
    ids = torch.tensor([1, 5], dtype=torch.int32, device="cuda")
    pack_cu, status = cp.select_cu(cu, ids)
    assert int(status.item()) == 1
    src = torch.arange(7 * 4, dtype=torch.float32, device="cuda").reshape(7, 4)
    dst = torch.full((8, 4), -1.0, device="cuda")
    cp.permute_samples(src, cu, pack_cu, ids, status, gather=True, dst=dst)
    assert (dst == -1).all()


def test_dcp_forward_matches_attention(cp):
    """A batch that needs several micro-batches and mixed CP sizes: select,
    attention, restore gives every sample's full attention in original order."""
    lengths = [2100, 300, 77, 1500, 4000, 1, 650, 129]
    H, D = 2, 128
    plan = cp.plan(lengths, 4, 1024, 4)
    plan_o = op.plan(lengths, 4, 1024, 4)
    assert list(plan["micro_batch"]) == plan_o["micro_batch"]
    assert plan["num_micro_batches"] > 1
    T = sum(lengths)
    q, k, v = workloads.qkv(T, H, D, 13)
    cu = workloads.cu_seqlens(lengths)
    scale = default_scale(D)
    out, lse = cp.dcp_fwd(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cu).cuda(), plan,
                          seqlens=lengths, max_cp=4, softmax_scale=scale)
    ref_o, ref_l = od.dcp_forward(*(workloads.to_f64(x) for x in (q, k, v)), cu, plan_o, scale)
    check_attention(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "dcp forward")
    # The prepared runner, called twice on the same buffers, gives the same
    # bits as the one-shot call.
    run = cp.DcpForward(lengths, plan, num_heads=H, head_dim=D, max_cp=4)
    for _ in range(2):
        o2, l2 = run(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cu).cuda(),
                     softmax_scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(o2, out) and torch.equal(l2, lse)
    full_o, full_l = oa.full_attention(*(workloads.to_f64(x) for x in (q, k, v)), cu, scale)
    assert np.max(np.abs(ref_o - full_o)) < 1e-12


def test_select_restore_full_size(cp):
    """The size the benchmark times: the 65,536-token packed batch, H=32,
    D=128 bf16, every sample moved in reversed order; the whole packed array
    against the oracle's selection (bit-exact), then restored bit for bit."""
    H, D = 32, 128
    lengths = workloads.packed_lengths(0, 65536)
    T = sum(lengths)
    g = torch.Generator(device="cuda").manual_seed(0)
    x = torch.randn((T, H, D), generator=g, device="cuda").to(torch.bfloat16)
    cu = workloads.cu_seqlens(lengths)
    ids = list(range(len(lengths) - 1, -1, -1))
    dcu = torch.from_numpy(cu).cuda()
    dids = torch.tensor(ids, dtype=torch.int32, device="cuda")
    pack_cu, status = cp.select_cu(dcu, dids)
    assert int(status.item()) == 0
    packed = torch.empty_like(x)
    cp.permute_samples(x, dcu, pack_cu, dids, status, gather=True, dst=packed)
    want, want_cu = od.select(x.cpu().view(torch.int16).numpy(), cu, ids)
    assert np.array_equal(pack_cu.cpu().numpy(), want_cu)
    assert np.array_equal(packed.cpu().view(torch.int16).numpy(), want)
    back = torch.empty_like(x)
    cp.permute_samples(packed, dcu, pack_cu, dids, status, gather=False, dst=back)
    assert torch.equal(back.view(torch.int16), x.view(torch.int16))
