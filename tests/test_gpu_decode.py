"""GPU parity of decode-time CP (cpattn_decode_partials, cpattn_merge_lse,
cpattn_decode) against oracle/decode.py.

The partials are computed in fp32 from bf16 inputs with fp32 probabilities
(no bf16 rounding inside), so they are held to fp32 rounding: max |dO_s| <=
1e-4 and |dlse_s| <= 1e-5 * max(1, |lse_s|).  The merge is fp32 throughout:
O within MERGE_RTOL of its row's max |O| (helpers.check_merge_o).  The fused
call writes bf16 O: the forward's tolerances."""

import numpy as np
import pytest
import torch

from helpers import check_attention, check_merge_o, default_scale
from long_context_gb300 import workloads
from oracle import decode as odc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_gb300 import build as lib_build
    lib_build.build()
    from long_context_gb300 import cpattn
    return cpattn


def _inputs(lengths, H, D, seed, std=1.0):
    T = int(sum(lengths))
    k, v, _ = workloads.qkv(T, H, D, seed, std)
    g = torch.Generator().manual_seed(seed + 77)
    q = (torch.randn((len(lengths), H, D), generator=g) * std).to(torch.bfloat16)
    cu = workloads.cu_seqlens(lengths)
    return q, k, v, cu


CASES = [
    ([1000, 1, 0, 37, 4096], 2, 128, 4),
    ([5, 3, 2, 1], 3, 64, 8),
    ([2048, 700], 4, 128, 1),
    ([900, 129, 128, 127], 2, 128, 3),
]


@pytest.mark.parametrize("lengths,H,D,c", CASES)
def test_partials_merge_and_decode(cp, lengths, H, D, c):
    q, k, v, cu = _inputs(lengths, H, D, seed=sum(lengths) % 31)
    scale = default_scale(D)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    cud = torch.from_numpy(cu).cuda()
    qf, kf, vf = (workloads.to_f64(x) for x in (q, k, v))
    ref_os, ref_ls = odc.shard_partials(qf, kf, vf, cu, c, scale)
    o_s, l_s = cp.decode_partials(qd, kd, vd, cud, cp=c, softmax_scale=scale)
    o_s, l_s = o_s.cpu().numpy(), l_s.cpu().numpy()
    assert np.array_equal(np.isneginf(l_s), np.isneginf(ref_ls))
    fin = np.isfinite(ref_ls)
    assert np.max(np.abs(o_s - ref_os)) <= 1e-4
    assert np.max(np.abs(l_s[fin] - ref_ls[fin]) / np.maximum(1, np.abs(ref_ls[fin]))) <= 1e-5
    # LSE-form merge of the GPU partials against the oracle's merge of them.
    mo, ml = cp.merge_lse(torch.from_numpy(o_s).cuda(), torch.from_numpy(l_s).cuda())
    ref_mo, ref_ml = odc.merge_lse(o_s, l_s)
    check_merge_o(mo.cpu().numpy(), ref_mo, "merge_lse %s" % lengths)
    mlc = ml.cpu().numpy()
    assert np.array_equal(np.isneginf(mlc), np.isneginf(ref_ml))
    f2 = np.isfinite(ref_ml)
    assert np.max(np.abs(mlc[f2] - ref_ml[f2]) / np.maximum(1, np.abs(ref_ml[f2]))) <= 1e-5
    # The fused call against the plain definition.
    out, lse = cp.decode(qd, kd, vd, cud, cp=c, softmax_scale=scale)
    ref_o, ref_l = odc.decode_attention(qf, kf, vf, cu, scale)
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    empty = np.diff(cu) == 0
    assert np.all(out[empty] == 0) and np.all(np.isneginf(lse[empty]))
    check_attention(out[~empty], lse[~empty], ref_o[~empty], ref_l[~empty], "decode")


def test_decode_cp_invariance_large_scores(cp):
    """Scores spread over many powers of two; every CP size gives the same
    answer (within tolerance) as the plain definition."""
    lengths, H, D = [3000, 17, 640], 2, 128
    q, k, v, cu = _inputs(lengths, H, D, seed=5, std=2.5)
    scale = default_scale(D)
    ref_o, ref_l = odc.decode_attention(*(workloads.to_f64(x) for x in (q, k, v)), cu, scale)
    for c in (1, 2, 4, 8, 16):
        out, lse = cp.decode(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cu).cuda(), cp=c,
                             softmax_scale=scale)
        check_attention(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, "cp %d" % c)


def test_decode_full_size_sampled(cp):
    """The size the benchmark times: 64 sequences with KV caches of uniform
    length in [4096, 32768] (about 1.2 M cached tokens, 9.8 GB), H=32, D=128,
    decode CP 4.  Every sequence's output on the GPU; eight sampled sequences
    (the shortest, the longest and six more) against the oracle."""
    B, H, D, c = 64, 32, 128, 4
    lengths = [int(x) for x in np.random.default_rng(0).integers(4096, 32769, B)]
    T = sum(lengths)
    g = torch.Generator(device="cuda").manual_seed(0)
    k = torch.randn((T, H, D), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((T, H, D), generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn((B, H, D), generator=g, device="cuda").to(torch.bfloat16)
    cu = workloads.cu_seqlens(lengths)
    scale = default_scale(D)
    out, lse = cp.decode(q, k, v, torch.from_numpy(cu).cuda(), cp=c, softmax_scale=scale)
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    picks = sorted({int(np.argmin(lengths)), int(np.argmax(lengths))}
                   | {int(b) for b in np.random.default_rng(3).choice(B, 6, replace=False)})
    for b in picks:
        s0, s1 = int(cu[b]), int(cu[b + 1])
        ref_o, ref_l = odc.decode_attention(
            workloads.to_f64(q[b:b + 1].cpu()), workloads.to_f64(k[s0:s1].cpu()),
            workloads.to_f64(v[s0:s1].cpu()), [0, s1 - s0], scale)
        check_attention(out[b:b + 1], lse[b:b + 1], ref_o, ref_l, "sequence %d" % b)
