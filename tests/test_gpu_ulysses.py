"""GPU parity of the Ulysses layout (cpattn_ulysses_layout,
cpattn_ulysses_seqlens) against oracle/ulysses.py: bit-exact on bytes and
indices; and Ulysses attention (head-group layout, one forward over all
groups, layout back) against the oracle's attention."""

import numpy as np
import pytest
import torch

from helpers import check_attention, default_scale, sample_tokens
from long_context_gb300 import workloads
from oracle import attention as oa
from oracle import ulysses as ou

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_gb300 import build as lib_build
    lib_build.build()
    from long_context_gb300 import cpattn
    return cpattn


def _bits(x):
    """Integer view of a CPU tensor as a NumPy array (bit-exact comparison)."""
    view = {torch.bfloat16: torch.int16, torch.float32: torch.int32}[x.dtype]
    return x.view(view).numpy()


# (T, H, P, per-head shape, dtype): 16-byte units with 1 KB, 256 B and 16 B
# chunks, 8-byte units (8 B chunks), 4-byte units (12 B and 4 B chunks),
# P = 1 and P = H.
CASES = [
    (1000, 32, 8, (128,), torch.bfloat16),
    (777, 4, 2, (64,), torch.bfloat16),
    (333, 6, 3, (3,), torch.bfloat16),
    (500, 32, 8, (), torch.float32),
    (129, 8, 4, (), torch.float32),
    (129, 8, 8, (), torch.float32),
    (65, 32, 1, (128,), torch.bfloat16),
    (65, 8, 8, (128,), torch.bfloat16),
    (1, 16, 4, (64,), torch.bfloat16),
]


@pytest.mark.parametrize("T,H,P,rest,dtype", CASES)
def test_layout_bit_exact(cp, T, H, P, rest, dtype):
    g = torch.Generator().manual_seed(T * 31 + H)
    x = torch.randn((T, H) + rest, generator=g).to(dtype)
    want = ou.to_head_groups(_bits(x), P)
    y = cp.ulysses_layout(x.cuda(), P, to_head_groups=True)
    assert tuple(y.shape) == (P, T, H // P) + rest
    assert np.array_equal(_bits(y.cpu()), want)
    back = cp.ulysses_layout(y, P, to_head_groups=False)
    assert np.array_equal(_bits(back.cpu()), ou.from_head_groups(want, P))
    assert np.array_equal(_bits(back.cpu()), _bits(x))


def test_layout_misaligned_buffers_use_word_copies(cp):
    """Buffers 4 bytes off a 16-byte boundary take the 4-byte-unit path and
    still give the oracle's layout."""
    T, H, P, D = 301, 8, 4, 16
    n = T * H * D
    g = torch.Generator().manual_seed(5)
    base = torch.randn(n + 1, generator=g)
    src = base.cuda()[1:].view(T, H, D)
    assert src.data_ptr() % 16 == 4
    dst_buf = torch.full((n + 1,), float("nan"), device="cuda")
    dst = dst_buf[1:].view(P, T, H // P, D)
    cp.ulysses_layout(src, P, to_head_groups=True, dst=dst)
    want = ou.to_head_groups(_bits(base[1:].view(T, H, D)), P)
    assert np.array_equal(_bits(dst.cpu()), want)
    assert np.isnan(dst_buf[0].item())          # nothing written before dst


def test_layout_empty(cp):
    x = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    y = cp.ulysses_layout(x, 4, to_head_groups=True)
    assert tuple(y.shape) == (4, 0, 2, 128)


@pytest.mark.parametrize("with_cp", [False, True])
def test_seqlens(cp, with_cp):
    lengths = [5, 0, 300, 1, 77]
    cu = workloads.cu_seqlens(lengths)
    T, P, B = int(cu[-1]), 4, len(lengths)
    cps = np.array([1, 2, 4, 1, 2], dtype=np.int32)
    dcps = torch.from_numpy(cps).cuda() if with_cp else None
    cu_g, cp_g = cp.ulysses_seqlens(torch.from_numpy(cu).cuda(), dcps, P, T)
    cu_g, cp_g = cu_g.cpu().numpy(), cp_g.cpu().numpy()
    # Group p's samples are the original samples, T rows further on; the
    # grouped batch's lengths are the original lengths repeated P times.
    assert cu_g[0] == 0 and cu_g[-1] == P * T
    assert list(np.diff(cu_g)) == lengths * P
    for p in range(P):
        assert list(cu_g[p * B:(p + 1) * B]) == [int(c) + p * T for c in cu[:-1]]
    assert list(cp_g) == (list(cps) if with_cp else [1] * B) * P
    e_cu, _ = cp.ulysses_seqlens(torch.zeros(1, dtype=torch.int32, device="cuda"), None, 4, 0)
    assert e_cu.cpu().tolist() == [0]


@pytest.mark.parametrize("P,D,hybrid", [(2, 128, False), (4, 128, True), (8, 64, False),
                                        (8, 128, True)])
def test_ulysses_fwd_matches_oracle(cp, P, D, hybrid):
    """Ulysses attention (optionally with ring CP inside every head group)
    equals the oracle's Ulysses attention, which equals full attention."""
    lengths = [700, 1, 129, 2048, 300, 64]
    H = 8
    T = sum(lengths)
    q, k, v = workloads.qkv(T, H, D, 40 + P)
    cu = workloads.cu_seqlens(lengths)
    scale = default_scale(D)
    cps = torch.tensor([2, 1, 1, 4, 2, 1] if hybrid else [1] * len(lengths),
                       dtype=torch.int32, device="cuda")
    out, lse = cp.ulysses_fwd(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cu).cuda(), P,
                              cps, max_seqlen=max(lengths), max_cp=4 if hybrid else 1,
                              softmax_scale=scale)
    f64 = [workloads.to_f64(x) for x in (q, k, v)]
    ref_o, ref_l = ou.ulysses_attention(*f64, cu, P, scale)
    check_attention(out.float().cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l,
                    "ulysses P=%d" % P)
    full_o, _ = oa.full_attention(*f64, cu, scale)
    assert np.max(np.abs(ref_o - full_o)) < 1e-12


def test_layout_full_size_sampled(cp):
    """131,072 tokens, H=32, D=128 bf16, P=8 (the size the benchmark moves):
    sampled tokens against the oracle, every token through the round trip."""
    T, H, D, P = 131072, 32, 128, 8
    g = torch.Generator(device="cuda").manual_seed(9)
    x = torch.randn((T, H, D), generator=g, device="cuda").to(torch.bfloat16)
    y = cp.ulysses_layout(x, P, to_head_groups=True)
    toks = sample_tokens([0, T], 64, 3, extra=(1023, 1024, 65535, 65536))
    xs = x[toks].cpu()
    ys = y[:, toks].cpu()
    want = ou.to_head_groups(_bits(xs), P)
    assert np.array_equal(_bits(ys), want)
    back = cp.ulysses_layout(y, P, to_head_groups=False)
    assert torch.equal(back.view(torch.int16), x.view(torch.int16))
    lse = torch.randn((T, H), generator=g, device="cuda")
    lg = cp.ulysses_layout(lse, P, to_head_groups=True)
    assert np.array_equal(_bits(lg[:, toks].cpu()), ou.to_head_groups(_bits(lse[toks].cpu()), P))
    assert torch.equal(cp.ulysses_layout(lg, P, to_head_groups=False), lse)
