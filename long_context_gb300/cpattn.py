"""Python binding of the cpattn C ABI (``include/cpattn.h``).

Argument marshalling only: tensors are checked for dtype, device, layout and
contiguity, then their device pointers are handed to ``libcpattn.so`` together
with PyTorch's current CUDA stream.  Every step of the computation runs in the
library's kernels; there is no fallback.  Importing this module raises
``ImportError`` when the library has not been built (``build.build()``).
"""

from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcpattn.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        "libcpattn.so is missing at %s; build it with "
        "long_context_gb300.build.build()" % _LIB_PATH)
_lib = ctypes.CDLL(_LIB_PATH)

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_WORKSPACE_TOO_SMALL = 3
ERR_PLAN_INFEASIBLE = 4
ERR_CUDA = 5
ERR_DEVICE_TIMEOUT = 6
MODE_FUSED = 0
MODE_UNFUSED = 1

_i32p = ctypes.POINTER(ctypes.c_int32)
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64

_lib.cpattn_plan.argtypes = [_i32p, _i32, _i32, _i32, _i32, _i32p, _i32p, _i32p,
                             _i32p, _i32p, _i32p]
_lib.cpattn_plan.restype = ctypes.c_int
_lib.cpattn_fwd_workspace_size.argtypes = [_i64, _i32, _i32, _i32, _i32, _i32]
_lib.cpattn_fwd_workspace_size.restype = ctypes.c_size_t
_lib.cpattn_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32,
                            _i32, ctypes.c_float, _i32, _i32, _vp, _vp, _vp,
                            ctypes.c_size_t, _vp]
_lib.cpattn_fwd.restype = ctypes.c_int
_lib.cpattn_fwd_partials.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32,
                                     _i32, _i32, ctypes.c_float, _i32, _i32, _vp, _vp,
                                     _vp, _vp, ctypes.c_size_t, _vp]
_lib.cpattn_fwd_partials.restype = ctypes.c_int
_lib.cpattn_fwd_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32,
                                    _i32, ctypes.c_float, _i32, _vp, _vp, _vp, _vp]
_lib.cpattn_fwd_noalloc.restype = ctypes.c_int
_lib.cpattn_merge.argtypes = [_vp, _vp, _vp, _i32, _i64, _i32, _i32, _vp, _vp, _vp, _vp]
_lib.cpattn_merge.restype = ctypes.c_int
_lib.cpattn_bwd_workspace_size.argtypes = [_i64, _i32, _i32, _i32, _i32]
_lib.cpattn_bwd_workspace_size.restype = ctypes.c_size_t
_lib.cpattn_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32,
                            _i32, _i32, ctypes.c_float, _i32, _vp, _vp, _vp, _vp,
                            ctypes.c_size_t, _vp]
_lib.cpattn_bwd.restype = ctypes.c_int
_lib.cpattn_select_cu.argtypes = [_vp, _i32, _vp, _i32, _vp, _vp, _vp]
_lib.cpattn_select_cu.restype = ctypes.c_int
_lib.cpattn_permute_samples.argtypes = [_vp, _vp, _i32, _vp, _vp, _i32, _i64, _i32, _vp, _vp,
                                        _vp]
_lib.cpattn_permute_samples.restype = ctypes.c_int
_lib.cpattn_decode_workspace_size.argtypes = [_i32, _i32, _i32, _i32]
_lib.cpattn_decode_workspace_size.restype = ctypes.c_size_t
_lib.cpattn_decode_partials.argtypes = [_vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32,
                                        ctypes.c_float, _i32, _vp, _vp, _vp]
_lib.cpattn_decode_partials.restype = ctypes.c_int
_lib.cpattn_merge_lse.argtypes = [_vp, _vp, _i32, _i64, _i32, _vp, _vp, _vp]
_lib.cpattn_merge_lse.restype = ctypes.c_int
_lib.cpattn_decode.argtypes = [_vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, ctypes.c_float,
                               _i32, _vp, _vp, _vp, ctypes.c_size_t, _vp]
_lib.cpattn_decode.restype = ctypes.c_int
_lib.cpattn_ulysses_layout.argtypes = [_vp, _vp, _i64, _i32, _i64, _i32, _i32, _vp]
_lib.cpattn_ulysses_layout.restype = ctypes.c_int
_lib.cpattn_ulysses_seqlens.argtypes = [_vp, _vp, _i32, _i64, _i32, _vp, _vp, _vp]
_lib.cpattn_ulysses_seqlens.restype = ctypes.c_int
_lib.cpattn_poll_error.argtypes = [_vp, _vp]
_lib.cpattn_poll_error.restype = ctypes.c_int
_lib.cpattn_status_string.argtypes = [ctypes.c_int]
_lib.cpattn_status_string.restype = ctypes.c_char_p
_lib.cpattn_version.argtypes = []
_lib.cpattn_version.restype = ctypes.c_int


class CpattnError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, status_string(status), status))


def status_string(status):
    return _lib.cpattn_status_string(int(status)).decode()


def version():
    v = _lib.cpattn_version()
    return (v >> 16, (v >> 8) & 0xFF, v & 0xFF)


def library_path():
    return _LIB_PATH


def _check(status, what):
    if status != OK:
        raise CpattnError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, device=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if device is not None and t.device != device:
        raise ValueError("%s must be on %s, got %s" % (name, device, t.device))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


# ---------------------------------------------------------------- planner --

def plan(seqlens, dpxcp_world_size, max_seqlen_per_dp_cp_rank, max_cp):
    """``cpattn_plan`` on host arrays; returns a dict of NumPy int32 arrays.

    Keys: ``cp_size``, ``micro_batch``, ``first_rank``, ``order`` (length n),
    ``num_micro_batches`` (int) and ``rank_load`` ([num_micro_batches, W]).
    Raises :class:`CpattnError` on invalid arguments or an infeasible plan.
    """
    lens = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32))
    n = int(lens.shape[0])
    W = int(dpxcp_world_size)
    outs = [np.zeros(max(n, 1), dtype=np.int32) for _ in range(4)]
    nmb = np.zeros(1, dtype=np.int32)
    load = np.zeros(max(n * W, 1) if W > 0 else 1, dtype=np.int32)
    p = lambda a: a.ctypes.data_as(_i32p)  # noqa: E731
    st = _lib.cpattn_plan(p(lens) if n else None, n, W, int(max_seqlen_per_dp_cp_rank),
                          int(max_cp), p(outs[0]), p(outs[1]), p(outs[2]), p(outs[3]),
                          p(nmb), p(load))
    _check(st, "cpattn_plan")
    k = int(nmb[0])
    return {
        "cp_size": outs[0][:n].copy(),
        "micro_batch": outs[1][:n].copy(),
        "first_rank": outs[2][:n].copy(),
        "order": outs[3][:n].copy(),
        "num_micro_batches": k,
        "rank_load": load[:k * W].reshape(k, W).copy(),
    }


# ---------------------------------------------------------------- forward --

def workspace_size(total_tokens, num_seqs, num_heads, head_dim, max_cp, mode=MODE_FUSED):
    n = _lib.cpattn_fwd_workspace_size(int(total_tokens), int(num_seqs), int(num_heads),
                                       int(head_dim), int(max_cp), int(mode))
    if n == 0:
        raise CpattnError(ERR_INVALID_ARG, "cpattn_fwd_workspace_size")
    return int(n)


def alloc_workspace(total_tokens, num_seqs, num_heads, head_dim, max_cp, mode=MODE_FUSED,
                    device=None):
    """A device workspace sized for the given problem (torch-owned)."""
    n = workspace_size(total_tokens, num_seqs, num_heads, head_dim, max_cp, mode)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def _fwd_common(q, k, v, cu_seqlens, cp_size):
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3:
        raise ValueError("q must be [T, H, D]")
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q, k, v must be CUDA tensors")
    _need(k, "k", torch.bfloat16, dev, q.shape)
    _need(v, "v", torch.bfloat16, dev, q.shape)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    if cp_size is not None:
        _need(cp_size, "cp_size", torch.int32, dev, (cu_seqlens.numel() - 1,))
    return dev


def fwd(q, k, v, cu_seqlens, cp_size=None, *, max_seqlen, max_cp=None, softmax_scale=None,
        causal=True, mode=MODE_FUSED, out=None, lse=None, workspace=None, stream=None):
    """Ring-attention forward (``cpattn_fwd``); returns ``(out, lse)``.

    ``q, k, v``: bf16 ``[T, H, D]``; ``cu_seqlens``: int32 ``[B + 1]``;
    ``cp_size``: int32 ``[B]`` or None (CP 1 everywhere), all on the GPU.
    ``max_seqlen`` and ``max_cp`` bound the sample lengths and CP sizes.
    """
    dev = _fwd_common(q, k, v, cu_seqlens, cp_size)
    T, H, D = q.shape
    B = cu_seqlens.numel() - 1
    if max_cp is None:
        max_cp = 1 if cp_size is None else int(cp_size.max().item()) if B else 1
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.bfloat16, dev, q.shape)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    else:
        _need(lse, "lse", torch.float32, dev, (T, H))
    if workspace is None:
        workspace = alloc_workspace(T, B, H, D, max_cp, mode, dev)
    st = _lib.cpattn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(cp_size), B, T,
                         int(max_seqlen), int(max_cp), H, D, float(softmax_scale),
                         1 if causal else 0, int(mode), _ptr(out), _ptr(lse),
                         _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "cpattn_fwd")
    return out, lse


def fwd_noalloc(q, k, v, cu_seqlens, cp_size=None, *, max_seqlen, max_cp=None,
                softmax_scale=None, causal=True, out, lse=None, status=None, stream=None):
    """``cpattn_fwd_noalloc``: the fused forward with the library's fixed
    scratch instead of a workspace, for callers that cannot allocate device
    memory.  ``out`` (and ``lse``, ``status`` if given) are caller-provided;
    ``status`` is a device int32 tensor of one element receiving the device
    status.  Returns ``(out, lse)``."""
    dev = _fwd_common(q, k, v, cu_seqlens, cp_size)
    T, H, D = q.shape
    B = cu_seqlens.numel() - 1
    if max_cp is None:
        max_cp = 1 if cp_size is None else int(cp_size.max().item()) if B else 1
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    _need(out, "out", torch.bfloat16, dev, q.shape)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev, (T, H))
    if status is not None:
        _need(status, "status", torch.int32, dev, (1,))
    st = _lib.cpattn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(cp_size),
                                 B, T, int(max_seqlen), int(max_cp), H, D,
                                 float(softmax_scale), 1 if causal else 0, _ptr(out),
                                 _ptr(lse), _ptr(status), _stream(stream))
    _check(st, "cpattn_fwd_noalloc")
    return out, lse


def fwd_partials(q, k, v, cu_seqlens, cp_size=None, *, max_seqlen, max_cp, num_steps=None,
                 softmax_scale=None, causal=True, o_steps=None, m_steps=None, l_steps=None,
                 workspace=None, stream=None):
    """Per-ring-step partials (``cpattn_fwd_partials``); returns ``(o, m, l)``."""
    dev = _fwd_common(q, k, v, cu_seqlens, cp_size)
    T, H, D = q.shape
    B = cu_seqlens.numel() - 1
    S = int(num_steps or max_cp)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if o_steps is None:
        o_steps = torch.empty((S, T, H, D), dtype=torch.float32, device=dev)
    if m_steps is None:
        m_steps = torch.empty((S, T, H), dtype=torch.float32, device=dev)
    if l_steps is None:
        l_steps = torch.empty((S, T, H), dtype=torch.float32, device=dev)
    _need(o_steps, "o_steps", torch.float32, dev, (S, T, H, D))
    _need(m_steps, "m_steps", torch.float32, dev, (S, T, H))
    _need(l_steps, "l_steps", torch.float32, dev, (S, T, H))
    if workspace is None:
        workspace = alloc_workspace(T, B, H, D, max_cp, MODE_FUSED, dev)
    st = _lib.cpattn_fwd_partials(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(cp_size),
                                  B, T, int(max_seqlen), int(max_cp), H, D,
                                  float(softmax_scale), 1 if causal else 0, S, _ptr(o_steps),
                                  _ptr(m_steps), _ptr(l_steps), _ptr(workspace),
                                  workspace.numel(), _stream(stream))
    _check(st, "cpattn_fwd_partials")
    return o_steps, m_steps, l_steps


# --------------------------------------------------------------- backward --

def bwd_workspace_size(total_tokens, num_seqs, num_heads, head_dim, max_cp):
    n = _lib.cpattn_bwd_workspace_size(int(total_tokens), int(num_seqs), int(num_heads),
                                       int(head_dim), int(max_cp))
    if n == 0:
        raise CpattnError(ERR_INVALID_ARG, "cpattn_bwd_workspace_size")
    return int(n)


def alloc_bwd_workspace(total_tokens, num_seqs, num_heads, head_dim, max_cp, device=None):
    """A device workspace sized for ``cpattn_bwd`` (torch-owned)."""
    n = bwd_workspace_size(total_tokens, num_seqs, num_heads, head_dim, max_cp)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def bwd(q, k, v, out, dout, lse, cu_seqlens, cp_size=None, *, max_seqlen, max_cp=None,
        softmax_scale=None, causal=True, dq=None, dk=None, dv=None, workspace=None,
        stream=None):
    """Ring-attention backward (``cpattn_bwd``); returns ``(dq, dk, dv)``.

    ``out`` and ``lse`` are the outputs of the :func:`fwd` call being
    differentiated (same ``q, k, v, cu_seqlens, cp_size``, scale and causal
    flag); ``dout`` is the upstream gradient, bf16 ``[T, H, D]``.
    """
    dev = _fwd_common(q, k, v, cu_seqlens, cp_size)
    T, H, D = q.shape
    B = cu_seqlens.numel() - 1
    _need(out, "out", torch.bfloat16, dev, q.shape)
    _need(dout, "dout", torch.bfloat16, dev, q.shape)
    _need(lse, "lse", torch.float32, dev, (T, H))
    if max_cp is None:
        max_cp = 1 if cp_size is None else int(cp_size.max().item()) if B else 1
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    grads = []
    for name, g in (("dq", dq), ("dk", dk), ("dv", dv)):
        if g is None:
            g = torch.empty_like(q)
        else:
            _need(g, name, torch.bfloat16, dev, q.shape)
        grads.append(g)
    if workspace is None:
        workspace = alloc_bwd_workspace(T, B, H, D, max_cp, dev)
    st = _lib.cpattn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                         _ptr(cu_seqlens), _ptr(cp_size), B, T, int(max_seqlen), int(max_cp),
                         H, D, float(softmax_scale), 1 if causal else 0, _ptr(grads[0]),
                         _ptr(grads[1]), _ptr(grads[2]), _ptr(workspace), workspace.numel(),
                         _stream(stream))
    _check(st, "cpattn_bwd")
    return tuple(grads)


# -------------------------------------------------------- DCP data movement --

def select_cu(cu_seqlens, ids, *, stream=None):
    """``cpattn_select_cu``: cu_seqlens of the packed selection of samples
    ``ids`` (device int32).  Returns ``(pack_cu, status)`` (device int32
    tensors; status 0 when every id is valid)."""
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    _need(ids, "ids", torch.int32, cu_seqlens.device)
    n = ids.numel()
    pack_cu = torch.empty(n + 1, dtype=torch.int32, device=cu_seqlens.device)
    status = torch.empty(1, dtype=torch.int32, device=cu_seqlens.device)
    st = _lib.cpattn_select_cu(_ptr(cu_seqlens), cu_seqlens.numel() - 1, _ptr(ids), n,
                               _ptr(pack_cu), _ptr(status), _stream(stream))
    _check(st, "cpattn_select_cu")
    return pack_cu, status


def permute_samples(src, orig_cu, pack_cu, ids, status, *, gather, dst, stream=None):
    """``cpattn_permute_samples`` on token-major tensors (``[T, ...]``, rows
    contiguous): ``gather=True`` copies samples ``ids`` of the original
    ``src`` into the packed ``dst``; ``gather=False`` copies the packed
    ``src`` back into the original ``dst``."""
    if src.dtype != dst.dtype or src.shape[1:] != dst.shape[1:]:
        raise ValueError("src and dst must have the same dtype and row shape")
    if not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("src and dst must be contiguous")
    row_bytes = src.element_size() * (src[0].numel() if src.shape[0] else dst[0].numel())
    st = _lib.cpattn_permute_samples(_ptr(src), _ptr(orig_cu), orig_cu.numel() - 1,
                                     _ptr(pack_cu), _ptr(ids), ids.numel(), int(row_bytes),
                                     1 if gather else 0, _ptr(dst), _ptr(status),
                                     _stream(stream))
    _check(st, "cpattn_permute_samples")
    return dst


def dcp_fwd(q, k, v, cu_seqlens, plan_result, *, max_cp, softmax_scale=None, causal=True,
            stream=None):
    """The forward run the dynamic-CP way on one device: for every micro-batch
    of ``plan_result`` (from :func:`plan` on the same lengths), select its
    samples into packed arrays (``cpattn_select_cu``, ``cpattn_permute_samples``),
    run ``cpattn_fwd`` at the planned CP sizes, and restore O and LSE to the
    original sample order.  Returns ``(out, lse)`` in the original order."""
    dev = _fwd_common(q, k, v, cu_seqlens, None)
    T, H, D = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    mb = np.asarray(plan_result["micro_batch"])
    order = np.asarray(plan_result["order"])
    cps = np.asarray(plan_result["cp_size"])
    lengths = np.diff(cu_seqlens.cpu().numpy())
    for m in range(int(plan_result["num_micro_batches"])):
        sel = [int(b) for b in order if mb[b] == m]
        ids = torch.tensor(sel, dtype=torch.int32, device=dev)
        pack_cu, status = select_cu(cu_seqlens, ids, stream=stream)
        rows = int(sum(lengths[b] for b in sel))
        packed = []
        for x in (q, k, v):
            buf = torch.empty((rows, H, D), dtype=x.dtype, device=dev)
            permute_samples(x, cu_seqlens, pack_cu, ids, status, gather=True, dst=buf,
                            stream=stream)
            packed.append(buf)
        cp_m = torch.tensor([int(cps[b]) for b in sel], dtype=torch.int32, device=dev)
        o_m, l_m = fwd(*packed, pack_cu, cp_m, max_seqlen=int(max(lengths[b] for b in sel)),
                       max_cp=max_cp, softmax_scale=softmax_scale, causal=causal,
                       stream=stream)
        permute_samples(o_m, cu_seqlens, pack_cu, ids, status, gather=False, dst=out,
                        stream=stream)
        permute_samples(l_m, cu_seqlens, pack_cu, ids, status, gather=False, dst=lse,
                        stream=stream)
    return out, lse


# ---------------------------------------------------------------- Ulysses --

def ulysses_layout(src, sp_size, *, to_head_groups, dst=None, stream=None):
    """``cpattn_ulysses_layout``.  ``to_head_groups=True``: ``src [T, H, ...]``
    -> ``[P, T, H / P, ...]``; ``False``: ``src [P, T, H / P, ...]`` ->
    ``[T, H, ...]`` (P = ``sp_size``).  Any dtype; contiguous CUDA tensors."""
    P = int(sp_size)
    if src.device.type != "cuda" or not src.is_contiguous():
        raise ValueError("src must be a contiguous CUDA tensor")
    if to_head_groups:
        if src.dim() < 2 or src.shape[1] % P != 0:
            raise ValueError("src must be [T, H, ...] with H divisible by sp_size")
        T, H, rest = src.shape[0], src.shape[1], tuple(src.shape[2:])
        shape = (P, T, H // P) + rest
    else:
        if src.dim() < 3 or src.shape[0] != P:
            raise ValueError("src must be [sp_size, T, H / sp_size, ...]")
        T, H, rest = src.shape[1], P * src.shape[2], tuple(src.shape[3:])
        shape = (T, H) + rest
    if dst is None:
        dst = torch.empty(shape, dtype=src.dtype, device=src.device)
    elif (tuple(dst.shape) != shape or dst.dtype != src.dtype or dst.device != src.device
          or not dst.is_contiguous()):
        raise ValueError("dst must be a contiguous %s tensor of shape %s" % (src.dtype, shape))
    head_bytes = src.element_size() * int(np.prod(rest, dtype=np.int64))
    st = _lib.cpattn_ulysses_layout(_ptr(src), _ptr(dst), T, H, head_bytes, P,
                                    1 if to_head_groups else 0, _stream(stream))
    _check(st, "cpattn_ulysses_layout")
    return dst


def ulysses_seqlens(cu_seqlens, cp_size, sp_size, num_tokens, *, stream=None):
    """``cpattn_ulysses_seqlens``: cu_seqlens and cp_size of the head-group
    layout as one packed batch of ``sp_size * B`` samples."""
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    dev = cu_seqlens.device
    B = cu_seqlens.numel() - 1
    if cp_size is not None:
        _need(cp_size, "cp_size", torch.int32, dev, (B,))
    P = int(sp_size)
    cu_out = torch.empty(P * B + 1, dtype=torch.int32, device=dev)
    cp_out = torch.empty(P * B, dtype=torch.int32, device=dev)
    st = _lib.cpattn_ulysses_seqlens(_ptr(cu_seqlens), _ptr(cp_size), B, int(num_tokens), P,
                                     _ptr(cu_out), _ptr(cp_out), _stream(stream))
    _check(st, "cpattn_ulysses_seqlens")
    return cu_out, cp_out


def ulysses_fwd(q, k, v, cu_seqlens, sp_size, cp_size=None, *, max_seqlen, max_cp=None,
                softmax_scale=None, causal=True, stream=None):
    """Attention the Ulysses way on one device: Q, K, V to the head-group
    layout, one ``cpattn_fwd`` over all P groups (each group a copy of the
    batch with H / P heads; ``cp_size`` adds ring CP inside every group),
    then O and LSE back to the sequence layout.  Returns ``(out, lse)``."""
    _fwd_common(q, k, v, cu_seqlens, cp_size)
    T, H, D = q.shape
    P = int(sp_size)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    grouped = [ulysses_layout(x, P, to_head_groups=True, stream=stream).view(P * T, H // P, D)
               for x in (q, k, v)]
    cu_g, cp_g = ulysses_seqlens(cu_seqlens, cp_size, P, T, stream=stream)
    if max_cp is None:
        max_cp = 1 if cp_size is None or cp_size.numel() == 0 else int(cp_size.max().item())
    o_g, l_g = fwd(*grouped, cu_g, cp_g, max_seqlen=max_seqlen, max_cp=max_cp,
                   softmax_scale=softmax_scale, causal=causal, stream=stream)
    out = ulysses_layout(o_g.view(P, T, H // P, D), P, to_head_groups=False, stream=stream)
    lse = ulysses_layout(l_g.view(P, T, H // P), P, to_head_groups=False, stream=stream)
    return out, lse


# -------------------------------------------------------------- decode CP --

def _decode_check(q, k, v, cu_seqlens):
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("q must be [B, H, D] and k, v [T, H, D]")
    dev = q.device
    _need(k, "k", torch.bfloat16, dev)
    _need(v, "v", torch.bfloat16, dev, k.shape)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev, (q.shape[0] + 1,))
    if tuple(k.shape[1:]) != tuple(q.shape[1:]):
        raise ValueError("q and k must share H and D")
    return dev


def decode_partials(q, k, v, cu_seqlens, *, cp, softmax_scale=None, stream=None):
    """``cpattn_decode_partials``: returns ``(o_steps [cp, B, H, D] fp32,
    lse_steps [cp, B, H] fp32)``."""
    dev = _decode_check(q, k, v, cu_seqlens)
    B, H, D = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    o_s = torch.empty((cp, B, H, D), dtype=torch.float32, device=dev)
    l_s = torch.empty((cp, B, H), dtype=torch.float32, device=dev)
    st = _lib.cpattn_decode_partials(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), B,
                                     k.shape[0], H, D, float(softmax_scale), int(cp), _ptr(o_s),
                                     _ptr(l_s), _stream(stream))
    _check(st, "cpattn_decode_partials")
    return o_s, l_s


def merge_lse(o_steps, lse_steps, *, stream=None):
    """``cpattn_merge_lse`` over the leading axis of normalised partials
    ``o_steps [S, ..., D]`` and ``lse_steps [S, ...]``; returns ``(O, LSE)``."""
    _need(o_steps, "o_steps", torch.float32)
    _need(lse_steps, "lse_steps", torch.float32, o_steps.device)
    S, D = o_steps.shape[0], o_steps.shape[-1]
    rows = lse_steps[0].numel()
    out = torch.empty(o_steps.shape[1:], dtype=torch.float32, device=o_steps.device)
    lse = torch.empty(lse_steps.shape[1:], dtype=torch.float32, device=o_steps.device)
    st = _lib.cpattn_merge_lse(_ptr(o_steps), _ptr(lse_steps), S, rows, D, _ptr(out), _ptr(lse),
                               _stream(stream))
    _check(st, "cpattn_merge_lse")
    return out, lse


def decode(q, k, v, cu_seqlens, *, cp, softmax_scale=None, out=None, lse=None, workspace=None,
           stream=None):
    """``cpattn_decode``: decode-time CP attention; returns ``(out bf16 [B, H, D],
    lse fp32 [B, H])``."""
    dev = _decode_check(q, k, v, cu_seqlens)
    B, H, D = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    if workspace is None:
        n = _lib.cpattn_decode_workspace_size(B, H, D, int(cp))
        if n == 0:
            raise CpattnError(ERR_INVALID_ARG, "cpattn_decode_workspace_size")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    st = _lib.cpattn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), B, k.shape[0], H, D,
                            float(softmax_scale), int(cp), _ptr(out), _ptr(lse), _ptr(workspace),
                            workspace.numel(), _stream(stream))
    _check(st, "cpattn_decode")
    return out, lse


def merge(o_steps, m_steps, l_steps, *, out_o=None, out_m=None, out_l=None, stream=None):
    """Fold stored partials (``cpattn_merge``); returns ``(O / l, m, l)`` in fp32."""
    _need(o_steps, "o_steps", torch.float32)
    if o_steps.dim() != 4 or o_steps.device.type != "cuda":
        raise ValueError("o_steps must be a CUDA [S, T, H, D] tensor")
    S, T, H, D = o_steps.shape
    dev = o_steps.device
    _need(m_steps, "m_steps", torch.float32, dev, (S, T, H))
    _need(l_steps, "l_steps", torch.float32, dev, (S, T, H))
    if out_o is None:
        out_o = torch.empty((T, H, D), dtype=torch.float32, device=dev)
    if out_m is None:
        out_m = torch.empty((T, H), dtype=torch.float32, device=dev)
    if out_l is None:
        out_l = torch.empty((T, H), dtype=torch.float32, device=dev)
    _need(out_o, "out_o", torch.float32, dev, (T, H, D))
    _need(out_m, "out_m", torch.float32, dev, (T, H))
    _need(out_l, "out_l", torch.float32, dev, (T, H))
    st = _lib.cpattn_merge(_ptr(o_steps), _ptr(m_steps), _ptr(l_steps), S, T, H, D,
                           _ptr(out_o), _ptr(out_m), _ptr(out_l), _stream(stream))
    _check(st, "cpattn_merge")
    return out_o, out_m, out_l


def poll_error(workspace, stream=None):
    """Synchronise the stream and return the workspace's error word."""
    return int(_lib.cpattn_poll_error(_ptr(workspace), _stream(stream)))
