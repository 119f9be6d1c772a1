"""Python binding of the cpattn C ABI (``include/cpattn.h``).

Argument marshalling only: tensors are checked for dtype, device, layout and
contiguity, then their device pointers are handed to ``libcpattn.so`` together
with PyTorch's current CUDA stream.  Every step of the computation runs in the
library's kernels; there is no fallback.  Importing this module raises
``ImportError`` when the library has not been built (``build.build()``).
"""

from __future__ import annotations

import ctypes
import functools
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
ERR_DEVICE_BOUNDS = 7
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


# ---------------------------------------------------------------- tracing --
# NVTX ranges around every public call (named after the C entry point), for
# profilers that filter or group by range (e.g. ncu --nvtx --nvtx-include
# "cpattn_fwd/").  Off by default -- a disabled range costs one flag test --
# and switched on by set_tracing(True) or CPATTN_NVTX=1 in the environment.
_TRACE = os.environ.get("CPATTN_NVTX", "") not in ("", "0")


def set_tracing(enabled):
    """Switch the NVTX ranges around the public calls on or off."""
    global _TRACE
    _TRACE = bool(enabled)


def tracing():
    return _TRACE


def _traced(name):
    def deco(fn):
        @functools.wraps(fn)
        def wrapper(*args, **kwargs):
            if not _TRACE:
                return fn(*args, **kwargs)
            torch.cuda.nvtx.range_push(name)
            try:
                return fn(*args, **kwargs)
            finally:
                torch.cuda.nvtx.range_pop()
        return wrapper
    return deco


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

@_traced("cpattn_plan")
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


def _max_cp(cp_size, max_cp):
    """``max_cp`` as given; 1 when there are no CP sizes.  With device CP sizes
    and no ``max_cp`` the call is refused: finding their maximum would read
    device memory and synchronise the host with the stream."""
    if max_cp is not None:
        return int(max_cp)
    if cp_size is None or cp_size.numel() == 0:
        return 1
    raise ValueError("max_cp is required when cp_size is given (an upper bound on the CP "
                     "sizes, e.g. the planner's max_cp)")


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


@_traced("cpattn_fwd")
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
    max_cp = _max_cp(cp_size, max_cp)
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


@_traced("cpattn_fwd_noalloc")
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
    max_cp = _max_cp(cp_size, max_cp)
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


@_traced("cpattn_fwd_partials")
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


@_traced("cpattn_bwd")
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
    max_cp = _max_cp(cp_size, max_cp)
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

@_traced("cpattn_select_cu")
def select_cu(cu_seqlens, ids, *, out=None, status=None, stream=None):
    """``cpattn_select_cu``: cu_seqlens of the packed selection of samples
    ``ids`` (device int32).  Returns ``(pack_cu, status)`` (device int32
    tensors, ``out`` / ``status`` if given; status 0 when every id is valid)."""
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    _need(ids, "ids", torch.int32, cu_seqlens.device)
    n = ids.numel()
    dev = cu_seqlens.device
    if out is None:
        out = torch.empty(n + 1, dtype=torch.int32, device=dev)
    else:
        _need(out, "out", torch.int32, dev, (n + 1,))
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=dev)
    else:
        _need(status, "status", torch.int32, dev, (1,))
    pack_cu = out
    st = _lib.cpattn_select_cu(_ptr(cu_seqlens), cu_seqlens.numel() - 1, _ptr(ids), n,
                               _ptr(pack_cu), _ptr(status), _stream(stream))
    _check(st, "cpattn_select_cu")
    return pack_cu, status


@_traced("cpattn_permute_samples")
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


class DcpForward:
    """The forward run the dynamic-CP way on one device, prepared once per
    plan ("Dynamic Context Parallelism (DCP)": every rank sees the same
    samples, selects its own, and the output order is restored afterwards).

    For every micro-batch of ``plan_result`` (from :func:`plan` on the host
    lengths ``seqlens``) a call selects the micro-batch's samples into packed
    arrays (``cpattn_select_cu``, ``cpattn_permute_samples``), runs
    ``cpattn_fwd`` at the planned CP sizes and writes O and LSE back to the
    samples' original rows.  Everything a call needs from the plan is worked
    out here on the host and uploaded once; the packed buffers and the
    forward's workspace are allocated once at the largest micro-batch.  A
    call therefore only enqueues kernels: it never reads device memory, so it
    does not wait for the stream.  Calls on one object share its buffers:
    run them in stream order (one stream), not concurrently.
    """

    def __init__(self, seqlens, plan_result, *, num_heads, head_dim, max_cp, device=None):
        lengths = [int(x) for x in seqlens]
        dev = torch.device(device or "cuda")
        mb = np.asarray(plan_result["micro_batch"])
        order = np.asarray(plan_result["order"])
        cps = np.asarray(plan_result["cp_size"])
        if len(mb) != len(lengths):
            raise ValueError("plan_result does not match seqlens")
        self.H, self.D, self.max_cp, self.dev = int(num_heads), int(head_dim), int(max_cp), dev
        self.B, self.T = len(lengths), sum(lengths)
        self.micro = []
        ids_all, cps_all = [], []
        for m in range(int(plan_result["num_micro_batches"])):
            sel = [int(b) for b in order if mb[b] == m]
            if not sel:
                continue
            self.micro.append(dict(off=len(ids_all), n=len(sel),
                                   rows=sum(lengths[b] for b in sel),
                                   max_seqlen=max(max(lengths[b] for b in sel), 1)))
            ids_all += sel
            cps_all += [int(cps[b]) for b in sel]
        if any(c > self.max_cp for c in cps_all):
            raise ValueError("a planned CP size exceeds max_cp")
        host = torch.tensor([ids_all, cps_all], dtype=torch.int32).reshape(2, -1)
        if dev.type == "cuda":
            host = host.pin_memory()
        dev_arr = host.to(dev, non_blocking=True)
        self.ids, self.cps = dev_arr[0], dev_arr[1]
        self.pack_cu = torch.empty(len(ids_all) + len(self.micro), dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        rows = max([x["rows"] for x in self.micro] + [0])
        nmax = max([x["n"] for x in self.micro] + [0])
        self.packed = [torch.empty((rows, self.H, self.D), dtype=torch.bfloat16, device=dev)
                       for _ in range(4)]   # Q, K, V, O
        self.packed_lse = torch.empty((rows, self.H), dtype=torch.float32, device=dev)
        self.workspace = alloc_workspace(rows, nmax, self.H, self.D, self.max_cp, MODE_FUSED,
                                         dev)
        self._host = host  # keeps the pinned source of the upload alive

    @_traced("cpattn.DcpForward")
    def __call__(self, q, k, v, cu_seqlens, *, softmax_scale=None, causal=True, out=None,
                 lse=None, stream=None):
        """Returns ``(out, lse)`` in the original sample order."""
        dev = _fwd_common(q, k, v, cu_seqlens, None)
        T, H, D = q.shape
        if (T, H, D) != (self.T, self.H, self.D) or cu_seqlens.numel() != self.B + 1:
            raise ValueError("q, k, v, cu_seqlens do not match the planned batch")
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        for i, x in enumerate(self.micro):
            ids = self.ids[x["off"]:x["off"] + x["n"]]
            cp_m = self.cps[x["off"]:x["off"] + x["n"]]
            pack_cu = self.pack_cu[x["off"] + i:x["off"] + i + x["n"] + 1]
            select_cu(cu_seqlens, ids, out=pack_cu, status=self.status, stream=stream)
            rows = x["rows"]
            pq, pk, pv, po = (b[:rows] for b in self.packed)
            pl = self.packed_lse[:rows]
            for src, dst in ((q, pq), (k, pk), (v, pv)):
                permute_samples(src, cu_seqlens, pack_cu, ids, self.status, gather=True,
                                dst=dst, stream=stream)
            fwd(pq, pk, pv, pack_cu, cp_m, max_seqlen=x["max_seqlen"], max_cp=self.max_cp,
                softmax_scale=softmax_scale, causal=causal, out=po, lse=pl,
                workspace=self.workspace, stream=stream)
            permute_samples(po, cu_seqlens, pack_cu, ids, self.status, gather=False, dst=out,
                            stream=stream)
            permute_samples(pl, cu_seqlens, pack_cu, ids, self.status, gather=False, dst=lse,
                            stream=stream)
        return out, lse


@_traced("cpattn.dcp_fwd")
def dcp_fwd(q, k, v, cu_seqlens, plan_result, *, seqlens, max_cp, softmax_scale=None,
            causal=True, stream=None):
    """One-shot :class:`DcpForward`: plan-derived buffers built for this call
    (``seqlens`` are the host lengths the plan was made from).  Returns
    ``(out, lse)`` in the original sample order."""
    T, H, D = q.shape
    run = DcpForward(seqlens, plan_result, num_heads=H, head_dim=D, max_cp=max_cp,
                     device=q.device)
    return run(q, k, v, cu_seqlens, softmax_scale=softmax_scale, causal=causal, stream=stream)


# ---------------------------------------------------------------- Ulysses --

@_traced("cpattn_ulysses_layout")
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


@_traced("cpattn_ulysses_seqlens")
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


@_traced("cpattn.ulysses_fwd")
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
    max_cp = _max_cp(cp_size, max_cp)
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


@_traced("cpattn_decode_partials")
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


@_traced("cpattn_merge_lse")
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


@_traced("cpattn_decode")
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


@_traced("cpattn_merge")
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
