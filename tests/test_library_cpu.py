"""Host-side checks of libcpattn.so that need no GPU.

* the library loads and exports every function ``include/cpattn.h`` declares;
* ``cpattn_plan`` (C++) is bit-exact with the oracle planner (Python) on the
  golden plans, the packed-16K and 256-sample workloads, and 10^4 random
  small instances;
* argument errors come back as status codes before any device work.
"""

import ctypes
import json
import os
import re

import numpy as np
import pytest

from long_context_gb300 import build as lib_build
from long_context_gb300 import workloads
from oracle import planner as op

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cp():
    lib_build.build()
    from long_context_gb300 import cpattn
    return cpattn


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "cpattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(cpattn_[a-z_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("cpattn_plan", "cpattn_fwd", "cpattn_merge",
                     "cpattn_fwd_workspace_size", "cpattn_poll_error"):
        assert required in names


def test_library_exports_every_declared_symbol(cp):
    lib = ctypes.CDLL(cp.library_path())
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(cp):
    assert cp.status_string(0) == "ok"
    assert "timed out" in cp.status_string(6)
    assert cp.version()[0] == 0


def _same_plan(c_plan, o_plan):
    for key in ("cp_size", "micro_batch", "first_rank", "order"):
        assert list(c_plan[key]) == list(o_plan[key]), key
    assert c_plan["num_micro_batches"] == o_plan["num_micro_batches"]
    assert c_plan["rank_load"].tolist() == o_plan["rank_load"]


def test_plan_golden(cp):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "dcp_plans.json")))
    for case in g["cases"]:
        r = cp.plan(case["seqlens"], case["world"], case["limit"], case["max_cp"])
        for key in ("cp_size", "micro_batch", "first_rank", "order"):
            assert list(r[key]) == case[key], (case["name"], key)
        assert r["num_micro_batches"] == case["num_micro_batches"]
        assert r["rank_load"].tolist() == case["rank_load"]
    for case in g["infeasible"]:
        with pytest.raises(cp.CpattnError) as e:
            cp.plan(case["seqlens"], case["world"], case["limit"], case["max_cp"])
        assert e.value.status == cp.ERR_PLAN_INFEASIBLE


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_plan_workloads_bit_exact(cp, seed):
    w = workloads.WORKLOADS["packed16k"]
    lens = workloads.packed_lengths(seed, w["budget"])
    _same_plan(cp.plan(lens, w["world"], w["limit"], w["max_cp"]),
               op.plan(lens, w["world"], w["limit"], w["max_cp"]))
    w = workloads.WORKLOADS["sweep256"]
    lens = workloads.uniform_lengths(seed, w["n"], w["lo"], w["hi"])
    _same_plan(cp.plan(lens, w["world"], w["limit"], w["max_cp"]),
               op.plan(lens, w["world"], w["limit"], w["max_cp"]))


def test_plan_random_bit_exact(cp):
    rng = np.random.default_rng(1234)
    for trial in range(10000):
        world = int(rng.choice([2, 4, 6, 8, 12, 16]))
        cands = [c for c in (1, 2, 4, 8, 16) if c <= world] + [world]
        max_cp = int(rng.choice(cands))
        limit = int(rng.integers(1, 64))
        n = int(rng.integers(0, 24))
        lens = [int(x) for x in rng.integers(0, limit * max_cp + 1, n)]
        _same_plan(cp.plan(lens, world, limit, max_cp), op.plan(lens, world, limit, max_cp))


def test_plan_argument_errors(cp):
    for args in [([1], 3, 10, 1), ([1], 0, 10, 1), ([1], 4, 0, 1), ([1], 4, 10, 3),
                 ([1], 4, 10, 8), ([-1], 4, 10, 2)]:
        with pytest.raises(cp.CpattnError) as e:
            cp.plan(*args)
        assert e.value.status == cp.ERR_INVALID_ARG
    r = cp.plan([], 2, 10, 2)
    assert r["num_micro_batches"] == 0


def test_workspace_size(cp):
    ws = cp.workspace_size(131072, 1, 16, 128, 4, cp.MODE_UNFUSED)
    partial_bytes = 4 * 131072 * 16 * (128 + 2) * 4
    assert partial_bytes <= ws <= partial_bytes + (1 << 20)
    assert cp.workspace_size(131072, 1, 16, 128, 4, cp.MODE_FUSED) < (1 << 20)
    with pytest.raises(cp.CpattnError):
        cp.workspace_size(10, 1, 1, 96, 1)  # head_dim 96 unsupported


def test_fwd_argument_errors_return_before_launch(cp):
    """Host-detected errors: nothing is enqueued, so no GPU is needed."""
    lib = ctypes.CDLL(cp.library_path())
    f = lib.cpattn_fwd
    f.argtypes = cp._lib.cpattn_fwd.argtypes
    f.restype = ctypes.c_int
    buf = ctypes.create_string_buffer(4096 + 256)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    p = ctypes.c_void_p(base)
    # head_dim 96 -> unsupported
    assert f(p, p, p, p, None, 1, 8, 8, 1, 1, 96, 0.1, 1, 0, p, None, p, 4096, None) == 2
    # misaligned q -> invalid argument
    assert f(ctypes.c_void_p(base + 2), p, p, p, None, 1, 8, 8, 1, 1, 64, 0.1, 1, 0, p, None,
             p, 4096, None) == 1
    # non-positive scale
    assert f(p, p, p, p, None, 1, 8, 8, 1, 1, 64, 0.0, 1, 0, p, None, p, 4096, None) == 1
    # workspace too small
    assert f(p, p, p, p, None, 1, 8, 8, 1, 1, 64, 0.1, 1, 0, p, None, p, 16, None) == 3
    # bad mode
    assert f(p, p, p, p, None, 1, 8, 8, 1, 1, 64, 0.1, 1, 7, p, None, p, 4096, None) == 1
    m = lib.cpattn_merge
    m.argtypes = cp._lib.cpattn_merge.argtypes
    m.restype = ctypes.c_int
    assert m(p, p, p, 0, 8, 1, 128, p, p, p, None) == 1     # zero steps
    assert m(p, p, p, 2, 8, 1, 80, p, p, p, None) == 2      # head_dim 80


def test_ulysses_argument_errors_return_before_launch(cp):
    lib = ctypes.CDLL(cp.library_path())
    f = lib.cpattn_ulysses_layout
    f.argtypes = cp._lib.cpattn_ulysses_layout.argtypes
    f.restype = ctypes.c_int
    buf = ctypes.create_string_buffer(4096 + 256)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    a, b = ctypes.c_void_p(base), ctypes.c_void_p(base + 1024)
    assert f(a, b, 8, 6, 256, 4, 1, None) == 1             # H % P != 0
    assert f(a, b, 8, 8, 6, 8, 1, None) == 1               # chunk of 6 bytes
    assert f(a, a, 8, 8, 256, 4, 1, None) == 1             # src == dst
    assert f(a, b, 8, 8, 256, 4, 2, None) == 1             # bad direction
    assert f(a, b, 1 << 29, 8, 256, 8, 1, None) == 1       # T * P >= 2^31
    assert f(ctypes.c_void_p(base + 2), b, 8, 8, 256, 4, 1, None) == 1  # misaligned
    assert f(None, None, 0, 8, 256, 4, 1, None) == 0       # empty: nothing to do
    s = lib.cpattn_ulysses_seqlens
    s.argtypes = cp._lib.cpattn_ulysses_seqlens.argtypes
    s.restype = ctypes.c_int
    assert s(a, None, 2, 8, 0, b, None, None) == 1         # sp_size 0
    assert s(None, None, 2, 8, 2, b, None, None) == 1      # no cu_seqlens
    assert s(a, None, 2, 1 << 30, 4, b, None, None) == 1   # P T >= 2^31


def test_tracing_ranges_wrap_public_calls():
    """With tracing on, the planner call runs inside an NVTX range (pushed and
    popped around it, also when it raises) and returns the same result."""
    from long_context_gb300 import cpattn
    base = cpattn.plan([100, 5000, 30], 4, 4096, 4)
    was = cpattn.tracing()
    try:
        cpattn.set_tracing(True)
        traced = cpattn.plan([100, 5000, 30], 4, 4096, 4)
        with pytest.raises(cpattn.CpattnError):
            cpattn.plan([100, 50000], 4, 4096, 4)
    finally:
        cpattn.set_tracing(was)
    for key in ("cp_size", "micro_batch", "first_rank", "order"):
        assert list(traced[key]) == list(base[key])
    assert cpattn.plan.__name__ == "plan" and cpattn.fwd.__name__ == "fwd"
