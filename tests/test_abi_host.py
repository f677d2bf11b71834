"""Host-only tests of the C ABI: the library loads, exports every entry point
declared in include/qmm.h, and reports argument errors before launching
anything. No test here makes a CUDA call that needs a GPU."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q():
    from bit_affine_quantized_group_gb300 import _build
    _build.build()
    import bit_affine_quantized_group_gb300 as q
    return q


def _header_functions():
    src = open(os.path.join(ROOT, "include", "qmm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(qmm_[a-z_]+)\s*\(", src, flags=re.M))


def test_header_declares_binding_exports(q):
    assert _header_functions() == set(q.EXPORTS)


def test_library_exports_every_declared_symbol(q):
    lib = ctypes.CDLL(q.LIB_PATH)
    for name in _header_functions():
        assert hasattr(lib, name), name


def test_status_strings(q):
    for st in range(8):
        assert q.status_string(st).startswith("QMM_")
    assert q.status_string(99) == "unknown qmm status"


GOOD = dict(K=5120, N=17408, bits=4, group=32, max_M=16, out_dtype="bf16", splits=0, max_banks=1)


@pytest.mark.parametrize("change,expect", [
    ({}, 0),
    ({"bits": 5}, 0), ({"bits": 6}, 0), ({"bits": 8}, 0), ({"group": 64}, 0),
    ({"bits": 3}, 0), ({"bits": 2}, 0), ({"bits": 7}, 2), ({"bits": 1}, 2), ({"group": 128}, 2), ({"group": 16}, 2),
    ({"bits": 0}, 1), ({"K": 0}, 1), ({"N": 0}, 1), ({"K": 5120 + 16}, 1),
    ({"max_M": 0}, 1), ({"max_M": 17}, 1), ({"splits": -1}, 1), ({"splits": 17}, 1),
    ({"max_banks": 0}, 1), ({"max_banks": 65}, 1),
    ({"K": 32 * 3, "bits": 4}, 2),                  # K*bits % 128 != 0
    ({"K": 32 * 2 * 3, "bits": 5}, 2),              # 5*192 = 960, not a multiple of 128
    ({"K": 32 * 34, "bits": 4, "group": 32}, 0),    # G = 34 even, 4352*4 % 128 == 0
    ({"K": 32 * 35, "bits": 8}, 2),                 # G odd
    ({"K": 2048, "group": 64, "splits": 4}, 0),     # 32 groups -> 4 chunks
    ({"K": 2048, "group": 64, "splits": 5}, 2),     # more slices than chunks
])
def test_validate_desc(q, change, expect):
    d = dict(GOOD)
    d.update(change)
    desc = q.make_desc(**d)
    assert q.validate_desc(desc) == expect


def test_out_dtype_codes(q):
    assert q.make_desc(**{**GOOD, "out_dtype": "f32"}).out_dtype == q.QMM_OUT_F32
    bad = q.make_desc(**GOOD)
    bad.out_dtype = 7
    assert q.validate_desc(bad) == q.QMM_ERR_INVALID_ARG
    assert q.lib.qmm_validate_desc(None) == q.QMM_ERR_INVALID_ARG


def test_workspace_bytes(q):
    d = q.make_desc(**GOOD)
    n = q.workspace_bytes(d)
    assert n > 0
    # splits = 1: only the error word (activations are staged in shared memory)
    n1 = q.workspace_bytes(q.make_desc(**{**GOOD, "splits": 1}))
    assert 0 < n1 < 1024 * 1024
    # splits = 0 (automatic) is sized for the largest automatic choice (here 20 chunks / 3 = 6)
    assert n >= n1 + 6 * 16 * 17408 * 4
    bad = q.make_desc(**{**GOOD, "bits": 7})
    assert q.workspace_bytes(bad) == 0
    # explicit slices need fp32 partials for max_banks * splits * max_M * N
    d2 = q.make_desc(K=17408, N=5120, bits=4, group=64, max_M=16, out_dtype="bf16", splits=8, max_banks=1)
    assert q.workspace_bytes(d2) >= 8 * 16 * 5120 * 4


def _args(**kw):
    a = dict(x=0x1000, M=4, w=[0x2000], s=[0x3000], b=[0x4000], K=5120, N=17408, bits=4, group=32, out=[0x5000])
    a.update(kw)
    return a


@pytest.mark.parametrize("kw,expect", [
    ({}, 0),
    ({"M": 0, "x": 0}, 0),                      # M = 0: no-op, x may be NULL
    ({"M": -1}, 1), ({"M": 17}, 1),
    ({"x": 0}, 1), ({"x": 0x1001}, 1),          # NULL / misaligned bf16
    ({"x": 0x1008}, 1),                         # x rows are bulk-copied: 16-byte alignment
    ({"w": [0]}, 1), ({"w": [0x2008]}, 1),      # packed rows need 16-byte alignment
    ({"s": [0x3004]}, 1), ({"b": [0]}, 1),      # G % 8 == 0 -> scales/biases 16-byte aligned
    ({"out": [0x5002]}, 0),                     # bf16 out: 2-byte alignment is enough
    ({"out": [0x5001]}, 1),
    ({"K": 4096}, 3), ({"N": 17409}, 3), ({"bits": 8}, 3), ({"group": 64}, 3),
    ({"w": [0x2000, 0x2100], "s": [0x3000, 0x3100], "b": [0x4000, 0x4100], "out": [0x5000, 0x5100]}, 1),
])
def test_check_forward_args(q, kw, expect):
    desc = q.make_desc(**GOOD)
    a = _args(**kw)
    st = q.check_forward_args(desc, a["x"], a["M"], a["w"], a["s"], a["b"], a["K"], a["N"], a["bits"],
                              a["group"], a["out"])
    assert st == expect


def test_check_forward_args_banks_and_f32(q):
    desc = q.make_desc(**{**GOOD, "max_banks": 4, "out_dtype": "f32"})
    ptr4 = lambda base: [base + 0x100 * i for i in range(4)]
    st = q.check_forward_args(desc, 0x1000, 3, ptr4(0x2000), ptr4(0x3000), ptr4(0x4000), 5120, 17408, 4, 32,
                              ptr4(0x5000))
    assert st == 0
    st = q.check_forward_args(desc, 0x1000, 3, ptr4(0x2000), ptr4(0x3000), ptr4(0x4000), 5120, 17408, 4, 32,
                              [0x5000, 0x5100, 0x5202, 0x5300])   # f32 out needs 4-byte alignment
    assert st == 1
    five = [0x2000 + 0x100 * i for i in range(5)]
    assert q.check_forward_args(desc, 0x1000, 3, five, five, five, 5120, 17408, 4, 32, five) == 1
    assert q.check_forward_args(None if False else desc, 0x1000, 3, None, [0x3000], [0x4000], 5120, 17408, 4, 32,
                                [0x5000]) == 1


def test_scale_alignment_relaxed_when_groups_not_multiple_of_8(q):
    # K/group = 34 groups: scale rows are only 4-byte aligned, so 4-byte pointers are accepted
    desc = q.make_desc(K=32 * 34, N=100, bits=4, group=32, max_M=8, out_dtype="bf16")
    st = q.check_forward_args(desc, 0x1000, 2, [0x2000], [0x3004], [0x4004], 32 * 34, 100, 4, 32, [0x5000])
    assert st == 0
    st = q.check_forward_args(desc, 0x1000, 2, [0x2000], [0x3002], [0x4004], 32 * 34, 100, 4, 32, [0x5000])
    assert st == 1


def test_null_plan_and_handles(q):
    lib = q.lib
    assert lib.qmm_forward(None, None, 1, None, None, None, 5120, 17408, 4, 32, None, None) == q.QMM_ERR_INVALID_ARG
    assert lib.qmm_plan_get_info(None, None) == q.QMM_ERR_INVALID_ARG
    assert lib.qmm_plan_error(None, None) == q.QMM_ERR_INVALID_ARG
    lib.qmm_destroy(None)   # accepted
    # invalid descriptors are rejected before any device query
    out = ctypes.c_void_p(1)
    bad = q.make_desc(**{**GOOD, "bits": 7})
    assert lib.qmm_plan(ctypes.byref(out), ctypes.byref(bad), None, 0) == q.QMM_ERR_UNSUPPORTED
    assert out.value is None
    assert lib.qmm_plan(None, ctypes.byref(bad), None, 0) == q.QMM_ERR_INVALID_ARG


def test_unpack_codes_argument_errors(q):
    lib = q.lib
    assert lib.qmm_unpack_codes(None, 64, 1, 7, None, None) == q.QMM_ERR_UNSUPPORTED
    assert lib.qmm_unpack_codes(None, 48, 1, 4, None, None) == q.QMM_ERR_INVALID_ARG
    assert lib.qmm_unpack_codes(None, 64, 1, 4, None, None) == q.QMM_ERR_INVALID_ARG
    assert lib.qmm_unpack_codes(None, 64, 0, 4, None, None) == q.QMM_OK


def test_plan_without_device_reports_cuda_error(q):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    out = ctypes.c_void_p()
    d = q.make_desc(**GOOD)
    assert q.lib.qmm_plan(ctypes.byref(out), ctypes.byref(d), None, 0) == q.QMM_ERR_CUDA
    assert out.value is None
