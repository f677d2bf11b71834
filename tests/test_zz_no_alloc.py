"""qmm_forward_noalloc: the forward for callers that cannot allocate device
memory (code running while another component owns the allocator, loops that
forbid allocation after start-up, plug-in hosts that only hand over tensors).

It keeps its per-call activation staging in a static device array instead of
a plan's workspace. These tests call it through the C ABI and check that two
calls in a row match qmm_forward (same tolerance as the other parity tests),
and that a call too large for the static scratch is refused up front. This
file is collected last so that a failure here comes after every other test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import datagen


@pytest.fixture(scope="module")
def q():
    from bit_affine_quantized_group_gb300 import _build
    _build.build()
    import bit_affine_quantized_group_gb300 as q
    return q


def _call(q, x, M, w, s, b, K, N, bits, group, out_dtype, out):
    return q.lib.qmm_forward_noalloc(ctypes.c_void_p(x), M, ctypes.c_void_p(w), ctypes.c_void_p(s),
                                     ctypes.c_void_p(b), K, N, bits, group, out_dtype, ctypes.c_void_p(out), None)


def test_noalloc_rejects_oversized_staging_before_touching_the_device(q):
    # 8-bit codes, groups of 64, 16 rows: the largest K that fits is 122368
    K, N, bits, group = 131072, 64, 8, 64
    st = _call(q, 0x1000, 16, 0x2000, 0x3000, 0x4000, K, N, bits, group, q.QMM_OUT_BF16, 0x5000)
    assert st == q.QMM_ERR_SCRATCH_LIMIT
    assert "scratch" in q.status_string(st)
    # ordinary argument errors are reported the same way as qmm_forward's
    assert _call(q, 0, 4, 0x2000, 0x3000, 0x4000, 2048, 64, 4, 64, q.QMM_OUT_F32, 0x5000) == q.QMM_ERR_INVALID_ARG
    assert _call(q, 0x1000, 17, 0x2000, 0x3000, 0x4000, 2048, 64, 4, 64, q.QMM_OUT_F32, 0x5000) == q.QMM_ERR_INVALID_ARG
    assert _call(q, 0x1000, 4, 0x2000, 0x3000, 0x4000, 2048, 64, 7, 64, q.QMM_OUT_F32, 0x5000) == q.QMM_ERR_UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("M,K,N,bits,group,out_dtype", [
    (4, 2048, 2048, 4, 64, "f32"),
    (9, 5120, 1000, 6, 32, "bf16"),
    (16, 1024, 520, 8, 32, "bf16"),
])
def test_noalloc_matches_plan_forward_twice(q, M, K, N, bits, group, out_dtype):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tests._gpu import dev_tensors, to_f64
    from tests._helpers import bf16_ulp
    inp = datagen.gen_qmm(4242 + bits + M, M, K, N, bits, group)
    x, w, s, b = dev_tensors(inp)
    plan = q.Plan(K, N, bits, group, max_M=M, out_dtype=out_dtype, splits=1)
    ref = torch.empty((M, N), dtype=plan.out_dtype, device="cuda")
    q.forward(plan, x, w, s, b, ref)
    torch.cuda.synchronize()
    y_ref = to_f64(ref)
    code = q.QMM_OUT_F32 if out_dtype == "f32" else q.QMM_OUT_BF16
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=plan.out_dtype, device="cuda")
        st = _call(q, x.data_ptr(), M, w.data_ptr(), s.data_ptr(), b.data_ptr(), K, N, bits, group, code,
                   out.data_ptr())
        assert st == q.QMM_OK, q.status_string(st)
        torch.cuda.synchronize()
        y = to_f64(out)
        scale = float(np.max(np.abs(y_ref)))
        if out_dtype == "f32":
            assert float(np.max(np.abs(y - y_ref))) <= 2e-3 * scale
        else:
            assert np.all(np.abs(y - y_ref) <= bf16_ulp(y_ref) + 1e-3 * scale)
