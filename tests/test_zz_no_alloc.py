"""qmm_forward_noalloc: the forward for callers that cannot allocate device
memory (code running while another component owns the allocator, loops that
forbid allocation after start-up, plug-in hosts that only hand over tensors).

It keeps its device scratch (the kernels' error word and the fp32 partial sums
of K-sliced projections) in a static device array instead of a plan's
workspace. These tests call it through the C ABI and check, on calls in a row:
its output against the oracle (the same tolerances as the other parity tests)
and bitwise against qmm_forward with the same K-slice count; that the free
device memory does not change across calls; that calls of different row
counts back to back share the array correctly; and that argument errors are
reported before the device is touched. This file is collected last so that a
failure here comes after every other test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import datagen

SCRATCH = 4 << 20
ERR_AREA = 256


@pytest.fixture(scope="module")
def q():
    from bit_affine_quantized_group_gb300 import _build
    _build.build()
    import bit_affine_quantized_group_gb300 as q
    return q


def _call(q, x, M, w, s, b, K, N, bits, group, out_dtype, out, stream=None):
    return q.lib.qmm_forward_noalloc(ctypes.c_void_p(x), M, ctypes.c_void_p(w), ctypes.c_void_p(s),
                                     ctypes.c_void_p(b), K, N, bits, group, out_dtype, ctypes.c_void_p(out),
                                     ctypes.c_void_p(stream) if stream else None)


def test_noalloc_argument_errors_before_touching_the_device(q):
    """Every rejected call below fails its host-side checks; none reaches the device."""
    assert _call(q, 0, 4, 0x2000, 0x3000, 0x4000, 2048, 64, 4, 64, q.QMM_OUT_F32, 0x5000) == q.QMM_ERR_INVALID_ARG
    assert _call(q, 0x1008, 4, 0x2000, 0x3000, 0x4000, 2048, 64, 4, 64, q.QMM_OUT_F32, 0x5000) == \
        q.QMM_ERR_INVALID_ARG                                   # x must be 16-byte aligned
    assert _call(q, 0x1000, 17, 0x2000, 0x3000, 0x4000, 2048, 64, 4, 64, q.QMM_OUT_F32, 0x5000) == \
        q.QMM_ERR_INVALID_ARG
    assert _call(q, 0x1000, 4, 0x2008, 0x3000, 0x4000, 2048, 64, 4, 64, q.QMM_OUT_F32, 0x5000) == \
        q.QMM_ERR_INVALID_ARG                                   # packed rows need 16-byte alignment
    assert _call(q, 0x1000, 4, 0x2000, 0x3000, 0x4000, 2048, 64, 7, 64, q.QMM_OUT_F32, 0x5000) == \
        q.QMM_ERR_UNSUPPORTED
    assert _call(q, 0x1000, 4, 0x2000, 0x3000, 0x4000, 2048, 64, 4, 64, 9, 0x5000) == q.QMM_ERR_INVALID_ARG
    assert _call(q, 0, 0, 0, 0, 0, 2048, 64, 4, 64, q.QMM_OUT_F32, 0) == q.QMM_OK   # M = 0: no-op


def _device_inputs(seed, M, K, N, bits, group):
    from tests._gpu import dev_tensors
    inp = datagen.gen_qmm(seed, M, K, N, bits, group)
    return inp, dev_tensors(inp)


def _check(q, y, y_ref, out_dtype):
    from tests._gpu import check
    check(y, y_ref, out_dtype)


def _plan_out(q, plan, x, w, s, b, M):
    import torch
    out = torch.empty((M, plan.N), dtype=plan.out_dtype, device="cuda")
    q.forward(plan, x[:M], w, s, b, out)
    torch.cuda.synchronize()
    return out


CASES = [
    # (M, K, N, bits, group, out_dtype)
    (4, 2048, 2048, 4, 64, "f32"),
    (9, 5120, 1000, 6, 32, "bf16"),
    (16, 1024, 520, 8, 32, "bf16"),
    (8, 5120, 17408, 4, 32, "bf16"),     # 112-128 rows a CTA: the wide consumer layout
    (8, 17408, 5120, 4, 64, "bf16"),     # long K: the automatic choice slices K, partials in the static array
    (16, 16384, 20480, 4, 64, "bf16"),   # partials of the automatic choice exceed the array: fewer slices
]


@pytest.mark.gpu
@pytest.mark.parametrize("M,K,N,bits,group,out_dtype", CASES)
def test_noalloc_matches_oracle_and_plan_twice(q, M, K, N, bits, group, out_dtype):
    import torch
    from tests._gpu import to_f64
    import oracle
    oracle.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    inp, (x, w, s, b) = _device_inputs(4242 + bits + M + K, M, K, N, bits, group)
    torch.cuda.synchronize()
    if M * K * N <= 2 ** 31:
        cols = np.arange(N, dtype=np.int64)
    else:
        rng = np.random.default_rng(5)
        cols = np.unique(np.concatenate([np.arange(64), np.arange(N - 64, N), rng.choice(N, 512, replace=False)]))
    y_ref = oracle.qmm_f64_cols(inp.x, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group, cols)
    code = q.QMM_OUT_F32 if out_dtype == "f32" else q.QMM_OUT_BF16
    outs = []
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.float32 if out_dtype == "f32" else torch.bfloat16,
                         device="cuda")
        st = _call(q, x.data_ptr(), M, w.data_ptr(), s.data_ptr(), b.data_ptr(), K, N, bits, group, code,
                   out.data_ptr())
        assert st == q.QMM_OK, q.status_string(st)
        torch.cuda.synchronize()
        y = to_f64(out)
        assert np.all(np.isfinite(y))
        _check(q, y[:, cols], y_ref, out_dtype)
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
    # bitwise equal to qmm_forward with the K-slice count the call used: one of
    # the counts whose partial sums fit the static array
    fits = [sp for sp in range(1, 9) if sp == 1 or ERR_AREA + sp * M * N * 4 <= SCRATCH]
    chunks = (K // group + 7) // 8
    matched = []
    for sp in fits:
        if sp > chunks:
            continue
        plan = q.Plan(K, N, bits, group, max_M=M, out_dtype=out_dtype, splits=sp)
        if torch.equal(_plan_out(q, plan, x, w, s, b, M), outs[0]):
            matched.append(sp)
        assert plan.error_flags() == 0
        plan.close()
    assert matched, "no K-slice count of qmm_forward reproduces the no-allocation result"


@pytest.mark.gpu
def test_noalloc_allocates_nothing_and_shares_the_scratch_across_row_counts(q):
    """After a first call (device set-up), calls of 16, 4 and 16 rows back to
    back on one stream leave the free device memory unchanged and each matches
    the oracle."""
    import torch
    from tests._gpu import to_f64
    import oracle
    oracle.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    K, N, bits, group = 17408, 2048, 4, 64          # long K: K-sliced, partials in the array
    inp, (x, w, s, b) = _device_inputs(777, 16, K, N, bits, group)
    y_ref = oracle.qmm_f64(inp.x, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    outs = {M: torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for M in (4, 16)}
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    for M in (16, 4):                                # set-up and warm-up of both row tiles
        assert _call(q, x.data_ptr(), M, w.data_ptr(), s.data_ptr(), b.data_ptr(), K, N, bits, group,
                     q.QMM_OUT_BF16, outs[M].data_ptr(), stream.cuda_stream) == q.QMM_OK
    results = [(M, torch.empty((M, N), dtype=torch.bfloat16, device="cuda")) for M in (16, 4, 16)]
    for _, out in results:
        out.fill_(float("nan"))
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for M, out in results:
        assert _call(q, x.data_ptr(), M, w.data_ptr(), s.data_ptr(), b.data_ptr(), K, N, bits, group,
                     q.QMM_OUT_BF16, out.data_ptr(), stream.cuda_stream) == q.QMM_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    # every tensor was allocated before free0 was read: the calls themselves
    # must leave the device's free memory exactly as it was
    assert free1 == free0, (free0, free1)
    for M, out in results:
        _check(q, to_f64(out), y_ref[:M], "bf16")
    assert torch.equal(results[0][1], results[2][1])
