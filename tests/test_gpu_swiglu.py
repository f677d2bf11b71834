"""Fused gate/up projection with the SwiGLU epilogue (qmm_forward_swiglu)
against the oracle's float64 silu(qmm(x, gate)) * qmm(x, up), over formats,
K slicing, rows and output types, in one main-kernel launch per call."""
from __future__ import annotations

import numpy as np
import pytest

import datagen
from tests._gpu import check, dev_tensors, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_affine_quantized_group_gb300 import _build
    _build.build()
    import bit_affine_quantized_group_gb300 as q
    return q


@pytest.fixture(scope="module")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.mark.parametrize("bits,group", [(4, 32), (6, 64), (8, 32), (2, 64), (5, 32)])
@pytest.mark.parametrize("splits", [1, 2, 0])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_swiglu_parity(q, oracle_mod, bits, group, splits, out_dtype):
    import torch
    G = 20
    K, N = G * group, 300
    gate = datagen.gen_qmm(700 + bits, 16, K, N, bits, group)
    up = datagen.gen_qmm(900 + bits, 16, K, N, bits, group)
    y_ref = oracle_mod.qmm_swiglu_f64(gate.x, gate.words[0], gate.scales[0], gate.biases[0],
                                      up.words[0], up.scales[0], up.biases[0], K, N, bits, group)
    x, wg, sg, bg = dev_tensors(gate)
    _, wu, su, bu = dev_tensors(up)
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype=out_dtype, splits=splits, max_banks=2)
    for M in (1, 7, 16):
        out = torch.empty((M, N), dtype=plan.out_dtype, device="cuda")
        q.forward_swiglu(plan, x[:M], wg, sg, bg, wu, su, bu, out)
        torch.cuda.synchronize()
        check(to_f64(out), y_ref[:M], out_dtype)
    assert plan.error_flags() == 0


def test_swiglu_needs_two_banks(q):
    import torch
    K, N, bits, group = 2048, 64, 4, 64
    inp = datagen.gen_qmm(5, 1, K, N, bits, group)
    x, w, s, b = dev_tensors(inp)
    plan = q.Plan(K, N, bits, group, max_M=1, out_dtype="f32", splits=1, max_banks=1)
    out = torch.empty((1, N), dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as e:
        q.forward_swiglu(plan, x, w, s, b, w, s, b, out)
    assert e.value.status == q.QMM_ERR_INVALID_ARG


def test_swiglu_matches_separate_projections(q):
    """The fused call equals silu(gate) * up computed from two separate calls of
    the same plan to within fp32 rounding of the epilogue."""
    import torch
    K, N, bits, group = 5120, 1536, 4, 32
    gate = datagen.gen_qmm(31, 16, K, N, bits, group)
    up = datagen.gen_qmm(32, 16, K, N, bits, group)
    x, wg, sg, bg = dev_tensors(gate)
    _, wu, su, bu = dev_tensors(up)
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype="f32", splits=1, max_banks=2)
    fused = torch.empty((16, N), dtype=torch.float32, device="cuda")
    g = torch.empty_like(fused)
    u = torch.empty_like(fused)
    q.forward_swiglu(plan, x, wg, sg, bg, wu, su, bu, fused)
    q.forward(plan, x, wg, sg, bg, g)
    q.forward(plan, x, wu, su, bu, u)
    torch.cuda.synchronize()
    ref = (torch.nn.functional.silu(g.double()) * u.double()).cpu().numpy()
    got = fused.double().cpu().numpy()
    assert np.max(np.abs(got - ref)) <= 1e-5 * np.max(np.abs(ref))
