"""Parity at production-sized row counts for every code format and for the
fused gate/up projection.

The small-shape tests give every CTA only a few 16-row slabs and mostly
partial chunks. Here N = 17408 puts 112 or 128 weight rows (7 or 8 whole
slabs) on each of the 152 CTAs of a GB300, so the 8-row kernel takes its wide
consumer layout wherever the format leaves it four weight stages, and K is a
whole number of 8-group chunks: every width and group size runs the kernel's
full-chunk, full-block path that the named workloads use, against the oracle:

* all 12 formats (2/3/4/5/6/8-bit codes, groups of 32 and 64), 1, 9 and 16
  rows, one and two K slices, both output types;
* the fused gate/up projection on the same row counts for five formats, and on
  the 5120 x 17408 MLP up-projection shape on 1024 sampled columns.

Tolerances are the operation's stated bars (see tests/_helpers.py).
"""
from __future__ import annotations

import numpy as np
import pytest

import datagen
from tests._gpu import check, dev_tensors, run_forward, to_f64

pytestmark = pytest.mark.gpu

N_FULL = 17408
FORMATS = [(2, 32), (2, 64), (3, 32), (3, 64), (4, 32), (4, 64), (5, 32), (5, 64), (6, 32), (6, 64), (8, 32),
           (8, 64)]


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


def _k_full_chunks(bits, group, chunks):
    K = chunks * 8 * group
    assert (K * bits) % 128 == 0
    return K


@pytest.mark.parametrize("bits,group", FORMATS)
@pytest.mark.parametrize("splits", [1, 2])
def test_full_blocks_every_format(q, oracle_mod, bits, group, splits):
    K = _k_full_chunks(bits, group, 3)
    N = N_FULL
    inp = datagen.gen_qmm(60000 + 10 * bits + group + splits, 16, K, N, bits, group)
    y_ref = oracle_mod.qmm_f64(inp.x, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    x, w, s, b = dev_tensors(inp)
    for out_dtype in ("bf16", "f32"):
        plan = q.Plan(K, N, bits, group, max_M=16, out_dtype=out_dtype, splits=splits)
        for M in (1, 9, 16):
            check(to_f64(run_forward(plan, x, w, s, b, M)), y_ref[:M], out_dtype)
        assert plan.error_flags() == 0


@pytest.mark.parametrize("bits,group", [(4, 32), (2, 64), (3, 32), (6, 64), (8, 64)])
def test_swiglu_full_blocks(q, oracle_mod, bits, group):
    import torch
    K = _k_full_chunks(bits, group, 2)
    N = N_FULL
    gate = datagen.gen_qmm(61000 + bits + group, 16, K, N, bits, group)
    up = datagen.gen_qmm(62000 + bits + group, 16, K, N, bits, group)
    y_ref = oracle_mod.qmm_swiglu_f64(gate.x, gate.words[0], gate.scales[0], gate.biases[0],
                                      up.words[0], up.scales[0], up.biases[0], K, N, bits, group)
    x, wg, sg, bg = dev_tensors(gate)
    _, wu, su, bu = dev_tensors(up)
    for out_dtype in ("bf16", "f32"):
        plan = q.Plan(K, N, bits, group, max_M=16, out_dtype=out_dtype, splits=1, max_banks=2)
        for M in (1, 9, 16):
            out = torch.empty((M, N), dtype=plan.out_dtype, device="cuda")
            q.forward_swiglu(plan, x[:M], wg, sg, bg, wu, su, bu, out)
            torch.cuda.synchronize()
            check(to_f64(out), y_ref[:M], out_dtype)
        assert plan.error_flags() == 0


def test_swiglu_mlp_up_shape_sampled_columns(q, oracle_mod):
    """5120 x 17408, 4-bit codes in groups of 32 (the MLP up-projection shape),
    automatic slices, bf16 out: 1024 columns (first and last 128, 768 spread at
    random) against the oracle, every output finite."""
    import torch
    wl = datagen.WORKLOADS["mlp_up"]
    K, N, group, bits = wl["K"], wl["N"], wl["group"], 4
    gate = datagen.gen_qmm(datagen.workload_seed("mlp_up"), 16, K, N, bits, group)
    up = datagen.gen_qmm(datagen.workload_seed("mlp_up") + 100, 16, K, N, bits, group)
    rng = np.random.default_rng(17)
    cols = np.unique(np.concatenate([np.arange(128), np.arange(N - 128, N),
                                     rng.choice(N, 768, replace=False)])).astype(np.int64)
    y_ref = oracle_mod.qmm_swiglu_f64_cols(gate.x, gate.words[0], gate.scales[0], gate.biases[0],
                                           up.words[0], up.scales[0], up.biases[0], K, N, bits, group, cols)
    x, wg, sg, bg = dev_tensors(gate)
    _, wu, su, bu = dev_tensors(up)
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype="bf16", splits=0, max_banks=2)
    for M in (1, 8, 16):
        out = torch.empty((M, N), dtype=plan.out_dtype, device="cuda")
        q.forward_swiglu(plan, x[:M], wg, sg, bg, wu, su, bu, out)
        torch.cuda.synchronize()
        y = to_f64(out)
        assert np.all(np.isfinite(y))
        check(y[:, cols], y_ref[:M], "bf16")
    assert plan.error_flags() == 0
