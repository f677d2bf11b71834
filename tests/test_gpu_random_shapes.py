"""Seeded random shapes against the oracle: every width and group size,
K/group from 2 to 40 (even), ragged N from 1 to 700, any M, automatic and
explicit K slices, fp32 and bf16 output. Shapes are drawn under the
validity rules of qmm_validate_desc (K*bits % 128 == 0, K/group even,
slices no more than chunks)."""
from __future__ import annotations

import numpy as np
import pytest

import datagen
from tests._gpu import check, dev_tensors, run_forward, to_f64

pytestmark = pytest.mark.gpu


def _cases(n=24, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        bits = int(rng.choice([2, 3, 4, 5, 6, 8]))
        group = int(rng.choice([32, 64]))
        G = 2 * int(rng.integers(1, 21))
        K = G * group
        if (K * bits) % 128:
            continue
        chunks = (G + 7) // 8
        splits = int(rng.choice([0, 1, 2, 3]))
        if splits > chunks:
            continue
        N = int(rng.integers(1, 701))
        M = int(rng.integers(1, 17))
        out_dtype = str(rng.choice(["f32", "bf16"]))
        out.append((bits, group, K, N, M, splits, out_dtype))
    return out


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


@pytest.mark.parametrize("bits,group,K,N,M,splits,out_dtype", _cases())
def test_random_shape(q, oracle_mod, bits, group, K, N, M, splits, out_dtype):
    inp = datagen.gen_qmm(K * 131 + N * 7 + M, M, K, N, bits, group)
    y_ref = oracle_mod.qmm_f64(inp.x, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    plan = q.Plan(K, N, bits, group, max_M=M, out_dtype=out_dtype, splits=splits)
    x, w, s, b = dev_tensors(inp)
    check(to_f64(run_forward(plan, x, w, s, b, M)), y_ref, out_dtype)
    assert plan.error_flags() == 0
