"""Full-size workloads (the shapes the benchmark times) against the oracle, in
the launch configuration the benchmark uses (same plan settings):

  pr1_ref       M=1,  K=2048,  N=2048,  4-bit g64, fp32 out
  mlp_up        M in {1,2,4,8,16}, K=5120, N=17408, 4-bit g32, bf16 out
  down_longk    M in {1,8,16}, K=17408, N=5120, 4-bit g64, splits {1,2,4,8}, bf16 out
  mixed_widths  M=8, K=5120, N=6144, bits {5,6,8}, g32, bf16 out
  banked        36 banks, M in {1,16}, K=2048, N=8192, 4-bit g64, bf16 out
  lm_head       M in {1,8,16}, K=4096, N=151936, 8-bit g64, bf16 out

Every output column is compared except in the banked workload, where two banks
are compared in full and the others on 64 sampled columns each, and in the
lm_head workload, where 2304 columns (the first and last 128 and 2048 spread
at random) are compared and every output is checked finite.
"""
from __future__ import annotations

import numpy as np
import pytest

import datagen
from tests._gpu import check, dev_tensors, run_forward, to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


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


def _run_workload(q, oracle_mod, name, bits, splits_list):
    wl = datagen.WORKLOADS[name]
    K, N, group = wl["K"], wl["N"], wl["group"]
    Mmax = max(wl["Ms"])
    inp = datagen.gen_qmm(datagen.workload_seed(name) + bits, Mmax, K, N, bits, group)
    y_ref = oracle_mod.qmm_f64(inp.x, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    x, w, s, b = dev_tensors(inp)
    for splits in splits_list:
        plan = q.Plan(K, N, bits, group, max_M=Mmax, out_dtype=wl["out"], splits=splits)
        for M in wl["Ms"]:
            y = to_f64(run_forward(plan, x, w, s, b, M))
            check(y, y_ref[:M], wl["out"])
        assert plan.error_flags() == 0


def test_pr1_ref(q, oracle_mod):
    _run_workload(q, oracle_mod, "pr1_ref", 4, [0])


def test_mlp_up(q, oracle_mod):
    _run_workload(q, oracle_mod, "mlp_up", 4, [0])


def test_down_longk(q, oracle_mod):
    _run_workload(q, oracle_mod, "down_longk", 4, [1, 2, 4, 8, 0])


@pytest.mark.parametrize("bits", [5, 6, 8])
def test_mixed_widths(q, oracle_mod, bits):
    _run_workload(q, oracle_mod, "mixed_widths", bits, [0, 1])


def test_banked(q, oracle_mod):
    import torch
    wl = datagen.WORKLOADS["banked"]
    K, N, group, B, bits = wl["K"], wl["N"], wl["group"], wl["banks"], 4
    inp = datagen.gen_qmm(datagen.workload_seed("banked"), 16, K, N, bits, group, banks=B)
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype="bf16", max_banks=B)
    devs = [dev_tensors(inp, bank=i) for i in range(B)]
    x = devs[0][0]
    rng = np.random.default_rng(4)
    for M in wl["Ms"]:
        outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(B)]
        q.forward_banked(plan, x[:M], [d[1] for d in devs], [d[2] for d in devs], [d[3] for d in devs], outs)
        torch.cuda.synchronize()
        for i in range(B):
            y = to_f64(outs[i])
            args = (inp.words[i], inp.scales[i], inp.biases[i], K, N, bits, group)
            if i in (0, B - 1):
                y_ref = oracle_mod.qmm_f64(inp.x[:M], *args)
                check(y, y_ref, "bf16")
            else:
                cols = np.sort(rng.choice(N, size=64, replace=False))
                y_ref = oracle_mod.qmm_f64_cols(inp.x[:M], *args, cols)
                # the tolerance's relative term uses the full row scale: take it from bank 0's scale
                from tests._helpers import bf16_ulp
                scale = max(float(np.max(np.abs(y_ref))), 1e-30)
                bound = bf16_ulp(y_ref) + 1e-3 * scale
                assert np.all(np.abs(y[:, cols] - y_ref) <= bound), f"bank {i}"
    assert plan.error_flags() == 0


def test_lm_head(q, oracle_mod):
    wl = datagen.WORKLOADS["lm_head"]
    K, N, group, bits = wl["K"], wl["N"], wl["group"], 8
    inp = datagen.gen_qmm(datagen.workload_seed("lm_head"), 16, K, N, bits, group)
    rng = np.random.default_rng(7)
    cols = np.unique(np.concatenate([np.arange(128), np.arange(N - 128, N),
                                     rng.choice(N, 2048, replace=False)])).astype(np.int64)
    y_ref = oracle_mod.qmm_f64_cols(inp.x, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group, cols)
    x, w, s, b = dev_tensors(inp)
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype="bf16", splits=0)
    for M in wl["Ms"]:
        y = to_f64(run_forward(plan, x, w, s, b, M))
        assert np.all(np.isfinite(y))
        check(y[:, cols], y_ref[:M], "bf16")
    assert plan.error_flags() == 0
