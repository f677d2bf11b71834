"""GPU vs oracle parity on small shapes (several chunks, ragged row tails,
partial last chunks), plus determinism, row independence, banked == single,
guard zones and the in-register unpack (bit-exact).

Tolerances (from the operation's stated bars):
  fp32 out: max|y - y_ref| <= 2e-3 * max|y_ref| over the call;
  bf16 out: |y - y_ref| <= ulp_bf16(|y_ref|) + 1e-3 * max|y_ref| elementwise.
"""
from __future__ import annotations

import numpy as np
import pytest

import datagen
from tests._gpu import check, dev_tensors, run_forward, to_f64

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


def _K_for(bits, group, G):
    K = G * group
    assert (K * bits) % 128 == 0, (bits, group, G)
    return K


# ---------------------------------------------------------------------------
# Unpack: bit-exact against the oracle's bit-at-a-time decoder
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
@pytest.mark.parametrize("K,N", [(256, 37), (2048, 9)])
def test_unpack_bit_exact(q, oracle_mod, bits, K, N):
    import torch
    rng = np.random.default_rng(bits * 1000 + K)
    words = rng.integers(0, 1 << 32, size=(N, K * bits // 32), dtype=np.uint64).astype(np.uint32)
    w = torch.from_numpy(words.view(np.int32)).cuda()
    codes = q.unpack_codes(w, K, N, bits)
    torch.cuda.synchronize()
    ref = oracle_mod.decode_bitwise(words, N, K, bits)
    assert np.array_equal(codes.cpu().numpy(), ref)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_unpack_every_value_every_offset(q, oracle_mod, bits):
    """Rows where position k holds (v + 7k) mod 2^bits: every value at every offset."""
    import torch
    from tests._helpers import pack_rows
    V, K = 1 << bits, 128
    codes = np.array([[(v + 7 * k) % V for k in range(K)] for v in range(V)], dtype=np.uint8)
    words = pack_rows(codes, bits)
    got = q.unpack_codes(torch.from_numpy(words.view(np.int32)).cuda(), K, V, bits)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), codes)


# ---------------------------------------------------------------------------
# Small-shape parity over formats x rows x output x slices
# ---------------------------------------------------------------------------
FORMATS = [(2, 32), (2, 64), (3, 32), (3, 64), (4, 32), (4, 64), (5, 32), (5, 64), (6, 32), (6, 64), (8, 32), (8, 64)]
MS = [1, 2, 3, 5, 8, 9, 12, 16]


@pytest.mark.parametrize("bits,group", FORMATS)
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("splits", [1, 2, 3])
def test_small_parity(q, oracle_mod, bits, group, out_dtype, splits):
    # G = 20 groups -> chunks of 8, 8, 4 (a partial last chunk); N ragged vs 16-row slabs
    G = 20
    K = _K_for(bits, group, G)
    N = 300
    inp = datagen.gen_qmm(hash((bits, group, splits)) % 100000, 16, K, N, bits, group)
    y_ref = oracle_mod.qmm_f64(inp.x, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype=out_dtype, splits=splits)
    assert plan.info()["splits"] == splits
    x, w, s, b = dev_tensors(inp)
    for M in MS:
        y = to_f64(run_forward(plan, x, w, s, b, M))
        check(y, y_ref[:M], out_dtype)
    assert plan.error_flags() == 0


@pytest.mark.parametrize("bits,group,G", [(4, 32, 10), (4, 64, 6), (6, 32, 14), (8, 64, 2), (5, 32, 12), (2, 64, 6), (3, 32, 12)])
@pytest.mark.parametrize("N", [1, 15, 17, 129, 1000])
def test_ragged_shapes(q, oracle_mod, bits, group, G, N):
    """K/group not a multiple of 8 (4-byte scale rows, partial chunks) and tiny/ragged N."""
    K = _K_for(bits, group, G)
    inp = datagen.gen_qmm(N * 31 + G, 16, K, N, bits, group)
    y_ref = oracle_mod.qmm_f64(inp.x, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype="f32")
    x, w, s, b = dev_tensors(inp)
    for M in (1, 7, 16):
        check(to_f64(run_forward(plan, x, w, s, b, M)), y_ref[:M], "f32")


def test_m_zero_is_noop(q):
    import torch
    inp = datagen.gen_qmm(3, 1, 512, 64, 4, 64)
    plan = q.Plan(512, 64, 4, 64, max_M=4, out_dtype="f32")
    x, w, s, b = dev_tensors(inp)
    out = torch.full((1, 64), 7.0, device="cuda")
    q.forward(plan, x[:0], w, s, b, out)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


def test_m_above_plan_max_rejected(q):
    import torch
    inp = datagen.gen_qmm(3, 5, 512, 64, 4, 64)
    plan = q.Plan(512, 64, 4, 64, max_M=4, out_dtype="f32")
    x, w, s, b = dev_tensors(inp)
    out = torch.empty((5, 64), device="cuda")
    with pytest.raises(q.QmmError) as e:
        q.forward(plan, x, w, s, b, out)
    assert e.value.status == q.QMM_ERR_INVALID_ARG


def test_plan_mismatch_rejected(q):
    import torch
    plan = q.Plan(512, 64, 4, 64, max_M=4, out_dtype="f32")
    inp = datagen.gen_qmm(3, 2, 512, 64, 4, 64)
    x, w, s, b = dev_tensors(inp)
    out = torch.empty((2, 64), device="cuda")
    st = q.lib.qmm_forward(plan.handle, x.data_ptr(), 2, w.data_ptr(), s.data_ptr(), b.data_ptr(), 512, 64, 4, 32,
                           out.data_ptr(), None)
    assert st == q.QMM_ERR_PLAN_MISMATCH


# ---------------------------------------------------------------------------
# Determinism, row independence, banked == single, guard zones
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("splits", [1, 2, 3, 4, 8])
def test_deterministic(q, splits):
    import torch
    K, N, bits, group = 64 * 96, 1000, 4, 64   # 12 chunks: room for 8 slices
    inp = datagen.gen_qmm(99, 16, K, N, bits, group)
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype="bf16", splits=splits)
    x, w, s, b = dev_tensors(inp)
    for M in (1, 16):
        outs = [run_forward(plan, x, w, s, b, M).clone() for _ in range(3)]
        assert all(torch.equal(outs[0], o) for o in outs[1:])


@pytest.mark.parametrize("bits,group,splits", [(4, 32, 1), (6, 64, 2), (8, 32, 3), (5, 32, 1), (2, 32, 2), (3, 64, 1)])
def test_row_independence(q, oracle_mod, bits, group, splits):
    """Row m of an M-row call equals the 1-row call on the same x row bitwise, for
    every m and M in {16, 9, 5} (8- and 16-row tiles): each activation row is an
    independent MMA column whose range factors depend on that row alone, and the
    split count is a property of the plan, not of M."""
    K, N = 2048, 512
    inp = datagen.gen_qmm(5 + bits, 16, K, N, bits, group)
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype="f32", splits=splits)
    x, w, s, b = dev_tensors(inp)
    y_ref = oracle_mod.qmm_f64(inp.x, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    ys = {M: to_f64(run_forward(plan, x, w, s, b, M)) for M in (16, 9, 5)}
    mismatched = []
    for m in range(16):
        y1 = to_f64(run_forward(plan, x[m:m + 1].contiguous(), w, s, b, 1))
        check(y1[0][None], y_ref[m][None], "f32")
        for M, yM in ys.items():
            if m < M and not np.array_equal(y1[0], yM[m]):
                mismatched.append((M, m))
    assert not mismatched, mismatched
    assert plan.error_flags() == 0


@pytest.mark.parametrize("bits", [4, 5, 8])
def test_consumer_layouts_agree(q, oracle_mod, bits):
    """The consumer layouts add the same terms in the same order: every layout
    sums a row block's even- and odd-index items apart and adds the two. A
    projection with 112 rows per CTA takes the wide layout at 1-8 rows, one with
    80 rows per CTA the narrow layout, one with 48 rows per CTA the pair layout
    (two items in flight); at 9-16 rows the first two are narrow and the third
    pair. On the same weights and x their shared rows must agree bitwise (K
    spans an even number of 8-group chunks, so each row block's items split the
    same way), and the smallest result must match the oracle."""
    import torch
    K, group = 5120, 32
    probe = q.Plan(K, 1024, bits, group, max_M=8, out_dtype="f32", splits=1)
    sms = probe.info()["num_sms"]
    probe.close()
    Ns = [sms * 112, sms * 80, sms * 48]
    inp = datagen.gen_qmm(77 + bits, 16, K, Ns[0], bits, group)
    x, w, s, b = dev_tensors(inp)
    row_bytes = K * bits // 8
    G = K // group

    def prefix(n):
        return (w.view(torch.uint8).view(Ns[0], row_bytes)[:n].contiguous().view(torch.int32),
                s.view(Ns[0], G)[:n].contiguous(), b.view(Ns[0], G)[:n].contiguous())
    plans = [q.Plan(K, n, bits, group, max_M=16, out_dtype="f32", splits=1) for n in Ns]
    for M in (1, 8, 16):
        ys = [to_f64(run_forward(pl, x, *prefix(n), M)) for pl, n in zip(plans, Ns)]
        for i in (1, 2):
            n = Ns[i]
            assert np.array_equal(ys[i - 1][:, :n], ys[i]), (M, i, np.abs(ys[i - 1][:, :n] - ys[i]).max())
        cols = np.arange(0, Ns[2], 11, dtype=np.int64)
        y_ref = oracle_mod.qmm_f64_cols(inp.x[:M], inp.words[0], inp.scales[0], inp.biases[0], K, Ns[0], bits,
                                        group, cols)
        check(ys[2][:, cols], y_ref, "f32")
    assert all(pl.error_flags() == 0 for pl in plans)


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_activation_dynamic_range(q, oracle_mod, bits):
    """Rows of x at very different magnitudes (2^-110 .. 2^100), a row whose
    groups alternate between 2^30 and 2^-30, a zero row and a zero chunk. The
    activations enter the tensor cores as binary16 under a power-of-two range
    factor per (row, 8-group chunk); each row must stay within tolerance of its
    own largest output (a row of zeros gives exact zeros)."""
    from tests._helpers import check_f32
    K, N, group = 1024, 200, 32          # 4 chunks
    inp = datagen.gen_qmm(77 + bits, 16, K, N, bits, group)
    xf = (inp.x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for m, e in enumerate([-110, -80, -40, -10, 0, 10, 40, 80, 100]):
        xf[m] *= 2.0 ** e
    xf[9] *= np.where((np.arange(K) // group) % 2 == 0, 2.0 ** 30, 2.0 ** -30)
    xf[10] = 0.0
    xf[11, 256:512] = 0.0
    inp.x = datagen.f64_to_bf16_bits(xf)
    y_ref = oracle_mod.qmm_f64(inp.x, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype="f32", splits=1)
    x, w, s, b = dev_tensors(inp)
    y = to_f64(run_forward(plan, x, w, s, b, 16))
    assert np.all(np.isfinite(y))
    for m in range(16):
        check_f32(y[m:m + 1], y_ref[m:m + 1])
    assert np.all(y[10] == 0.0)
    assert plan.error_flags() == 0


def test_banked_equals_single(q):
    import torch
    K, N, bits, group, B = 1024, 700, 4, 64, 5
    inp = datagen.gen_qmm(17, 9, K, N, bits, group, banks=B)
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype="bf16", max_banks=B)
    devs = [dev_tensors(inp, bank=i) for i in range(B)]
    x = devs[0][0]
    for M in (1, 9):
        outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(B)]
        q.forward_banked(plan, x[:M], [d[1] for d in devs], [d[2] for d in devs], [d[3] for d in devs], outs)
        torch.cuda.synchronize()
        for i in range(B):
            single = run_forward(plan, x, devs[i][1], devs[i][2], devs[i][3], M)
            assert torch.equal(outs[i], single), f"bank {i} M={M}"


@pytest.mark.parametrize("splits", [1, 4])
def test_guard_zones(q, splits):
    """Canary words before and after `out` (and the plan's unused workspace tail) stay untouched."""
    import torch
    K, N, bits, group, M = 4096, 333, 5, 32, 11
    inp = datagen.gen_qmm(23, M, K, N, bits, group)
    plan = q.Plan(K, N, bits, group, max_M=16, out_dtype="f32", splits=splits)
    x, w, s, b = dev_tensors(inp)
    pad = 1024
    buf = torch.full((2 * pad + M * N,), -12345.0, device="cuda")
    out = buf[pad:pad + M * N].view(M, N)
    tail_before = plan.workspace[-64:].clone()
    run_forward(plan, x, w, s, b, M, out=out)
    assert torch.all(buf[:pad] == -12345.0) and torch.all(buf[pad + M * N:] == -12345.0)
    assert torch.all(out != -12345.0)
    assert torch.equal(plan.workspace[-64:], tail_before)


def test_pointers_are_16_byte_aligned_in_tests(q):
    inp = datagen.gen_qmm(1, 2, 512, 64, 4, 64)
    for t in dev_tensors(inp):
        assert t.data_ptr() % 16 == 0
