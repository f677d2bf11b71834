"""Calls whose input is the previous call's output, back to back on one stream
with nothing in between: the staging of call i + 1 must see every element call
i wrote (it reads x only after the work before it on the stream has finished,
while the call's weight loads may already run). Each step is checked against
the oracle on the bf16 input that step actually read, read back after the whole
chain; a captured chain replays to the same values."""
from __future__ import annotations

import numpy as np
import pytest

import datagen
from tests._gpu import check, dev_tensors, to_f64

pytestmark = pytest.mark.gpu

# projection A: 2048 -> 1536 (4-bit, group 64); projection B: 1536 -> 2048 (6-bit, group 32)
KA, NA, BITS_A, GROUP_A = 2048, 1536, 4, 64
KB, NB, BITS_B, GROUP_B = 1536, 2048, 6, 32
STEPS = 3


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


def _weights(seed, M, K, N, bits, group):
    inp = datagen.gen_qmm(seed, M, K, N, bits, group)
    return inp, dev_tensors(inp)


def _chain(q, plans, wa, wb, bufs, M, stream):
    """x0 -> A -> y0 -> B -> x1 -> A -> y1 -> ... on `stream`, every step into its own buffer."""
    pa, pb = plans
    for i in range(STEPS):
        q.forward(pa, bufs[2 * i][:M], *wa, bufs[2 * i + 1][:M], stream=stream)
        q.forward(pb, bufs[2 * i + 1][:M], *wb, bufs[2 * i + 2][:M], stream=stream)


def _verify(oracle_mod, ia, ib, bufs, M):
    import torch
    for i in range(2 * STEPS):
        inp, K, N, bits, group = (ia, KA, NA, BITS_A, GROUP_A) if i % 2 == 0 else (ib, KB, NB, BITS_B, GROUP_B)
        xb = bufs[i][:M].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
        y_ref = oracle_mod.qmm_f64(xb, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
        check(to_f64(bufs[i + 1][:M]), y_ref, "bf16")


@pytest.mark.parametrize("M", [3, 8, 16])
def test_chained_calls(q, oracle_mod, M):
    import torch
    ia, (x0, *wa) = _weights(901, 16, KA, NA, BITS_A, GROUP_A)
    ib, (_, *wb) = _weights(902, 16, KB, NB, BITS_B, GROUP_B)
    pa = q.Plan(KA, NA, BITS_A, GROUP_A, max_M=16, out_dtype="bf16")
    pb = q.Plan(KB, NB, BITS_B, GROUP_B, max_M=16, out_dtype="bf16")
    widths = [KA if i % 2 == 0 else KB for i in range(2 * STEPS + 1)]
    bufs = [torch.empty((16, w), dtype=torch.bfloat16, device="cuda") for w in widths]
    bufs[0].copy_(x0)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    _chain(q, (pa, pb), wa, wb, bufs, M, stream)
    stream.synchronize()
    _verify(oracle_mod, ia, ib, bufs, M)
    assert pa.error_flags() == 0 and pb.error_flags() == 0


def test_chained_calls_captured(q):
    """The chain captured in a CUDA graph replays to the eager values."""
    import torch
    M = 8
    ia, (x0, *wa) = _weights(903, 16, KA, NA, BITS_A, GROUP_A)
    ib, (_, *wb) = _weights(904, 16, KB, NB, BITS_B, GROUP_B)
    pa = q.Plan(KA, NA, BITS_A, GROUP_A, max_M=16, out_dtype="bf16")
    pb = q.Plan(KB, NB, BITS_B, GROUP_B, max_M=16, out_dtype="bf16")
    widths = [KA if i % 2 == 0 else KB for i in range(2 * STEPS + 1)]
    bufs = [torch.empty((16, w), dtype=torch.bfloat16, device="cuda") for w in widths]
    bufs[0].copy_(x0)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    _chain(q, (pa, pb), wa, wb, bufs, M, stream)
    stream.synchronize()
    eager = [b[:M].clone() for b in bufs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        _chain(q, (pa, pb), wa, wb, bufs, M, stream)
    for _ in range(2):
        for b in bufs[1:]:
            b.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for i, b in enumerate(bufs):
            assert torch.equal(b[:M], eager[i]), i
    assert pa.error_flags() == 0 and pb.error_flags() == 0
