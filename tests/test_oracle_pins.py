"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test is chosen so that a plausible mistake in the oracle (a dropped term,
a wrong sign, a transposed operand, MSB-first decoding, an off-by-one group
index, a wrong binary16 exponent bias) fails at least one of them:

* conversions: every binary16 / bfloat16 bit pattern against numpy's own casts;
* decoders: exhaustive over every code value at every bit offset, against codes
  packed by an independently written packer, and against each other;
* dequant layout: one-hot x rows give y = s*q + b exactly, for every k;
* exact special case: integer x, power-of-two scales, dyadic biases -> y exact,
  compared with exact rational arithmetic;
* brute force: tiny shapes against exact rational arithmetic (fractions);
* library routine: bits=8, s=1, b=0 is an integer-weight GEMM -> torch.matmul;
* identity: the pages' s*P + b*XS form equals dequantize-then-multiply;
* row independence and linearity in x.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest

from tests._helpers import pack_rows, read_fixture

pytestmark = pytest.mark.usefixtures("oracle_lib")

ALL_BITS = [2, 3, 4, 5, 6, 8]


def _oracle():
    import oracle
    return oracle


# ---------------------------------------------------------------------------
# Conversions
# ---------------------------------------------------------------------------
def test_f16_conversion_all_patterns():
    o = _oracle()
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = o.f16_to_f64(h)
    ref = h.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # spot values: smallest subnormal, largest finite, -2
    assert got[0x0001] == 2.0 ** -24 and got[0x7BFF] == 65504.0 and got[0xC000] == -2.0


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
def test_bf16_conversion_all_patterns():
    o = _oracle()
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = o.bf16_to_f64(h)
    ref = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x3F80] == 1.0 and got[0x0001] == 2.0 ** -133


# ---------------------------------------------------------------------------
# Decoders
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("bits", ALL_BITS)
def test_decoders_exhaustive_values_and_offsets(bits):
    """Row v holds code (v + 7k) mod 2^bits at position k: across rows, every
    position (hence every start offset k*bits mod 32) takes every value."""
    o = _oracle()
    V = 1 << bits
    K = 64
    codes = np.array([[(v + 7 * k) % V for k in range(K)] for v in range(V)], dtype=np.uint8)
    offsets = {(k * bits) % 32 for k in range(K)}
    assert offsets == set(range(0, 32, np.gcd(bits, 32)))
    words = pack_rows(codes, bits)
    assert np.array_equal(o.decode_bitwise(words, V, K, bits), codes)
    assert np.array_equal(o.decode_wordwise(words, V, K, bits), codes)


@pytest.mark.parametrize("bits", ALL_BITS)
def test_decoders_agree_on_random_streams(bits):
    o = _oracle()
    rng = np.random.default_rng(100 + bits)
    N, K = 37, 256
    words = rng.integers(0, 1 << 32, size=(N, K * bits // 32), dtype=np.uint64).astype(np.uint32)
    a = o.decode_bitwise(words, N, K, bits)
    b = o.decode_wordwise(words, N, K, bits)
    assert np.array_equal(a, b)
    # round trip through the independent packer
    assert np.array_equal(pack_rows(a, bits), words)


def test_decoder_is_lsb_first():
    """The first code occupies the lowest bits of the first word."""
    o = _oracle()
    w = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    assert list(o.decode_bitwise(w, 1, 16, 4)[0]) == list(range(16))
    w5 = np.zeros((1, 5), dtype=np.uint32)
    w5[0, 0] = 0b11 << 30          # code 6 spans bits 30..34: its low two bits here
    w5[0, 1] = 0b101               # ... and three bits in word 1
    c = o.decode_wordwise(w5, 1, 32, 5)[0]
    assert c[6] == (0b11 | (0b101 << 2)) and c[7] == 0 and c[5] == 0


# ---------------------------------------------------------------------------
# Golden hand-worked fixtures
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["handworked_4bit_g32.txt", "handworked_6bit_g32.txt"])
def test_golden_handworked(name):
    o = _oracle()
    d = read_fixture(name)
    K, N, bits, group = d["K"], d["N"], d["bits"], d["group"]
    y = o.qmm_f64(d["x"], d["words"], d["scales"], d["biases"], K, N, bits, group)
    assert np.array_equal(y, d["y"]), (y, d["y"])
    y2 = o.qmm_spbxs_f64(d["x"], d["words"], d["scales"], d["biases"], K, N, bits, group)
    assert np.array_equal(y2, d["y"])


def test_golden_words_match_independent_packer():
    d = read_fixture("handworked_6bit_g32.txt")
    codes = np.array([[k + 32 * (k % 2) for k in range(32)]])
    assert np.array_equal(pack_rows(codes, 6), d["words"])
    d4 = read_fixture("handworked_4bit_g32.txt")
    c4 = np.array([[k % 16 for k in range(64)], [15 - k % 16 for k in range(64)]])
    assert np.array_equal(pack_rows(c4, 4), d4["words"])


# ---------------------------------------------------------------------------
# Dequant layout: one-hot activations
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("bits,group", [(4, 32), (4, 64), (5, 32), (6, 32), (8, 32), (8, 64), (2, 64), (3, 32)])
def test_one_hot_gives_dequantized_weight(bits, group):
    o = _oracle()
    rng = np.random.default_rng(7 * bits + group)
    K, N = 2 * group + (group if bits % 2 else 0), 5
    while (K * bits) % 32:
        K += group
    G = K // group
    codes = rng.integers(0, 1 << bits, size=(N, K)).astype(np.uint8)
    words = pack_rows(codes, bits)
    s = rng.uniform(0.002, 0.5, size=(N, G)).astype(np.float16)
    b = rng.uniform(-3, 3, size=(N, G)).astype(np.float16)
    x = np.zeros((K, K), dtype=np.uint16)
    x[np.arange(K), np.arange(K)] = 0x3F80          # row k = one-hot at k
    y = o.qmm_f64(x, words, s.view(np.uint16), b.view(np.uint16), K, N, bits, group)
    gi = np.arange(K) // group
    for n in range(N):
        expect = s[n, gi].astype(np.float64) * codes[n].astype(np.float64) + b[n, gi].astype(np.float64)
        assert np.array_equal(y[:, n], expect)       # s*q needs <= 19 bits: exact in float64


@pytest.mark.parametrize("bits,group", [(2, 32), (3, 64), (4, 32), (4, 64), (5, 32), (6, 64), (8, 32), (8, 64)])
def test_dequant_matches_definition_row_by_row(bits, group):
    """dequant_f64 against W[n,k] = s[n, k//group] * q[n,k] + b[n, k//group]
    written here with numpy's binary16 and codes packed by the test's own
    packer; then against the columns of qmm_f64 on identity activations (the
    one-hot row k of x picks column k of W). Rows have distinct scales, so a
    wrong row offset into the scales or biases fails."""
    o = _oracle()
    rng = np.random.default_rng(41 * bits + group)
    N = 7
    K = 4 * group
    while (K * bits) % 32:
        K += group
    G = K // group
    codes = rng.integers(0, 1 << bits, size=(N, K)).astype(np.uint8)
    words = pack_rows(codes, bits)
    s = (rng.uniform(0.002, 0.5, size=(N, G)) * (1 + np.arange(N))[:, None]).astype(np.float16)
    b = rng.uniform(-3, 3, size=(N, G)).astype(np.float16)
    W = o.dequant_f64(words, s.view(np.uint16), b.view(np.uint16), K, N, bits, group)
    assert W.shape == (N, K)
    gi = np.arange(K) // group
    for n in range(N):
        expect = s[n, gi].astype(np.float64) * codes[n].astype(np.float64) + b[n, gi].astype(np.float64)
        assert np.array_equal(W[n], expect), n      # s*q needs <= 19 bits: exact in float64
    x = np.zeros((K, K), dtype=np.uint16)
    x[np.arange(K), np.arange(K)] = 0x3F80           # bfloat16 1.0 on the diagonal
    y = o.qmm_f64(x, words, s.view(np.uint16), b.view(np.uint16), K, N, bits, group)
    assert np.array_equal(y, W.T)


# ---------------------------------------------------------------------------
# Exact special case and brute force with rational arithmetic
# ---------------------------------------------------------------------------
def _exact_qmm(x_bits, codes, s_bits, b_bits, group):
    """Exact rational y from the definition, via numpy's binary16 and the
    binary32 view of bfloat16 (independent of the oracle's own conversions)."""
    xv = (x_bits.astype(np.uint32) << 16).view(np.float32)
    sv = s_bits.view(np.float16)
    bv = b_bits.view(np.float16)
    M, K = x_bits.shape
    N = codes.shape[0]
    y = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                g = k // group
                w = Fraction(float(sv[n, g])) * int(codes[n, k]) + Fraction(float(bv[n, g]))
                acc += Fraction(float(xv[m, k])) * w
            y[m][n] = acc
    return y


@pytest.mark.parametrize("bits,group", [(4, 32), (5, 32), (6, 64), (8, 32)])
def test_exact_dyadic_case(bits, group):
    """Small-integer x, power-of-two scales, dyadic biases: every partial sum is
    an exactly representable double, so the oracle must be exact."""
    o = _oracle()
    rng = np.random.default_rng(3 * bits + group)
    M, N, K = 2, 3, 2 * group
    while (K * bits) % 32:
        K += group
    G = K // group
    codes = rng.integers(0, 1 << bits, size=(N, K)).astype(np.uint8)
    x = rng.integers(-8, 9, size=(M, K)).astype(np.float32)
    x_bits = (x.view(np.uint32) >> 16).astype(np.uint16)   # small ints are exact in bf16
    s = np.exp2(rng.integers(-6, 2, size=(N, G))).astype(np.float16)
    b = (rng.integers(-256, 257, size=(N, G)) / 64.0).astype(np.float16)
    y = o.qmm_f64(x_bits, pack_rows(codes, bits), s.view(np.uint16), b.view(np.uint16), K, N, bits, group)
    ex = _exact_qmm(x_bits, codes, s.view(np.uint16), b.view(np.uint16), group)
    for m in range(M):
        for n in range(N):
            assert Fraction(float(y[m, n])) == ex[m][n]


@pytest.mark.parametrize("bits,group,K,N,M", [(4, 32, 32, 3, 2), (4, 64, 128, 2, 2), (5, 32, 64, 3, 1),
                                              (6, 32, 32, 2, 2), (8, 64, 64, 3, 2), (3, 32, 64, 2, 2)])
def test_brute_force_tiny(bits, group, K, N, M):
    """Random bf16 x and binary16 s, b: compare with the exact rational value.
    The oracle rounds each product and sum once in float64, so its error is at
    most ~2K ulps of the largest partial magnitude."""
    import datagen
    o = _oracle()
    inp = datagen.gen_qmm(1000 + K + bits, M, K, N, bits, group)
    words, s, b = inp.words[0], inp.scales[0], inp.biases[0]
    y = o.qmm_f64(inp.x, words, s, b, K, N, bits, group)
    codes = o.decode_bitwise(words, N, K, bits)
    assert np.array_equal(pack_rows(codes, bits), words)
    ex = _exact_qmm(inp.x, codes, s, b, group)
    xv = np.abs((inp.x.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    for m in range(M):
        for n in range(N):
            gi = np.arange(K) // group
            wabs = np.abs(s.view(np.float16)[n, gi].astype(np.float64) * codes[n] +
                          b.view(np.float16)[n, gi].astype(np.float64))
            bound = 4 * K * 2.0 ** -52 * float(np.sum(xv[m] * wabs))
            assert abs(Fraction(float(y[m, n])) - ex[m][n]) <= Fraction(bound)


# ---------------------------------------------------------------------------
# Library routine: integer-weight GEMM
# ---------------------------------------------------------------------------
def test_int8_identity_weights_match_torch_matmul():
    import torch
    o = _oracle()
    rng = np.random.default_rng(11)
    M, N, K, bits, group = 5, 33, 256, 8, 32
    codes = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    words = pack_rows(codes, bits)
    G = K // group
    s = np.full((N, G), 0x3C00, dtype=np.uint16)    # 1.0
    b = np.zeros((N, G), dtype=np.uint16)           # 0.0
    import datagen
    x = datagen.gen_x(12, M, K)
    y = o.qmm_f64(x, words, s, b, K, N, bits, group)
    xt = torch.from_numpy((x.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    qt = torch.from_numpy(codes.astype(np.float64))
    ref = torch.matmul(xt, qt.T).numpy()
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))


# ---------------------------------------------------------------------------
# The pages' form, row independence, linearity
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("bits,group", [(4, 32), (4, 64), (5, 32), (6, 32), (8, 32)])
def test_spbxs_identity(bits, group):
    """sum_g (s*P + b*XS) == dequantize-then-multiply, within float64 rounding."""
    import datagen
    o = _oracle()
    M, K, N = 4, 512, 40
    inp = datagen.gen_qmm(77 + bits + group, M, K, N, bits, group)
    a = o.qmm_f64(inp.x, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    c = o.qmm_spbxs_f64(inp.x, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    W = o.dequant_f64(inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    xv = np.abs(o.bf16_to_f64(inp.x))
    terms = xv @ np.abs(W).T
    assert np.all(np.abs(a - c) <= 1e-12 * terms)
    # and both differ from a sign-flipped bias (the check has teeth)
    flipped = (inp.biases[0] ^ 0x8000).astype(np.uint16)
    d = o.qmm_f64(inp.x, inp.words[0], inp.scales[0], flipped, K, N, bits, group)
    assert np.max(np.abs(d - a)) > 1e-3 * np.max(np.abs(a))


def test_row_independence_bitwise():
    import datagen
    o = _oracle()
    M, K, N, bits, group = 16, 1024, 24, 4, 64
    inp = datagen.gen_qmm(5, M, K, N, bits, group)
    y = o.qmm_f64(inp.x, inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    for m in range(M):
        y1 = o.qmm_f64(inp.x[m:m + 1], inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
        assert np.array_equal(y[m], y1[0])


def test_linearity_in_x():
    """x1, x2 small integers (so x1 + x2 is exact in bf16): y(x1+x2) = y(x1)+y(x2)."""
    import datagen
    o = _oracle()
    K, N, bits, group = 256, 16, 5, 32
    inp = datagen.gen_qmm(9, 1, K, N, bits, group)
    rng = np.random.default_rng(9)
    x1 = rng.integers(-20, 21, size=(1, K)).astype(np.float32)
    x2 = rng.integers(-20, 21, size=(1, K)).astype(np.float32)
    to_bits = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)
    args = (inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    y1 = o.qmm_f64(to_bits(x1), *args)
    y2 = o.qmm_f64(to_bits(x2), *args)
    y12 = o.qmm_f64(to_bits(x1 + x2), *args)
    assert np.max(np.abs(y12 - (y1 + y2))) <= 1e-12 * (np.max(np.abs(y1)) + np.max(np.abs(y2)))


def test_column_subset_matches_full():
    import datagen
    o = _oracle()
    M, K, N, bits, group = 3, 256, 50, 6, 32
    inp = datagen.gen_qmm(21, M, K, N, bits, group)
    args = (inp.words[0], inp.scales[0], inp.biases[0], K, N, bits, group)
    y = o.qmm_f64(inp.x, *args)
    cols = np.array([0, 7, 49, 7, 31])
    assert np.array_equal(o.qmm_f64_cols(inp.x, *args, cols), y[:, cols])


def test_oracle_rejects_bad_shapes():
    o = _oracle()
    with pytest.raises(ValueError):
        o.decode_bitwise(np.zeros((1, 1), np.uint32), 1, 3, 5)       # 15 bits: not word aligned
    with pytest.raises(ValueError):
        o.qmm_f64(np.zeros((1, 48), np.uint16), np.zeros((1, 6), np.uint32),
                  np.zeros((1, 1), np.uint16), np.zeros((1, 1), np.uint16), 48, 1, 4, 32)


# ---------------------------------------------------------------------------
# Fused gate/up projection with the SwiGLU epilogue
# ---------------------------------------------------------------------------
def _silu_tanh(v: float) -> float:
    """silu through a different closed form: v * sigmoid(v) = v * (1 + tanh(v/2)) / 2."""
    import math
    return v * (1.0 + math.tanh(v / 2.0)) / 2.0


def test_swiglu_one_hot_matches_closed_form():
    """One-hot x rows pick single dequantized weights, so g and u are exact
    dyadic numbers; y must equal silu(g) * u evaluated through tanh."""
    import math
    o = _oracle()
    bits, group, K, N = 4, 32, 64, 3
    rng = np.random.default_rng(3)
    cg = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    cu = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    G = K // group
    sg = np.full((N, G), 0.5, np.float16).view(np.uint16)
    bg = np.full((N, G), -4.0, np.float16).view(np.uint16)
    su = np.full((N, G), 0.25, np.float16).view(np.uint16)
    bu = np.full((N, G), 1.0, np.float16).view(np.uint16)
    ks = [0, 5, 33, 63]
    x = np.zeros((len(ks), K), np.uint16)
    for i, k in enumerate(ks):
        x[i, k] = 0x3F80            # bfloat16 1.0
    y = o.qmm_swiglu_f64(x, pack_rows(cg, bits), sg, bg, pack_rows(cu, bits), su, bu, K, N, bits, group)
    for i, k in enumerate(ks):
        for n in range(N):
            g = 0.5 * float(cg[n, k]) - 4.0
            u = 0.25 * float(cu[n, k]) + 1.0
            want = _silu_tanh(g) * u
            assert math.isclose(y[i, n], want, rel_tol=1e-14, abs_tol=1e-15), (i, n, y[i, n], want)
            if g == 0.0:
                assert y[i, n] == 0.0


def test_swiglu_saturation():
    """Large positive gates pass through (silu(g) = g in float64 for g >= 40);
    large negative gates vanish."""
    o = _oracle()
    bits, group, K, N = 8, 32, 32, 2
    codes = np.full((N, K), 0, np.uint8)
    G = 1
    sg = np.full((N, G), 1.0, np.float16).view(np.uint16)
    bg = np.array([[40.0], [-40.0]], np.float16).view(np.uint16)
    su = np.full((N, G), 1.0, np.float16).view(np.uint16)
    bu = np.full((N, G), 3.0, np.float16).view(np.uint16)
    x = np.zeros((1, K), np.uint16)
    x[0, 7] = 0x3F80
    y = o.qmm_swiglu_f64(x, pack_rows(codes, bits), sg, bg, pack_rows(codes, bits), su, bu, K, N, bits, group)
    assert y[0, 0] == 120.0
    assert 0.0 > y[0, 1] > -1e-14


def test_swiglu_brute_force_tiny():
    """Random tiny case against a triple loop written here (dequantize, dot,
    silu through exp)."""
    import math
    import datagen
    o = _oracle()
    bits, group, K, N, M = 5, 32, 64, 3, 2
    a = datagen.gen_qmm(41, M, K, N, bits, group)
    c = datagen.gen_qmm(42, M, K, N, bits, group)
    y = o.qmm_swiglu_f64(a.x, a.words[0], a.scales[0], a.biases[0], c.words[0], c.scales[0], c.biases[0],
                         K, N, bits, group)
    xs = (a.x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    def proj(inp):
        codes = o.decode_bitwise(inp.words[0], N, K, bits).astype(np.float64)
        s = inp.scales[0].view(np.float16).astype(np.float64)
        b = inp.biases[0].view(np.float16).astype(np.float64)
        out = np.zeros((M, N))
        for m in range(M):
            for n in range(N):
                out[m, n] = sum(xs[m, k] * (s[n, k // group] * codes[n, k] + b[n, k // group]) for k in range(K))
        return out
    g, u = proj(a), proj(c)
    for m in range(M):
        for n in range(N):
            want = g[m, n] / (1.0 + math.exp(-g[m, n])) * u[m, n]
            assert math.isclose(y[m, n], want, rel_tol=1e-11, abs_tol=1e-12)


def test_swiglu_column_subset():
    """The column-subset form on a tiny case, columns out of order and repeated,
    against a triple loop written here (dequantize, dot, silu through tanh),
    and bitwise equal to the full form's columns on a larger case."""
    import datagen
    o = _oracle()
    bits, group, K, N, M = 3, 64, 128, 4, 3
    a = datagen.gen_qmm(51, M, K, N, bits, group)
    c = datagen.gen_qmm(52, M, K, N, bits, group)
    cols = np.array([3, 0, 3, 1], dtype=np.int64)
    y = o.qmm_swiglu_f64_cols(a.x, a.words[0], a.scales[0], a.biases[0], c.words[0], c.scales[0], c.biases[0],
                              K, N, bits, group, cols)
    assert y.shape == (M, cols.size)
    xs = (a.x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    gi = np.arange(K) // group

    def proj(inp, n):
        codes = inp.words[0][n]
        q = np.array([(int(sum(int(w) << (32 * i) for i, w in enumerate(codes))) >> (k * bits)) & ((1 << bits) - 1)
                      for k in range(K)], dtype=np.float64)
        s = inp.scales[0].view(np.float16)[n, gi].astype(np.float64)
        b = inp.biases[0].view(np.float16)[n, gi].astype(np.float64)
        return xs @ (s * q + b)

    for j, n in enumerate(cols):
        g, u = proj(a, n), proj(c, n)
        want = np.array([_silu_tanh(v) for v in g]) * u
        assert np.allclose(y[:, j], want, rtol=1e-12, atol=1e-14 * np.max(np.abs(want)))
    K2, N2 = 512, 40
    a2 = datagen.gen_qmm(53, 2, K2, N2, 4, 32)
    c2 = datagen.gen_qmm(54, 2, K2, N2, 4, 32)
    args = (a2.x, a2.words[0], a2.scales[0], a2.biases[0], c2.words[0], c2.scales[0], c2.biases[0], K2, N2, 4, 32)
    cols2 = np.array([39, 7, 0, 21], dtype=np.int64)
    assert np.array_equal(o.qmm_swiglu_f64_cols(*args, cols2), o.qmm_swiglu_f64(*args)[:, cols2])
