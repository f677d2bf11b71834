"""Test-side helpers: an independent code packer, fixture reader, tolerances.

The packer here is written independently of the oracle's decoders (it builds
each row as one Python integer) so that pack -> decode round trips pin the
oracle's reading of the LSB-first stream.
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pack_rows(codes: np.ndarray, bits: int) -> np.ndarray:
    """codes [N, K] -> uint32 words [N, K*bits/32]; code k in stream bits k*bits.. (LSB first)."""
    codes = np.asarray(codes)
    N, K = codes.shape
    assert (K * bits) % 32 == 0
    nw = K * bits // 32
    out = np.zeros((N, nw), dtype=np.uint32)
    for n in range(N):
        stream = 0
        for k in range(K):
            c = int(codes[n, k])
            assert 0 <= c < (1 << bits)
            stream |= c << (k * bits)
        for i in range(nw):
            out[n, i] = (stream >> (32 * i)) & 0xFFFFFFFF
    return out


def read_fixture(name: str) -> dict:
    """Parse a tests/golden/*.txt fixture."""
    d = {"words": [], "scales": [], "biases": [], "x": [], "y": []}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key in ("M", "K", "N", "bits", "group"):
                d[key] = int(vals[0])
            elif key in ("words", "scales", "biases"):
                d[key].append([int(v, 16) for v in vals])
            elif key == "x":
                d["x"].append(vals)
            elif key == "y":
                d["y"].append([float(v) for v in vals])
    K = d["K"]
    x = np.zeros((len(d["x"]), K), dtype=np.uint16)
    for m, spec in enumerate(d["x"]):
        if spec[0] == "ones":
            x[m, :] = 0x3F80                 # bfloat16 1.0
        elif spec[0] == "onehot":
            x[m, int(spec[1])] = 0x3F80
        else:
            raise ValueError(spec)
    d["x"] = x
    d["words"] = np.array(d["words"], dtype=np.uint32)
    d["scales"] = np.array(d["scales"], dtype=np.uint16)
    d["biases"] = np.array(d["biases"], dtype=np.uint16)
    d["y"] = np.array(d["y"], dtype=np.float64)
    return d


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bfloat16 numbers at |v| (normal range): 2**(floor(log2|v|) - 7)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    a = np.maximum(a, np.float64(2.0 ** -126))
    e = np.floor(np.log2(a))
    return np.exp2(e - 7)


def bf16_bits_to_f64(u: np.ndarray) -> np.ndarray:
    """Test-side view of bfloat16 bits as float64 (via the binary32 upper half)."""
    u = np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# Worst error of every check, as a fraction of its tolerance, keyed by the
# running test; tests/conftest.py prints the largest fractions at the end of the
# session so the headroom of the GPU arithmetic is on record in the test log.
HEADROOM: dict[str, float] = {}


def _record_headroom(frac: float) -> None:
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    HEADROOM[test] = max(HEADROOM.get(test, 0.0), float(frac))


def check_f32(y: np.ndarray, y_ref: np.ndarray, rel: float = 2e-3):
    """fp32 output: max|y - y_ref| <= rel * max|y_ref| over the whole call."""
    y = np.asarray(y, dtype=np.float64)
    scale = float(np.max(np.abs(y_ref))) if y_ref.size else 0.0
    err = float(np.max(np.abs(y - y_ref))) if y_ref.size else 0.0
    assert np.all(np.isfinite(y)), "non-finite output"
    if scale > 0.0:
        _record_headroom(err / (rel * scale))
    assert err <= rel * scale, f"fp32 max err {err:.3e} > {rel} * {scale:.3e}"
    return err, scale


def check_bf16(y: np.ndarray, y_ref: np.ndarray, rel: float = 1e-3):
    """bf16 output: |y - y_ref| <= ulp_bf16(|y_ref|) + rel * max|y_ref|, elementwise."""
    y = np.asarray(y, dtype=np.float64)
    scale = float(np.max(np.abs(y_ref))) if y_ref.size else 0.0
    bound = bf16_ulp(y_ref) + rel * scale
    diff = np.abs(y - y_ref)
    assert np.all(np.isfinite(y)), "non-finite output"
    if diff.size:
        _record_headroom(float(np.max(diff / bound)))
    bad = diff > bound
    assert not np.any(bad), (
        f"{int(bad.sum())} bf16 outputs out of tolerance; worst excess "
        f"{float(np.max(diff - bound)):.3e}")
    return float(np.max(diff)) if diff.size else 0.0, scale
