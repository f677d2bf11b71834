"""CPU oracle for the group-wise affine-quantized multi-row matmul.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product library
(``bit_affine_quantized_group_gb300``) never does, and shares no code with it.

The arithmetic lives in ``qmm_oracle.cpp`` (plain C++, float64). This module
builds it with g++ on first use and exposes numpy-facing wrappers:

* ``decode_bitwise`` / ``decode_wordwise`` -- two independent readers of the
  LSB-first code stream.
* ``dequant_f64`` -- ``W = s*q + b`` in float64.
* ``qmm_f64`` / ``qmm_f64_cols`` -- the definition ``y = x @ W.T`` in float64,
  k ascending (all columns, or a chosen subset).
* ``qmm_swiglu_f64`` / ``qmm_swiglu_f64_cols`` -- silu(qmm(x, gate)) * qmm(x, up)
  in float64 (all columns, or a chosen subset).
* ``qmm_spbxs_f64`` -- the dequant-after-dot form ``sum_g s*P + b*XS``
  ("C += s*P + b*XS", vmlx-swift PR #565, LaneQMM commit), used only to check
  that it equals the definition.
* ``f16_to_f64`` / ``bf16_to_f64`` -- conversions written from the IEEE-754
  format definitions.

Every pin of these functions is under ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle_qmm.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with g++ (OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["g++", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c++17", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_f16_to_f64_array.argtypes = [vp, i64, vp]
            lib.oracle_bf16_to_f64_array.argtypes = [vp, i64, vp]
            lib.oracle_decode_bitwise.argtypes = [vp, i64, i64, i32, vp]
            lib.oracle_decode_wordwise.argtypes = [vp, i64, i64, i32, vp]
            lib.oracle_dequant_f64.argtypes = [vp, vp, vp, i64, i64, i32, i32, vp]
            lib.oracle_qmm_f64.argtypes = [vp, i64, vp, vp, vp, i64, i64, i32, i32, vp]
            lib.oracle_qmm_f64_cols.argtypes = [vp, i64, vp, vp, vp, i64, i64, i32, i32, vp, i64, vp]
            lib.oracle_qmm_spbxs_f64.argtypes = [vp, i64, vp, vp, vp, i64, i64, i32, i32, vp]
            lib.oracle_qmm_swiglu_f64.argtypes = [vp, i64, vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, vp]
            lib.oracle_qmm_swiglu_f64_cols.argtypes = [vp, i64, vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, vp,
                                                       i64, vp]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            for name in ("oracle_decode_bitwise", "oracle_decode_wordwise", "oracle_dequant_f64",
                         "oracle_qmm_f64", "oracle_qmm_f64_cols", "oracle_qmm_spbxs_f64",
                         "oracle_qmm_swiglu_f64", "oracle_qmm_swiglu_f64_cols"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle: {what} rejected its arguments")


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def f16_to_f64(h) -> np.ndarray:
    h = _c(np.asarray(h), np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    _load().oracle_f16_to_f64_array(_p(h), h.size, _p(out))
    return out


def bf16_to_f64(h) -> np.ndarray:
    h = _c(np.asarray(h), np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    _load().oracle_bf16_to_f64_array(_p(h), h.size, _p(out))
    return out


def decode_bitwise(words: np.ndarray, N: int, K: int, bits: int) -> np.ndarray:
    w = _c(words, np.uint32)
    codes = np.empty((N, K), dtype=np.uint8)
    _check(_load().oracle_decode_bitwise(_p(w), N, K, bits, _p(codes)), "decode_bitwise")
    return codes


def decode_wordwise(words: np.ndarray, N: int, K: int, bits: int) -> np.ndarray:
    w = _c(words, np.uint32)
    codes = np.empty((N, K), dtype=np.uint8)
    _check(_load().oracle_decode_wordwise(_p(w), N, K, bits, _p(codes)), "decode_wordwise")
    return codes


def dequant_f64(words, scales, biases, K: int, N: int, bits: int, group: int) -> np.ndarray:
    w, s, b = _c(words, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    W = np.empty((N, K), dtype=np.float64)
    _check(_load().oracle_dequant_f64(_p(w), _p(s), _p(b), K, N, bits, group, _p(W)), "dequant_f64")
    return W


def qmm_f64(x_bf16, words, scales, biases, K: int, N: int, bits: int, group: int) -> np.ndarray:
    """y[m,n] = sum_k x[m,k] * (s[n,k/group]*q[n,k] + b[n,k/group]) in float64."""
    x = _c(x_bf16, np.uint16).reshape(-1, K)
    w, s, b = _c(words, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    M = x.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    _check(_load().oracle_qmm_f64(_p(x), M, _p(w), _p(s), _p(b), K, N, bits, group, _p(y)), "qmm_f64")
    return y


def qmm_f64_cols(x_bf16, words, scales, biases, K: int, N: int, bits: int, group: int, cols) -> np.ndarray:
    """Same as qmm_f64 for the listed output columns only; returns [M, len(cols)]."""
    x = _c(x_bf16, np.uint16).reshape(-1, K)
    w, s, b = _c(words, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    cols = _c(cols, np.int64).reshape(-1)
    M = x.shape[0]
    y = np.empty((M, cols.size), dtype=np.float64)
    _check(_load().oracle_qmm_f64_cols(_p(x), M, _p(w), _p(s), _p(b), K, N, bits, group,
                                       _p(cols), cols.size, _p(y)), "qmm_f64_cols")
    return y


def qmm_swiglu_f64(x_bf16, words_gate, scales_gate, biases_gate, words_up, scales_up, biases_up,
                   K: int, N: int, bits: int, group: int) -> np.ndarray:
    """y = silu(qmm(x, gate)) * qmm(x, up) in float64; returns [M, N]."""
    x = _c(x_bf16, np.uint16).reshape(-1, K)
    wg, sg, bg = _c(words_gate, np.uint32), _c(scales_gate, np.uint16), _c(biases_gate, np.uint16)
    wu, su, bu = _c(words_up, np.uint32), _c(scales_up, np.uint16), _c(biases_up, np.uint16)
    M = x.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    _check(_load().oracle_qmm_swiglu_f64(_p(x), M, _p(wg), _p(sg), _p(bg), _p(wu), _p(su), _p(bu), K, N, bits,
                                         group, _p(y)), "qmm_swiglu_f64")
    return y


def qmm_swiglu_f64_cols(x_bf16, words_gate, scales_gate, biases_gate, words_up, scales_up, biases_up,
                        K: int, N: int, bits: int, group: int, cols) -> np.ndarray:
    """qmm_swiglu_f64 for the listed output columns only; returns [M, len(cols)]."""
    x = _c(x_bf16, np.uint16).reshape(-1, K)
    wg, sg, bg = _c(words_gate, np.uint32), _c(scales_gate, np.uint16), _c(biases_gate, np.uint16)
    wu, su, bu = _c(words_up, np.uint32), _c(scales_up, np.uint16), _c(biases_up, np.uint16)
    cols = _c(cols, np.int64).reshape(-1)
    M = x.shape[0]
    y = np.empty((M, cols.size), dtype=np.float64)
    _check(_load().oracle_qmm_swiglu_f64_cols(_p(x), M, _p(wg), _p(sg), _p(bg), _p(wu), _p(su), _p(bu), K, N,
                                              bits, group, _p(cols), cols.size, _p(y)), "qmm_swiglu_f64_cols")
    return y


def qmm_spbxs_f64(x_bf16, words, scales, biases, K: int, N: int, bits: int, group: int) -> np.ndarray:
    """y = sum_g ( s*P + b*XS ) in float64 (the pages' dequant-after-dot form)."""
    x = _c(x_bf16, np.uint16).reshape(-1, K)
    w, s, b = _c(words, np.uint32), _c(scales, np.uint16), _c(biases, np.uint16)
    M = x.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    _check(_load().oracle_qmm_spbxs_f64(_p(x), M, _p(w), _p(s), _p(b), K, N, bits, group, _p(y)),
           "qmm_spbxs_f64")
    return y
