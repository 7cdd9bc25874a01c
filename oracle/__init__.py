"""CPU oracle for the Q8_0 W8A16 decode matmul -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``q8ref.c`` (plain C, binary64
arithmetic, no code shared with the CUDA library) through ctypes, and builds it
with gcc on first use.

Functions and what they follow (page titles of the source pages):

* ``quantize_rows`` -- "MODEL-BASELINE-RESULTS" (fak), ACT 3 item 1 (32-wide
  blocks, d = maxabs/127, int8 codes, ~1.06 B/weight -> binary16 scale) and
  ACT 4 "Correctness" (round half away from zero, 0.49999997 -> 0).
* ``matmul`` -- "Frigg" README, Finding 8 (W8A16: int8 weights x bf16
  activations); dequantise-then-dot in binary64, plus the tolerance bound
  B = sum |w' x|.
* ``f32_to_f16`` / ``f16_to_f64`` / ``code`` -- the binary16 rounding and the
  single-weight code rule, exposed for exhaustive pins.
* ``quantize_rows_fl32`` / ``code_fl32`` -- the compatibility code rule: the
  binary32 quotient w / d32 rounded half away from zero ("MODEL-BASELINE-
  RESULTS" (fak), ACT 4 "Correctness": q8round of a float32 value), with the
  same binary16 stored scale.
* ``chain_next`` / ``f64_to_bf16`` -- the input of the next matmul of a
  dependent chain: RMS normalisation (no learnable weight, eps 1e-6) of the
  first K outputs, or of SwiGLU over the two halves ("Frigg" README, the
  model card), rounded once to bf16.
* ``gguf_to_planar`` / ``planar_to_gguf`` -- the GGUF Q8_0 block (34 bytes:
  binary16 scale, then 32 int8 codes; the model files of the "aubier" README,
  "Layout") split into planar codes and scales, and back: a numpy view of
  the byte array as records, no arithmetic.

Every function is pinned by the CPU test suite (see tests/test_oracle_*.py);
none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q8ref.c")
_LIB = os.path.join(_HERE, "libq8ref.so")
_lock = threading.Lock()
_lib = None

FLAG_NONFINITE = 1
FLAG_SCALE_OVF = 2


def build(force: bool = False) -> str:
    """Compile q8ref.c with gcc (no fast-math, no FP contraction)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call([
                "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.q8ref_f32_to_f16.argtypes = [ctypes.c_float]
        lib.q8ref_f32_to_f16.restype = ctypes.c_uint16
        lib.q8ref_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.q8ref_f16_to_f64.restype = ctypes.c_double
        lib.q8ref_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.q8ref_bf16_to_f64.restype = ctypes.c_double
        lib.q8ref_quantize_rows.argtypes = [P, I64, I64, P, P, P]
        lib.q8ref_quantize_rows.restype = ctypes.c_uint32
        lib.q8ref_matmul.argtypes = [P, P, I64, I64, P, I64, I64, I64, I64, P, P, I64]
        lib.q8ref_matmul.restype = None
        lib.q8ref_f32_to_f16_array.argtypes = [P, P, I64]
        lib.q8ref_f16_to_f64_array.argtypes = [P, P, I64]
        lib.q8ref_code_array.argtypes = [P, I64, ctypes.c_uint16, P]
        lib.q8ref_code_fl32_array.argtypes = [P, I64, ctypes.c_float, P]
        lib.q8ref_quantize_rows_fl32.argtypes = [P, I64, I64, P, P, P]
        lib.q8ref_quantize_rows_fl32.restype = ctypes.c_uint32
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def f32_to_f16(x) -> np.ndarray:
    """binary32 -> binary16 bits (uint16), round to nearest even."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().q8ref_f32_to_f16_array(_ptr(a), _ptr(out), a.size)
    return out


def f16_to_f64(h) -> np.ndarray:
    a = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(a.shape, dtype=np.float64)
    _load().q8ref_f16_to_f64_array(_ptr(a), _ptr(out), a.size)
    return out


def code(w, s_bits: int) -> np.ndarray:
    """Codes of the weights ``w`` against one stored binary16 scale."""
    a = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.int8)
    _load().q8ref_code_array(_ptr(a), a.size, ctypes.c_uint16(int(s_bits)), _ptr(out))
    return out


def code_fl32(w, d32: float) -> np.ndarray:
    """Compatibility codes of ``w`` against the binary32 scale ``d32``:
    round half away from zero of the binary32 quotient w / d32."""
    a = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.int8)
    _load().q8ref_code_fl32_array(_ptr(a), a.size, ctypes.c_float(float(np.float32(d32))), _ptr(out))
    return out


def quantize_rows_fl32(w: np.ndarray, with_flags: bool = False):
    """As ``quantize_rows``, with the compatibility codes (``code_fl32`` of
    each weight against d32 = amax/127 in binary32); same scales and flags."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    if w.ndim != 2 or w.shape[1] % 32:
        raise ValueError("w must be [rows][K] with K a multiple of 32")
    rows, K = w.shape
    q = np.empty((rows, K), dtype=np.int8)
    s = np.empty((rows, K // 32), dtype=np.uint16)
    fl = np.empty((rows, K // 32), dtype=np.uint32)
    allf = _load().q8ref_quantize_rows_fl32(_ptr(w), rows, K, _ptr(q), _ptr(s), _ptr(fl))
    return q, s, (fl if with_flags else int(allf))


def quantize_rows(w: np.ndarray, with_flags: bool = False):
    """Q8_0-quantize a [rows][K] binary32 matrix along K.

    Returns (q int8 [rows][K], s uint16 binary16 bits [rows][K/32], flags) where
    flags is the OR of all block flags, or the per-block array if
    ``with_flags``.
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    if w.ndim != 2 or w.shape[1] % 32:
        raise ValueError("w must be [rows][K] with K a multiple of 32")
    rows, K = w.shape
    q = np.empty((rows, K), dtype=np.int8)
    s = np.empty((rows, K // 32), dtype=np.uint16)
    fl = np.empty((rows, K // 32), dtype=np.uint32)
    allf = _load().q8ref_quantize_rows(_ptr(w), rows, K, _ptr(q), _ptr(s), _ptr(fl))
    return q, s, (fl if with_flags else int(allf))


_GGUF_Q8_0 = np.dtype([("d", "<u2"), ("qs", "i1", (32,))])  # 34 bytes, no padding


def gguf_to_planar(blocks: np.ndarray, rows: int, K: int):
    """Planar (q int8 [rows][K], s uint16 [rows][K/32]) of a GGUF Q8_0 byte
    array holding rows * K/32 consecutive blocks."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
    if b.size != rows * (K // 32) * 34:
        raise ValueError("blocks must hold rows * K/32 blocks of 34 bytes")
    rec = b.view(_GGUF_Q8_0)
    return rec["qs"].reshape(rows, K).copy(), rec["d"].reshape(rows, K // 32).copy()


def planar_to_gguf(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """GGUF Q8_0 bytes of planar codes q [rows][K] and scales s [rows][K/32]."""
    rows, K = q.shape
    rec = np.empty(rows * (K // 32), dtype=_GGUF_Q8_0)
    rec["d"] = np.asarray(s, dtype=np.uint16).reshape(-1)
    rec["qs"] = np.asarray(q, dtype=np.int8).reshape(-1, 32)
    return rec.view(np.uint8).copy()


def matmul(q: np.ndarray, s: np.ndarray, x_bf16: np.ndarray, rows=None, threads: int = 1):
    """Binary64 reference y[m][n] and bound B[m][n] for output rows ``rows``.

    ``rows`` is None (all N rows) or an increasing array of row indices; the
    result then has one column per listed row.  ``threads`` > 1 splits the rows
    over host threads; every output is computed by one call in the same order,
    so the bits do not depend on the thread count.
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    N, K = q.shape
    M = x.shape[0]
    if s.shape != (N, K // 32) or x.shape[1] != K:
        raise ValueError("shape mismatch")
    if rows is None:
        y = np.empty((M, N), dtype=np.float64)
        B = np.empty((M, N), dtype=np.float64)
        chunks = np.array_split(np.arange(N), max(1, threads))

        def run(c):
            if len(c):
                lib.q8ref_matmul(_ptr(q), _ptr(s), N, K, _ptr(x), K, M,
                                 int(c[0]), int(c[-1]) + 1, _ptr(y), _ptr(B), N)

        if threads > 1:
            with ThreadPoolExecutor(threads) as ex:
                list(ex.map(run, chunks))
        else:
            run(np.arange(N))
        return y, B
    rows = np.asarray(rows, dtype=np.int64)
    qs = np.ascontiguousarray(q[rows])
    ss = np.ascontiguousarray(s[rows])
    return matmul(qs, ss, x, None, threads)


def matmul_w8a8(q: np.ndarray, s: np.ndarray, x_bf16: np.ndarray):
    """W8A8 reference: each activation row is Q8_0-quantized by the same rule
    as the weights (``quantize_rows`` of its binary32 value), then
    y[m][n] = sum_b s_w[n][b] s_x[m][b] sum_{k in b} q_w[n][k] q_x[m][k].
    That is the plain dot product of the dequantised weights and the
    dequantised activations, taken here in binary64 by a library matmul
    (every product s q is exact in binary64).  Source: "MODEL-BASELINE-
    RESULTS" (fak), ACT 3 item 1 (weights and activations both in 32-element
    Q8_0 blocks) and item 3 (the int8 block dot product).  Returns (y, B)
    with B = sum |w'| |x'| for the tolerance."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    N, K = q.shape
    if s.shape != (N, K // 32) or x.shape[1] != K:
        raise ValueError("shape mismatch")
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    qx, sx, _ = quantize_rows(xf)
    wd = q.astype(np.float64) * np.repeat(f16_to_f64(s), 32, axis=1)
    xd = qx.astype(np.float64) * np.repeat(f16_to_f64(sx), 32, axis=1)
    return xd @ wd.T, np.abs(xd) @ np.abs(wd).T


def f64_to_bf16(v) -> np.ndarray:
    """binary64 -> bf16 bits (uint16), one rounding to nearest, ties to even.

    bf16 is binary32 with 8 significant bits: normal values x = m 2^e with
    1 <= |m| < 2 keep m to 2^-7, values below 2^-126 are multiples of
    2^-133, and values at or above (2 - 2^-8) 2^127 round to infinity."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.uint16)
    a = np.abs(v)
    sign = np.where(np.signbit(v), 0x8000, 0).astype(np.uint32)
    with np.errstate(over="ignore", invalid="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
        # log2 of a binary64 may land one off next to a power of two
        e = np.where(np.ldexp(1.0, e.astype(np.int64)) > a, e - 1, e)
        e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= a, e + 1, e)
        step = np.ldexp(1.0, (np.maximum(e, -126) - 7).astype(np.int64))  # the spacing at a
        r = np.rint(a / step) * step  # exact: a / step and its product are exact in binary64
    r = np.where(a == 0, 0.0, r)
    big = r >= np.ldexp(1.0, 128)
    bits32 = np.where(big, 0x7F800000, np.where(big, 0.0, r).astype(np.float32).view(np.uint32)).astype(np.uint32)
    bits32 = np.where(np.isnan(v), 0x7FC00000, bits32)
    bits32 = np.where(np.isinf(v), 0x7F800000, bits32)
    out[...] = ((bits32 >> 16) | sign).astype(np.uint16)
    return out


def chain_next(y: np.ndarray, K: int, swiglu: bool) -> np.ndarray:
    """The next input of a dependent matmul chain, from y [M][N] (binary64
    arithmetic on the given values): per row, v = y[0:K] or, with SwiGLU,
    v[k] = silu(y[k]) * y[K + k] with silu(a) = a / (1 + e^-a); then
    x = v / sqrt(mean(v^2) + 1e-6), rounded once to bf16 (``f64_to_bf16``).
    Source: "Frigg" README, the model card (RMSNorm with no learnable weight,
    eps 1e-6; the SwiGLU MLP between gate+up and down).  Returns bf16 bits
    [M][K]."""
    y = np.asarray(y, dtype=np.float64)
    if y.ndim == 1:
        y = y[None, :]
    if swiglu:
        a, b = y[:, :K], y[:, K:2 * K]
        v = a / (1.0 + np.exp(-a)) * b
    else:
        v = y[:, :K]
    ms = np.mean(v * v, axis=1, keepdims=True)
    return f64_to_bf16(v / np.sqrt(ms + 1e-6))
