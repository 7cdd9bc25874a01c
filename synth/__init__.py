"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the method (no block maxima, no scales, no
rounding of codes, no dot products).  It only draws random numbers and lays
out special values, so that the oracle and the CUDA path see the same inputs.

Every tensor is drawn from ``numpy.random.PCG64`` seeded with
``SeedSequence([seed, crc32(tag), chunk])``: the same (seed, tag) always gives
the same numbers on any machine, and different tags give independent streams.

Workload recipe (shapes, distributions) follows the decode matmul it feeds:
weights ~ N(0, 0.02) in binary32 (quantized to Q8_0 before use), activations
~ N(0, 1) rounded to bfloat16 (the vocab projection uses a unit-norm vector, an
RMS-normalised row scaled by 1/sqrt(K)).
"""
from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

W_STD = 0.02


def rng(seed: int, tag: str) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed) & 0xFFFFFFFF, zlib.crc32(tag.encode())])
    return np.random.Generator(np.random.PCG64(ss))


_CHUNK = 1 << 22


def normal_f32(shape, seed: int, tag: str, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) binary32 draws.  The flat array is filled in fixed chunks of
    2^22 values, chunk i from its own stream (seed, crc32(tag), i), so the
    values do not depend on how many threads fill it."""
    shape = (shape,) if isinstance(shape, (int, np.integer)) else tuple(shape)
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.float32)
    crc = zlib.crc32(tag.encode())
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def fill(i):
        ss = np.random.SeedSequence([int(seed) & 0xFFFFFFFF, crc, i])
        g = np.random.Generator(np.random.PCG64(ss))
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        g.standard_normal(out=out[lo:hi], dtype=np.float32)
        if std != 1.0:
            out[lo:hi] *= np.float32(std)

    if nchunks > 1:
        with ThreadPoolExecutor(min(nchunks, os.cpu_count() or 4)) as ex:
            list(ex.map(fill, range(nchunks)))
    elif n:
        fill(0)
    return out.reshape(shape)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """binary32 -> bfloat16 bits, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def weights(N: int, K: int, seed: int = 0, tag: str = "W") -> np.ndarray:
    """Binary32 weight matrix [N][K] ~ N(0, 0.02)."""
    return normal_f32((N, K), seed, tag, W_STD)


def activations(M: int, K: int, seed: int = 0, tag: str = "x") -> np.ndarray:
    """bf16 bits [M][K] of N(0, 1) draws."""
    return f32_to_bf16_bits(normal_f32((M, K), seed, tag))


def wide_range_activations(M: int, K: int, seed: int = 0, tag: str = "xwide") -> np.ndarray:
    """bf16 bits [M][K] of N(0, 1) draws times magnitudes spread over the whole
    bf16 range: per element one of 2^-130 (bf16 subnormal), 2^-60, 2^-20, 1,
    2^20, 2^60; every 7th element zero; row 0 keeps only the tiny magnitudes
    and row 1 holds one huge element (2^100) among values near 1."""
    r = rng(seed, tag)
    g = normal_f32((M, K), seed, tag)
    mags = np.array([2.0 ** -130, 2.0 ** -60, 2.0 ** -20, 1.0, 2.0 ** 20, 2.0 ** 60])
    pick = r.integers(0, len(mags), size=(M, K))
    x = g.astype(np.float64) * mags[pick]
    x[:, ::7] = 0.0
    if M > 0:
        x[0] = g[0] * mags[r.integers(0, 2, size=K)]
    if M > 1:
        x[1] = g[1]
        x[1, K // 3] = 2.0 ** 100
    return f32_to_bf16_bits(x.astype(np.float32))


def unit_activation(K: int, seed: int = 0, tag: str = "x_vocab") -> np.ndarray:
    """bf16 bits [1][K] of g/||g||_2, g ~ N(0,1)^K (RMS-normalised, times 1/sqrt(K))."""
    g = rng(seed, tag).standard_normal(size=K, dtype=np.float64)
    g /= np.sqrt(np.sum(g * g))
    return f32_to_bf16_bits(g.astype(np.float32))[None, :]


# --------------------------------------------------------------------------
# Named workloads (sizes of the decode matmuls being modelled)
# --------------------------------------------------------------------------
HIDDEN = 1536
INTER = 4096
# one layer of a 16-layer module: (name, K, N)
LAYER_MATRICES = (("qkv", HIDDEN, 3 * HIDDEN),
                  ("o_proj", HIDDEN, HIDDEN),
                  ("gate_up", HIDDEN, 2 * INTER),
                  ("down", INTER, HIDDEN))
LAYERS = 16
PASSES = 8
VOCAB = 262144
SWEEP_M = (2, 4, 8, 16, 32)
SWEEP_SHAPES = ((HIDDEN, 2 * INTER), (INTER, HIDDEN))  # (K, N)
PREFILL_M = 512
ODD_K_SHAPE = (2080, 4608)  # (K, N): K % 256 = 32, a shape off the 256 grid


def layer_weight_tag(layer: int, name: str) -> str:
    return f"L{layer}.{name}"


def layer_x_tag(pass_idx: int, K: int) -> str:
    return f"P{pass_idx}.x{K}"


# --------------------------------------------------------------------------
# Quantizer stress rows: 32 x 4096 binary32, N(0, 0.02) with injected blocks
# --------------------------------------------------------------------------
def _f16_normal_value(exp: int, mant: int) -> np.float32:
    """A binary16-representable normal value (1 + mant/1024) * 2^exp as binary32."""
    return np.float32(np.ldexp(1.0 + mant / 1024.0, exp))


def exact_half_block(s: np.float32, sign: float = 1.0, rng_=None) -> np.ndarray:
    """32 values: one +-127*s (the block maximum) and +-(k+1/2)*s for k in a spread
    of 0..126, all exactly representable, so that the block scale is s and every
    other element sits exactly on a rounding tie."""
    ks = np.arange(31) * 4 % 127 if rng_ is None else rng_.integers(0, 127, size=31)
    vals = (ks.astype(np.float64) + 0.5) * float(s)
    signs = np.where(np.arange(31) % 2 == 0, 1.0, -1.0) * sign
    blk = np.empty(32, dtype=np.float64)
    blk[0] = 127.0 * float(s) * sign
    blk[1:] = vals * signs
    out = blk.astype(np.float32)
    assert np.array_equal(out.astype(np.float64), blk), "construction must be exact"
    return out


def quant_stress_rows(rows: int = 32, K: int = 4096, seed: int = 0) -> np.ndarray:
    """Binary32 [rows][K] ~ N(0, 0.02) with special blocks injected:
    all-zero, all -0.0, binary32 denormals, exact halves (several scales),
    a single spike, a negative block maximum, tiny blocks whose scale is a
    binary16 subnormal, blocks just around the binary16 normal threshold, and
    the 0.49999997 pitfall value."""
    w = weights(rows, K, seed, "quant_stress")
    g = rng(seed, "quant_stress.special")
    nb = K // 32
    blocks = w.reshape(rows, nb, 32)
    kinds = []
    for r in range(rows):
        for b in range(0, nb, 7):
            kind = (r * 131 + b) % 11
            kinds.append(kind)
            if kind == 0:
                blocks[r, b] = 0.0
            elif kind == 1:
                blocks[r, b] = np.float32(-0.0)
            elif kind == 2:  # binary32 denormals
                blocks[r, b] = (g.integers(-2**20, 2**20, size=32).astype(np.float32)
                                * np.float32(2.0 ** -149))
            elif kind == 3:  # exact halves, scale a normal binary16 value
                s = _f16_normal_value(int(g.integers(-14, 10)), int(g.integers(0, 1024)))
                blocks[r, b] = exact_half_block(s, 1.0 if r % 2 else -1.0, g)
            elif kind == 4:  # single spike
                blocks[r, b] = g.standard_normal(32).astype(np.float32) * np.float32(1e-3)
                blocks[r, b, int(g.integers(0, 32))] = np.float32(3.0)
            elif kind == 5:  # negative maximum
                blocks[r, b] = np.abs(g.standard_normal(32)).astype(np.float32) * np.float32(0.01)
                blocks[r, b, int(g.integers(0, 32))] = np.float32(-0.5)
            elif kind == 6:  # scale becomes a binary16 subnormal
                blocks[r, b] = (g.standard_normal(32) * 1e-4).astype(np.float32)
            elif kind == 7:  # around the binary16 normal threshold 127 * 2^-14
                blocks[r, b] = (g.uniform(-1, 1, 32) * 127 * 2.0 ** -14
                                * (1 + g.uniform(-0.01, 0.01))).astype(np.float32)
            elif kind == 8:  # the pitfall value 0.49999997 with scale exactly 1
                blocks[r, b] = g.uniform(-0.4, 0.4, 32).astype(np.float32)
                blocks[r, b, 0] = np.float32(127.0)
                blocks[r, b, 1] = np.float32(0.49999997)
                blocks[r, b, 2] = np.float32(-0.49999997)
                blocks[r, b, 3] = np.float32(0.5)
                blocks[r, b, 4] = np.float32(-2.5)
            elif kind == 9:  # large but finite values, scale near the binary16 maximum
                blocks[r, b] = (g.uniform(-1, 1, 32) * 127 * 60000.0).astype(np.float32)
            else:  # plain block, left as drawn
                pass
    return blocks.reshape(rows, K)


# --------------------------------------------------------------------------
# Exactly representable matmul inputs: every product and partial sum is an
# integer multiple of a power of two below 2^24, so binary32 sums in any order
# are exact and the GPU must equal the oracle bit for bit.
# --------------------------------------------------------------------------
def exact_case(N: int, K: int, M: int, seed: int = 0, tag: str = "exact"):
    """Returns (q int8 [N][K], s binary16 bits [N][K/32], x bf16 bits [M][K])."""
    g = rng(seed, tag)
    q = g.integers(-7, 8, size=(N, K)).astype(np.int8)
    # scales 2^e for e in [-3, 2]: binary16 bits = (e + 15) << 10
    e = g.integers(-3, 3, size=(N, K // 32))
    s = ((e + 15) << 10).astype(np.uint16)
    xi = g.integers(-8, 9, size=(M, K)).astype(np.float32)
    x = f32_to_bf16_bits(xi)
    return q, s, x


def chunk_select_x(M: int, K: int, shift: int = 0, width: int = 8) -> np.ndarray:
    """bf16 bits [M][K]: token m is 1 on the `width` consecutive k of chunk
    (m + shift) mod (K / width) and 0 elsewhere, so each output reads exactly
    one chunk of one weight row (a stale or early-overwritten weight stage
    shows up in the outputs of the tokens that read it)."""
    x = np.zeros((M, K), dtype=np.float32)
    chunk = (np.arange(M) + shift) % (K // width)
    for m in range(M):
        x[m, width * chunk[m]: width * chunk[m] + width] = 1.0
    return f32_to_bf16_bits(x)


def unit_vector_x(K: int, k: int) -> np.ndarray:
    x = np.zeros((1, K), dtype=np.float32)
    x[0, k] = 1.0
    return f32_to_bf16_bits(x)
