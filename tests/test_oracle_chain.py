"""Pins of the oracle's chain step (``chain_next``) and its bf16 rounding
(``f64_to_bf16``) against values fixed by the definitions: the bf16 format
(8 significant bits, binary32's exponent range, ties to even), hand-derived
cases of RMS normalisation (no learnable weight, eps 1e-6) and of SwiGLU,
and an independent rounding route for every binary32 input."""
import math

import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("v,bits", [
    (1.0, 0x3F80), (-2.0, 0xC000), (0.0, 0x0000), (-0.0, 0x8000),
    (1 + 2 ** -7, 0x3F81),                 # representable
    (1 + 2 ** -8, 0x3F80),                 # tie -> even (down)
    (1 + 3 * 2 ** -8, 0x3F82),             # tie -> even (up)
    (1 + 2 ** -8 + 2 ** -40, 0x3F81),      # just above the tie
    (2.0 ** -126, 0x0080),                 # smallest normal
    (2.0 ** -133, 0x0001),                 # smallest subnormal
    (3 * 2.0 ** -134, 0x0002),             # subnormal tie -> even (up)
    (2.0 ** -134, 0x0000),                 # subnormal tie -> even (down to zero)
    ((2 - 2 ** -7) * 2.0 ** 127, 0x7F7F),  # largest finite
    ((2 - 2 ** -8) * 2.0 ** 127, 0x7F80),  # rounds to infinity
    (1e300, 0x7F80), (-math.inf, 0xFF80),
])
def test_f64_to_bf16_values(v, bits):
    assert int(oracle.f64_to_bf16(v)) == bits


def test_f64_to_bf16_nan():
    b = int(oracle.f64_to_bf16(float("nan")))
    assert (b & 0x7F80) == 0x7F80 and (b & 0x7F) != 0


def test_f64_to_bf16_matches_integer_rounding_of_binary32():
    """For a binary32 input the binary64 route must agree with rounding the
    binary32 bit pattern to its upper 16 bits by adding 0x7FFF plus the kept
    lowest bit (round to nearest, ties to even, carrying into the exponent),
    over normal, subnormal and near-overflow values of both signs."""
    g = np.random.default_rng(7)
    bits = g.integers(0, 1 << 32, size=200000, dtype=np.uint64).astype(np.uint32)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]  # finite only
    f = bits.view(np.float32)
    want = ((bits.astype(np.uint64) + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)
    got = oracle.f64_to_bf16(f.astype(np.float64))
    assert np.array_equal(got, want)


def test_chain_next_rmsnorm_constant_rows():
    # a row of c's: c / sqrt(c^2 + 1e-6); c = 2 -> 0.99999987 -> bf16 1.0;
    # c = 1e-3 -> 1 / sqrt(2) = 0.70710678 -> 1.0110101 x 2^-1 -> 0x3F35
    y = np.array([[2.0] * 8 + [5.0] * 4, [1e-3] * 8 + [7.0] * 4])
    x = oracle.chain_next(y, 8, swiglu=False)
    assert x.shape == (2, 8)
    assert np.all(x[0] == 0x3F80) and np.all(x[1] == 0x3F35)


def test_chain_next_swiglu_hand_case():
    # a = (ln 3, -ln 3), b = (1, 1): silu(ln 3) = ln 3 / (1 + 1/3) = 0.75 ln 3,
    # silu(-ln 3) = -ln 3 / 4; v = ln 3 (0.75, -0.25), mean v^2 = 0.3125 ln^2 3,
    # so x = (0.75, -0.25) / sqrt(0.3125) = (1.34164, -0.44721) up to eps:
    # 1.34164 -> 1 + 44/128 (0x3FAC); 0.44721 = 1.78885 x 2^-2 -> 1 + 101/128 (0xBEE5)
    a = math.log(3.0)
    x = oracle.chain_next(np.array([[a, -a, 1.0, 1.0]]), 2, swiglu=True)
    assert [int(v) for v in x[0]] == [0x3FAC, 0xBEE5]


def test_chain_next_zero_gates_and_rows():
    g = np.random.default_rng(3)
    b = g.standard_normal((3, 64))
    # silu(0) = 0 and a zero b give a zero row (of either sign); eps keeps it finite
    def zero(x):
        return not (x & 0x7FFF).any()
    assert zero(oracle.chain_next(np.concatenate([np.zeros((3, 64)), b], axis=1), 64, True))
    assert zero(oracle.chain_next(np.concatenate([b, np.zeros((3, 64))], axis=1), 64, True))
    assert not oracle.chain_next(np.zeros((2, 100)), 100, False).any()


def test_chain_next_rms_is_one_and_reads_only_its_columns():
    g = np.random.default_rng(5)
    y = g.standard_normal((4, 4608)) * 3.0
    x = oracle.chain_next(y, 1536, swiglu=False)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ms = np.mean(y[:, :1536] ** 2, axis=1)
    # mean(x^2) = ms / (ms + eps) before rounding; each value within 2^-8
    assert np.allclose(np.mean(xf * xf, axis=1), ms / (ms + 1e-6), rtol=2 ** -7)
    # the outputs past K do not enter
    y2 = y.copy()
    y2[:, 1536:] = 1e30
    assert np.array_equal(oracle.chain_next(y2, 1536, False), x)
    # signs follow y, and a larger |y| never gives a smaller |x| (one positive
    # factor per row, then a monotone rounding)
    assert np.array_equal(np.sign(xf), np.sign(y[:, :1536]))
    order = np.argsort(np.abs(y[0, :1536]))
    assert np.all(np.diff(np.abs(xf[0][order])) >= 0)
