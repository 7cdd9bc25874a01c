"""Prefill-shaped GEMM (q8_gemm, M > 32, tcgen05) vs the oracle.

The weight tile is dequantised to bf16(s*q) (round to nearest even) before the
tensor-core product, and y is bf16, so the bound is T1 widened by half a bf16
ulp of the reference (the C9 reading); exactly representable cases must equal
bf16_rn(exact) bit for bit."""
import numpy as np
import pytest
import torch

import synth
from helpers import TOL_ABS, TOL_REL, weights_dev, x_dev

pytestmark = pytest.mark.gpu


def bf16_rn_bits(a: np.ndarray) -> np.ndarray:
    return synth.f32_to_bf16_bits(a.astype(np.float32))


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(b).astype(np.float64)


TILES = [1, 2, 3]  # Q8_GEMM_TILE_256x128, 128x128, 64x128
# (tile, splits): automatic, each tile unsplit, and splits of K over clusters
COMBOS = [(0, 0), (1, 1), (2, 1), (3, 1), (1, 2), (1, 3), (2, 3), (3, 4), (1, 8), (2, 8)]


def run_gemm(qn, sn, xn, tile=0, splits=0):
    from block_quantized_int8_gb300 import q8
    q, s = weights_dev(qn, sn)
    x = x_dev(xn)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    N = qn.shape[0]
    M = xn.shape[0]
    ldy = (N + 7) // 8 * 8
    ybuf = torch.full((M, ldy), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = ybuf[:, :N]
    q8.q8_gemm(q, s, x, y, dev_status=st, tile=tile, splits=splits)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return ybuf.cpu().view(torch.int16).numpy().view(np.uint16)[:, :N]


def _skip_if_too_many_splits(K, splits):
    if splits > (K + 255) // 256:
        pytest.skip("more splits than groups of 256 in K")


@pytest.mark.parametrize("tile,splits", COMBOS)
@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (256, 384, 1536), (200, 300, 96), (33, 129, 4096), (96, 200, 384), (64, 256, 640),
                                   (512, 1536, 4096), (300, 520, 160), (40, 200, 8192)])
def test_gemm_exact_cases(oracle, M, N, K, tile, splits):
    _skip_if_too_many_splits(K, splits)
    q, s, x = synth.exact_case(N, K, M, 0, f"gx{M}.{N}.{K}")
    y_ref, _ = oracle.matmul(q, s, x, threads=8)
    # exact sums are small integers times powers of two: fp32 holds them exactly,
    # so the only rounding is the final bf16 one
    got = run_gemm(q, s, x, tile, splits)
    assert np.array_equal(got, bf16_rn_bits(y_ref))


def _check_sampled(oracle, qn, sn, xn, got, tag, ncols=256):
    N = qn.shape[0]
    cols = np.unique(np.concatenate([synth.rng(0, tag).choice(N, min(ncols, N), replace=False), [0, N - 1]]))
    y_ref, B = oracle.matmul(qn[cols], sn[cols], xn, threads=16)
    half_ulp = np.abs(bf16_to_f64(bf16_rn_bits(y_ref))) * 2.0 ** -8
    err = np.abs(got[:, cols] - y_ref)
    lim = TOL_REL * B + TOL_ABS + half_ulp
    ratio = float(np.max(np.maximum(err - half_ulp, 0) / B))
    assert np.all(err <= lim), f"max err {err.max()}, max (err - ulp/2)/B {ratio:.3e}"
    return ratio


@pytest.mark.parametrize("K,N", list(synth.SWEEP_SHAPES) + [(8192, 1024)])
def test_gemm_prefill_full_size_sampled(oracle, K, N):
    """The M = 512 prefill shapes in the launch configuration the bench times
    (automatic tile and split), sampled columns against the oracle; plus a
    K = 8192 shape."""
    M = synth.PREFILL_M
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"pf{K}.{N}"))
    xn = synth.activations(M, K, 0, f"pfx{K}")
    got = bf16_to_f64(run_gemm(qn, sn, xn))
    _check_sampled(oracle, qn, sn, xn, got, f"pf.cols{N}")


@pytest.mark.parametrize("tile,splits", COMBOS)
@pytest.mark.parametrize("M,N,K", [(40, 520, 1536), (300, 77, 160), (129, 1000, 4096), (257, 130, 6144),
                                   (70, 260, 8224)])
def test_gemm_ragged_tolerance(oracle, M, N, K, tile, splits):
    _skip_if_too_many_splits(K, splits)
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"gr{M}.{N}.{K}"))
    xn = synth.activations(M, K, 0, f"grx{M}.{K}")
    got = bf16_to_f64(run_gemm(qn, sn, xn, tile, splits))
    y_ref, B = oracle.matmul(qn, sn, xn, threads=16)
    half_ulp = np.abs(bf16_to_f64(bf16_rn_bits(y_ref))) * 2.0 ** -8
    assert np.all(np.abs(got - y_ref) <= TOL_REL * B + TOL_ABS + half_ulp)


@pytest.mark.parametrize("splits", [1, 2, 4])
def test_gemm_tiles_agree_bitwise(oracle, splits):
    """With the same K split, every tile shape sums each output in the same
    order: the same bits."""
    N, K, M = 520, 1536, 300
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, "gtile"))
    xn = synth.activations(M, K, 0, "gtilex")
    outs = [run_gemm(qn, sn, xn, t, splits) for t in TILES]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


@pytest.mark.parametrize("tile,splits", [(1, 1), (2, 1), (3, 1), (1, 4)])
def test_gemm_weight_stage_reuse(oracle, tile, splits):
    """Every token reads one 8-code chunk of every weight row, so a code or A
    stage read after its refill began (or before its fill ended) changes the
    outputs of the tokens that read it.  Such a race depends on timing:
    several launches, three chunk assignments, bit-exact each time."""
    M, N, K = 512, 1536, 4096
    q, s, _ = synth.exact_case(N, K, M, 0, f"gx{M}.{N}.{K}")
    for shift in (0, 64, 128):
        x = synth.chunk_select_x(M, K, shift)
        y_ref, _ = oracle.matmul(q, s, x, threads=8)
        want = bf16_rn_bits(y_ref)
        for _ in range(3):
            assert np.array_equal(run_gemm(q, s, x, tile, splits), want)


def test_gemm_deterministic(oracle):
    N, K, M = 1536, 4096, 512
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, "gdet"))
    xn = synth.activations(M, K, 0, "gdetx")
    for tile, splits in ((0, 0), (1, 8), (2, 3)):
        a = run_gemm(qn, sn, xn, tile, splits)
        b = run_gemm(qn, sn, xn, tile, splits)
        assert np.array_equal(a, b)


def test_gemm_wide_range_activations(oracle):
    """Activations spanning the bf16 range (tiny, huge, zero): within the
    bound with and without a split of K."""
    N, K, M = 300, 2048, 96
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, "gwr"))
    xn = synth.wide_range_activations(M, K, 0, "gwrx")
    y_ref, B = oracle.matmul(qn, sn, xn, threads=16)
    half_ulp = np.abs(bf16_to_f64(bf16_rn_bits(y_ref))) * 2.0 ** -8
    for tile, splits in ((1, 1), (2, 4)):
        got = bf16_to_f64(run_gemm(qn, sn, xn, tile, splits))
        ok = np.isfinite(y_ref) & (np.abs(y_ref) < 3e38)
        assert np.all(np.abs(got - y_ref)[ok] <= (TOL_REL * B + TOL_ABS + half_ulp)[ok])
