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


TILES = [0, 1, 2, 3]  # Q8_GEMM_TILE_AUTO, 256x128, 128x128, 128x64


def run_gemm(qn, sn, xn, tile=0):
    from block_quantized_int8_gb300 import q8
    q, s = weights_dev(qn, sn)
    x = x_dev(xn)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    N = qn.shape[0]
    M = xn.shape[0]
    ldy = (N + 7) // 8 * 8
    ybuf = torch.full((M, ldy), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = ybuf[:, :N]
    q8.q8_gemm(q, s, x, y, dev_status=st, tile=tile)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return ybuf.cpu().view(torch.int16).numpy().view(np.uint16)[:, :N]


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("M,N,K", [(128, 128, 64), (256, 384, 1536), (200, 300, 96), (33, 129, 4096),
                                   (512, 1536, 4096), (300, 520, 160)])
def test_gemm_exact_cases(oracle, M, N, K, tile):
    q, s, x = synth.exact_case(N, K, M, 0, f"gx{M}.{N}.{K}")
    y_ref, _ = oracle.matmul(q, s, x, threads=8)
    # exact sums are small integers times powers of two: fp32 holds them exactly,
    # so the only rounding is the final bf16 one
    got = run_gemm(q, s, x, tile)
    assert np.array_equal(got, bf16_rn_bits(y_ref))


@pytest.mark.parametrize("K,N", synth.SWEEP_SHAPES)
def test_gemm_prefill_full_size_sampled(oracle, K, N):
    M = synth.PREFILL_M
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"pf{K}.{N}"))
    xn = synth.activations(M, K, 0, f"pfx{K}")
    got = bf16_to_f64(run_gemm(qn, sn, xn))
    cols = np.unique(np.concatenate([synth.rng(0, f"pf.cols{N}").choice(N, 256, replace=False), [0, N - 1]]))
    y_ref, B = oracle.matmul(qn[cols], sn[cols], xn, threads=16)
    half_ulp = np.abs(bf16_to_f64(bf16_rn_bits(y_ref))) * 2.0 ** -8
    err = np.abs(got[:, cols] - y_ref)
    lim = TOL_REL * B + TOL_ABS + half_ulp
    ratio = float(np.max(np.maximum(err - half_ulp, 0) / B))
    assert np.all(err <= lim), f"max err {err.max()}, max (err - ulp/2)/B {ratio:.3e}"


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("M,N,K", [(40, 520, 1536), (300, 77, 160), (129, 1000, 4096), (257, 130, 6144)])
def test_gemm_ragged_tolerance(oracle, M, N, K, tile):
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"gr{M}.{N}.{K}"))
    xn = synth.activations(M, K, 0, f"grx{M}.{K}")
    got = bf16_to_f64(run_gemm(qn, sn, xn, tile))
    y_ref, B = oracle.matmul(qn, sn, xn, threads=16)
    half_ulp = np.abs(bf16_to_f64(bf16_rn_bits(y_ref))) * 2.0 ** -8
    assert np.all(np.abs(got - y_ref) <= TOL_REL * B + TOL_ABS + half_ulp)


def test_gemm_tiles_agree_bitwise(oracle):
    """Every tile shape sums each output over K in the same order."""
    N, K, M = 520, 1536, 300
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, "gtile"))
    xn = synth.activations(M, K, 0, "gtilex")
    outs = [run_gemm(qn, sn, xn, t) for t in TILES]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_gemm_deterministic(oracle):
    N, K, M = 1536, 4096, 512
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, "gdet"))
    xn = synth.activations(M, K, 0, "gdetx")
    a = run_gemm(qn, sn, xn)
    b = run_gemm(qn, sn, xn)
    assert np.array_equal(a, b)


def test_gemm_rejects_too_large_k():
    from block_quantized_int8_gb300 import q8
    N, K, M = 128, 8192, 64
    q = torch.zeros((N, K), dtype=torch.int8, device="cuda")
    s = torch.zeros((N, K // 32), dtype=torch.float16, device="cuda")
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(q8.Q8Error) as e:
        q8.q8_gemm(q, s, x)
    assert e.value.status == q8.Q8_ERR_UNSUPPORTED
