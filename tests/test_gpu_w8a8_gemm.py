"""q8_gemm_w8a8: the W8A8 product for any M (a prefill of 512 rows, M with a
remainder of rows, and M = 2100: more slices than one launch takes) against
the oracle's W8A8 definition, and bit for
bit equal to the W8A8 variant of q8_linear_batch run on each 32-row slice
(the slices are the matrices of its launches)."""
import numpy as np
import pytest
import torch

import synth
from helpers import check_tol, weights_dev, x_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K,M", [(8192, 1536, 512), (1536, 4096, 512), (1000, 2080, 100), (300, 1536, 33),
                                   (260, 1536, 2100)])
def test_gemm_w8a8_against_oracle(oracle, N, K, M):
    from block_quantized_int8_gb300 import q8
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"gw{N}.{K}"))
    xn = synth.activations(M, K, 0, f"gwx{M}.{K}")
    q, s = weights_dev(qn, sn)
    x = x_dev(xn)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = q8.q8_gemm_w8a8(q, s, x, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    y_ref, B = oracle.matmul_w8a8(qn, sn, xn)
    check_tol(y.cpu().numpy(), y_ref, B, f"W8A8 GEMM N={N} K={K} M={M}")
    # each 32-row slice alone through the W8A8 variant gives the same bits
    for r0 in range(0, M, 32):
        xs = x[r0:r0 + 32]
        ys = torch.empty((xs.shape[0], N), dtype=torch.float32, device="cuda")
        q8.q8_linear_batch([(q, s, xs, ys)], variant=q8.Q8_VARIANT_W8A8)
        torch.cuda.synchronize()
        assert torch.equal(ys.view(torch.int32), y[r0:r0 + 32].view(torch.int32)), f"slice at row {r0}"


def test_gemm_w8a8_repeat_and_graph(oracle):
    """Repeated calls and graph replays on one workspace give the same bits."""
    from block_quantized_int8_gb300 import q8
    N, K, M = 1536, 1536, 200
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, "gwr"))
    q, s = weights_dev(qn, sn)
    x = x_dev(synth.activations(M, K, 0, "gwrx"))
    ws = q8.workspace(int(q8.lib().q8_gemm_w8a8_workspace_size(N, K, M)))
    y0 = q8.q8_gemm_w8a8(q, s, x, ws=ws)
    y1 = q8.q8_gemm_w8a8(q, s, x, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int32), y1.view(torch.int32))
    y2 = torch.full_like(y0, float("nan"))
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            q8.q8_gemm_w8a8(q, s, x, y=y2, ws=ws, stream=stream)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int32), y2.view(torch.int32))
