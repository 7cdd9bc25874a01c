"""GGUF Q8_0 repack on the GPU against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _raw(nblocks, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 256, size=34 * nblocks, dtype=np.uint8)


@pytest.mark.parametrize("rows,K", [(1, 32), (1, 64), (3, 96), (7, 160), (33, 1536), (257, 4096), (1000, 2080)])
def test_ingest_matches_oracle(oracle, rows, K):
    from block_quantized_int8_gb300 import q8
    raw = _raw(rows * K // 32, rows * 7919 + K)
    q_ref, s_ref = oracle.gguf_to_planar(raw, rows, K)
    q, s = q8.q8_gguf_to_planar(torch.from_numpy(raw).cuda(), rows, K)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().view(torch.int16).numpy().view(np.uint16), s_ref)


@pytest.mark.parametrize("rows,K", [(1, 32), (5, 96), (257, 4096), (999, 1536)])
def test_export_matches_oracle_and_round_trips(oracle, rows, K):
    from block_quantized_int8_gb300 import q8
    rng = np.random.default_rng(rows + K)
    q_np = rng.integers(-128, 128, size=(rows, K), dtype=np.int8)
    s_np = rng.integers(0, 65536, size=(rows, K // 32), dtype=np.uint16)
    raw_ref = oracle.planar_to_gguf(q_np, s_np)
    q = torch.from_numpy(q_np).cuda()
    s = torch.from_numpy(s_np.view(np.int16)).cuda().view(torch.float16)
    raw = q8.q8_planar_to_gguf(q, s)
    q2, s2 = q8.q8_gguf_to_planar(raw, rows, K)
    torch.cuda.synchronize()
    assert np.array_equal(raw.cpu().numpy(), raw_ref)
    assert torch.equal(q2, q) and torch.equal(s2.view(torch.int16), s.view(torch.int16))


def test_ingested_weights_multiply_like_quantized_ones(oracle):
    """A matrix quantized here, written as GGUF and read back, gives the same
    matmul bits as the original planar tensors."""
    from block_quantized_int8_gb300 import q8
    N, K = 1536, 1536
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, "gguf.w"))
    raw = oracle.planar_to_gguf(qn, sn)
    q, s = q8.q8_gguf_to_planar(torch.from_numpy(raw).cuda(), N, K)
    x = torch.from_numpy(synth.activations(1, K, 0, "gguf.x").view(np.int16)).cuda().view(torch.bfloat16)
    y1 = torch.empty((1, N), dtype=torch.float32, device="cuda")
    y2 = torch.empty_like(y1)
    q8.q8_linear_batch([(q, s, x, y1)])
    q0 = torch.from_numpy(qn).cuda()
    s0 = torch.from_numpy(sn.view(np.int16)).cuda().view(torch.float16)
    q8.q8_linear_batch([(q0, s0, x, y2)])
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_argument_checks():
    from block_quantized_int8_gb300 import q8
    L = q8.lib()
    b = torch.zeros(34 * 4, dtype=torch.uint8, device="cuda")
    q = torch.zeros((2, 64), dtype=torch.int8, device="cuda")
    s = torch.zeros((2, 2), dtype=torch.float16, device="cuda")
    assert L.q8_gguf_to_planar(q8._p(b), 2, 48, q8._p(q), q8._p(s), None) == q8.Q8_ERR_SHAPE
    assert L.q8_gguf_to_planar(None, 2, 64, q8._p(q), q8._p(s), None) == q8.Q8_ERR_ARG
    assert L.q8_gguf_to_planar(b.data_ptr() + 2, 2, 64, q8._p(q), q8._p(s), None) == q8.Q8_ERR_ALIGN
    assert L.q8_planar_to_gguf(q8._p(q), q8._p(s), 2, 64, b.data_ptr() + 2, None) == q8.Q8_ERR_ALIGN
    assert L.q8_gguf_to_planar(q8._p(b), 0, 64, None, None, None) == q8.Q8_OK
