"""Quantizer kernel vs the oracle: bit-exact codes and binary16 scale bits,
and the same device status flags (q8_quantize_rows)."""
import hashlib

import numpy as np
import pytest
import torch

import synth
from helpers import dev

pytestmark = pytest.mark.gpu


def gpu_quantize(w: np.ndarray):
    from block_quantized_int8_gb300 import q8
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, s = q8.q8_quantize_rows(dev(w), dev_status=st)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().view(torch.int16).numpy().view(np.uint16), int(st.item())


def digest(q, s):
    return hashlib.sha256(q.tobytes() + s.tobytes()).hexdigest()


def test_quantize_stress_rows_bit_exact(oracle):
    w = synth.quant_stress_rows(32, 4096, 0)
    q_ref, s_ref, fl = oracle.quantize_rows(w)
    q, s, st = gpu_quantize(w)
    assert fl == 0 and st == 0
    assert np.array_equal(q, q_ref)
    assert np.array_equal(s, s_ref)
    assert digest(q, s) == digest(q_ref, s_ref)


@pytest.mark.parametrize("rows,K", [(1, 32), (3, 96), (257, 1536), (1000, 4096), (4096, 1536)])
def test_quantize_random_bit_exact(oracle, rows, K):
    w = synth.weights(rows, K, 0, f"qr{rows}.{K}")
    q_ref, s_ref, _ = oracle.quantize_rows(w)
    q, s, st = gpu_quantize(w)
    assert st == 0
    assert np.array_equal(q, q_ref) and np.array_equal(s, s_ref)


def test_quantize_exact_halves_all_scales(oracle):
    # every binary16 exponent, with tie elements in every position
    g = synth.rng(0, "halves")
    rows = []
    for e in range(-14, 16):
        for _ in range(4):
            s = np.float32(np.ldexp(1.0 + int(g.integers(0, 1024)) / 1024.0, e))
            if 127.0 * float(s) > 3.0e38 or 127.0 * float(s) > 127 * 65504:
                continue
            rows.append(synth.exact_half_block(s, 1.0 if len(rows) % 2 else -1.0, g))
    n = len(rows) // 8 * 8
    w = np.stack(rows[:n]).reshape(-1, 32 * 8)
    q_ref, s_ref, fl = oracle.quantize_rows(w)
    q, s, st = gpu_quantize(w)
    assert fl == 0 and st == 0
    assert np.array_equal(q, q_ref) and np.array_equal(s, s_ref)


def test_quantize_nonfinite_and_overflow_flags(oracle):
    w = synth.weights(4, 256, 0, "qflags")
    w[0, 5] = np.nan
    w[1, 40] = -np.inf
    w[2, 200] = np.float32(127.0 * 65520.0)
    w[3, 31] = np.float32(127.0 * 65504.0)
    q_ref, s_ref, fl = oracle.quantize_rows(w)
    q, s, st = gpu_quantize(w)
    assert np.array_equal(q, q_ref) and np.array_equal(s, s_ref)
    assert st == fl == (oracle.FLAG_NONFINITE | oracle.FLAG_SCALE_OVF)


def test_quantize_vocab_weight_creation_bit_exact(oracle):
    # the 262144 x 1536 vocab matrix as created for the vocab-projection GEMV
    w = synth.weights(synth.VOCAB, synth.HIDDEN, 0, "vocab")
    q, s, st = gpu_quantize(w)
    assert st == 0
    # the oracle on a spread of row ranges (whole blocks, many tiles)
    for r0 in [0, 1, 4095, 100000, synth.VOCAB - 700]:
        rr = slice(r0, r0 + 700)
        q_ref, s_ref, _ = oracle.quantize_rows(w[rr])
        assert np.array_equal(q[rr], q_ref) and np.array_equal(s[rr], s_ref)


def test_quantize_empty_is_noop():
    from block_quantized_int8_gb300 import q8
    w = torch.empty((0, 64), dtype=torch.float32, device="cuda")
    q, s = q8.q8_quantize_rows(w)
    assert q.shape == (0, 64) and s.shape == (0, 2)


# ---------------------------------------------------------------------------
# compatibility mode: half-away rounding of the binary32 quotient w / d32
# ---------------------------------------------------------------------------
def gpu_quantize_fl32(w: np.ndarray):
    from block_quantized_int8_gb300 import q8
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, s = q8.q8_quantize_rows(dev(w), dev_status=st, mode=q8.Q8_QUANT_FL32)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().view(torch.int16).numpy().view(np.uint16), int(st.item())


def test_fl32_stress_rows_bit_exact(oracle):
    w = synth.quant_stress_rows(32, 4096, 0)
    q_ref, s_ref, fl = oracle.quantize_rows_fl32(w)
    q, s, st = gpu_quantize_fl32(w)
    assert fl == st == 0
    assert np.array_equal(q, q_ref) and np.array_equal(s, s_ref)


@pytest.mark.parametrize("rows,K", [(1, 32), (3, 96), (257, 1536), (1000, 4096)])
def test_fl32_random_bit_exact_and_close_to_exact_mode(oracle, rows, K):
    w = synth.weights(rows, K, 0, f"qf{rows}.{K}")
    q_ref, s_ref, _ = oracle.quantize_rows_fl32(w)
    q, s, st = gpu_quantize_fl32(w)
    assert st == 0
    assert np.array_equal(q, q_ref) and np.array_equal(s, s_ref)
    # same scales as the exact rule, codes at most one apart
    q_e, s_e, _ = oracle.quantize_rows(w)
    assert np.array_equal(s, s_e)
    assert int(np.max(np.abs(q.astype(np.int32) - q_e.astype(np.int32)))) <= 1


def test_fl32_exact_halves_and_flags(oracle):
    g = synth.rng(0, "halves.fl32")
    rows = []
    for e in range(-14, 16):
        for _ in range(4):
            s = np.float32(np.ldexp(1.0 + int(g.integers(0, 1024)) / 1024.0, e))
            if 127.0 * float(s) > 127 * 65504:
                continue
            rows.append(synth.exact_half_block(s, 1.0 if len(rows) % 2 else -1.0, g))
    n = len(rows) // 8 * 8
    w = np.stack(rows[:n]).reshape(-1, 32 * 8).copy()
    w[0, 5] = np.nan
    w[1, 40] = np.float32(127.0 * 65520.0)
    q_ref, s_ref, fl = oracle.quantize_rows_fl32(w)
    q, s, st = gpu_quantize_fl32(w)
    assert np.array_equal(q, q_ref) and np.array_equal(s, s_ref)
    assert st == fl == (oracle.FLAG_NONFINITE | oracle.FLAG_SCALE_OVF)


def test_quantize_mode_argument():
    from block_quantized_int8_gb300 import q8
    w = torch.zeros((1, 32), dtype=torch.float32, device="cuda")
    q = torch.empty((1, 32), dtype=torch.int8, device="cuda")
    s = torch.empty((1, 1), dtype=torch.float16, device="cuda")
    assert q8.lib().q8_quantize_rows_ex(q8._p(w), 1, 32, q8._p(q), q8._p(s), 2, None, None) == q8.Q8_ERR_ARG
