"""q8_linear_chain: a dependent chain of skinny matmuls whose inputs are made
on the device (RMS normalisation, after SwiGLU between gate+up and down).
Each step is checked against the oracle on the GPU's own input of that step:
y_i within the matmul tolerance of oracle.matmul(W_i, x_i), and x_{i+1}
against oracle.chain_next(y_i) to one bf16 unit in the last place (the
device works in binary32, the oracle in binary64, and each rounds once to
bf16).  The layer follows the decoder's matrix order (QKV, o_proj,
gate+up, down)."""
import numpy as np
import pytest
import torch

import synth
from helpers import check_tol, weights_dev, x_dev

pytestmark = pytest.mark.gpu

# (name, K, N, how the next input is made from this output)
LAYER = [("qkv", 1536, 4608, 1), ("o_proj", 1536, 1536, 1), ("gate_up", 1536, 8192, 2), ("down", 4096, 1536, 1)]


def bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp_diff(a, b):
    """|a - b| in bf16 units in the last place (sign-magnitude ordering)."""
    def key(v):
        v = np.asarray(v, dtype=np.int64)
        return np.where(v & 0x8000, -(v & 0x7FFF), v & 0x7FFF)
    return np.abs(key(a) - key(b))


def build_chain(oracle, M, layers, tag, ends=True):
    """Host weights and device buffers of `layers` decoder layers; returns
    (host steps [(q, s)], device step tuples for make_chain)."""
    from block_quantized_int8_gb300 import q8
    host, dev_steps = [], []
    x0 = synth.activations(M, LAYER[0][1], 0, f"{tag}.x0")
    nsteps = layers * len(LAYER)
    for i in range(nsteps):
        name, K, N, nxt = LAYER[i % len(LAYER)]
        qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"{tag}.{i // len(LAYER)}.{name}"))
        host.append((qn, sn))
        q, s = weights_dev(qn, sn)
        x = x_dev(x0) if i == 0 else torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        if ends and i == nsteps - 1:
            nxt = q8.Q8_CHAIN_END
        dev_steps.append((q, s, x, y, nxt))
    return host, dev_steps


@pytest.mark.parametrize("M", [1, 3, 8, 16, 32])
def test_chain_steps_against_oracle(oracle, M):
    from block_quantized_int8_gb300 import q8
    host, dev_steps = build_chain(oracle, M, 2, f"ch{M}")
    steps, m = q8.make_chain(dev_steps)
    assert m == M
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q8.q8_linear_chain(steps, M, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    exact = total = 0
    for i, ((qn, sn), (q, s, x, y, nxt)) in enumerate(zip(host, dev_steps)):
        xb = x.view(torch.int16).cpu().numpy().view(np.uint16)
        yg = y.cpu().numpy()
        y_ref, B = oracle.matmul(qn, sn, xb, threads=8)
        check_tol(yg, y_ref, B, f"chain step {i} ({LAYER[i % 4][0]}) M={M}")
        if i + 1 < len(dev_steps):
            xn = dev_steps[i + 1][2].view(torch.int16).cpu().numpy().view(np.uint16)
            want = oracle.chain_next(yg, xn.shape[1], swiglu=(nxt == q8.Q8_CHAIN_SWIGLU_RMSNORM))
            d = ulp_diff(xn, want)
            assert d.max() <= 1, f"step {i} -> {i + 1}: x off by {int(d.max())} bf16 ulps"
            exact += int((d == 0).sum())
            total += d.size
    # rounding the binary32 value and the binary64 value differ only next to a tie
    assert exact >= 0.99 * total, f"{exact} of {total} next inputs exact"


def test_chain_graph_replay_is_bitwise_stable(oracle):
    """The chain captured in a CUDA graph replays to the bits of an eager run
    (fixed-order sums everywhere; the workspace's counters left at zero)."""
    from block_quantized_int8_gb300 import q8
    M = 1
    _, dev_steps = build_chain(oracle, M, 2, "chg")
    steps, _ = q8.make_chain(dev_steps)
    ws = q8.workspace(q8.q8_linear_chain_workspace_size(steps, M))
    q8.q8_linear_chain(steps, M, ws=ws)
    torch.cuda.synchronize()
    eager = [t[3].clone() for t in dev_steps]
    for t in dev_steps:
        t[3].fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            q8.q8_linear_chain(steps, M, ws=ws, stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, t in zip(eager, dev_steps):
        assert torch.equal(a.view(torch.int32), t[3].view(torch.int32))


def test_chain_one_step_equals_linear_batch(oracle):
    """A one-step chain is one matmul: the same bits as q8_linear_batch."""
    from block_quantized_int8_gb300 import q8
    for M in (1, 5, 20):
        host, dev_steps = build_chain(oracle, M, 1, f"ch1.{M}")
        q, s, x, y, _ = dev_steps[0]
        steps, _ = q8.make_chain([(q, s, x, y, q8.Q8_CHAIN_END)])
        q8.q8_linear_chain(steps, M)
        y2 = torch.empty_like(y)
        q8.q8_linear_batch([(q, s, x, y2)])
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int32), y2.view(torch.int32))


@pytest.mark.parametrize("M", [1, 8, 12, 32])
def test_chain_off_the_256_grid(oracle, M):
    """A chain whose K are not multiples of 256 (2080 and 4128, so the tile
    kernel's partial last chunk, the pipeline or the GEMV serve the steps),
    with a shape repeated later in the chain (the steps of one shape share a
    workspace region).  Each step against the oracle on its own input."""
    from block_quantized_int8_gb300 import q8
    plan = [(2080, 4608, q8.Q8_CHAIN_RMSNORM), (2080, 8256, q8.Q8_CHAIN_SWIGLU_RMSNORM),
            (4128, 2080, q8.Q8_CHAIN_RMSNORM), (2080, 4608, q8.Q8_CHAIN_RMSNORM),
            (2080, 2080, q8.Q8_CHAIN_END)]
    host, dev_steps = [], []
    for i, (K, N, nxt) in enumerate(plan):
        qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"cho{i}"))
        host.append((qn, sn))
        q, s = weights_dev(qn, sn)
        x = x_dev(synth.activations(M, K, 0, f"chox{M}")) if i == 0 else \
            torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        dev_steps.append((q, s, x, y, nxt))
    steps, _ = q8.make_chain(dev_steps)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q8.q8_linear_chain(steps, M, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for i, ((qn, sn), (q, s, x, y, nxt)) in enumerate(zip(host, dev_steps)):
        xb = x.view(torch.int16).cpu().numpy().view(np.uint16)
        yg = y.cpu().numpy()
        y_ref, B = oracle.matmul(qn, sn, xb, threads=8)
        check_tol(yg, y_ref, B, f"odd-K chain step {i} M={M}")
        if i + 1 < len(dev_steps):
            xn = dev_steps[i + 1][2].view(torch.int16).cpu().numpy().view(np.uint16)
            want = oracle.chain_next(yg, xn.shape[1], swiglu=(nxt == q8.Q8_CHAIN_SWIGLU_RMSNORM))
            assert ulp_diff(xn, want).max() <= 1, f"odd-K chain step {i} -> {i + 1}"


@pytest.mark.parametrize("M", [1, 4])
def test_chain_normalisation_widths(oracle, M):
    """Next inputs of 512 values (one per thread of the register kernel) and
    of 12800 (beyond its 8192: the strided kernel), against the oracle."""
    from block_quantized_int8_gb300 import q8
    plan = [(1536, 512, q8.Q8_CHAIN_RMSNORM), (512, 12800, q8.Q8_CHAIN_RMSNORM), (12800, 1536, q8.Q8_CHAIN_END)]
    host, dev_steps = [], []
    for i, (K, N, nxt) in enumerate(plan):
        qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"chw{i}"))
        host.append((qn, sn))
        q, s = weights_dev(qn, sn)
        x = x_dev(synth.activations(M, K, 0, f"chwx{M}")) if i == 0 else \
            torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        dev_steps.append((q, s, x, y, nxt))
    steps, _ = q8.make_chain(dev_steps)
    q8.q8_linear_chain(steps, M)
    torch.cuda.synchronize()
    for i, ((qn, sn), (q, s, x, y, nxt)) in enumerate(zip(host, dev_steps)):
        xb = x.view(torch.int16).cpu().numpy().view(np.uint16)
        yg = y.cpu().numpy()
        y_ref, B = oracle.matmul(qn, sn, xb, threads=8)
        check_tol(yg, y_ref, B, f"width chain step {i} M={M}")
        if i + 1 < len(dev_steps):
            xn = dev_steps[i + 1][2].view(torch.int16).cpu().numpy().view(np.uint16)
            want = oracle.chain_next(yg, xn.shape[1], swiglu=False)
            assert ulp_diff(xn, want).max() <= 1, f"width chain step {i} -> {i + 1}"
