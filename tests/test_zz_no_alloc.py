"""q8_gemm_skinny_noalloc: the skinny matmul for callers that cannot allocate
device memory (fixed memory pools, loops that must not enter the allocator,
hosts that hand over only inputs and outputs).  Its split-K scratch is the
library's built-in device array instead of a caller workspace.

Checked through the C ABI against the oracle (within the matmul tolerance)
and against the existing q8_gemm_skinny entry point, on two calls in a row
(the second call reuses the scratch the first one left behind).  This file
is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from helpers import TOL_ABS, TOL_REL, weights_dev, x_dev

pytestmark = pytest.mark.gpu

# shapes that split K (so the scratch is really used) plus one that does not;
# (1536, 4000, 12) takes the tile kernel with a partial last chunk (K not a
# multiple of 256, M > 8), whose shared row blocks count on tickets in the
# scratch.  (No automatic route reaches the general kernel's split-K any
# more: K off the 256 grid goes to the tiles or the pipeline, and K < 256
# is never split.)
CASES = [(1536, 4096, 4), (1536, 4096, 32), (8192, 1536, 16), (300, 1536, 3), (4097, 1536, 1),
         (1536, 4000, 12)]


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("N,K,M", CASES)
def test_noalloc_matches_oracle_and_q8_gemm_skinny(oracle, N, K, M):
    from block_quantized_int8_gb300 import q8
    L = q8.lib()
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"na{N}.{K}"))
    xn = synth.activations(M, K, 0, f"nax{M}.{K}")
    y_oracle, B = oracle.matmul(qn, sn, xn, threads=8)
    lim = TOL_REL * B + TOL_ABS
    q, s = weights_dev(qn, sn)
    x = x_dev(xn)
    assert q8.q8_workspace_size(N, K, M) <= q8.Q8_NOALLOC_SCRATCH_BYTES
    # the existing entry point, with its own workspace
    y_ws = q8.q8_gemm_skinny(q, s, x)
    torch.cuda.synchronize()
    y_ws = y_ws.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(y_ws - y_oracle) <= lim)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        st = L.q8_gemm_skinny_noalloc(_ptr(q), _ptr(s), N, K, _ptr(x), K, M, _ptr(y), N, _ptr(st_dev), stream)
        assert st == q8.Q8_OK, q8.status_str(st)
        torch.cuda.synchronize()
        assert int(st_dev.item()) == 0
        got = y.cpu().numpy().astype(np.float64)
        err = np.abs(got - y_oracle)
        assert np.all(err <= lim), f"call {call}: max err vs oracle {err.max()}"
        # the same kernels with the same split of K: also within the
        # tolerance of the workspace entry point's result
        assert np.all(np.abs(got - y_ws) <= lim), f"call {call}: differs from q8_gemm_skinny"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    from block_quantized_int8_gb300 import q8
    L = q8.lib()
    N, K, M = 65536, 4096, 32
    assert q8.q8_workspace_size(N, K, M) > q8.Q8_NOALLOC_SCRATCH_BYTES
    a = 1 << 20  # the size check comes before any pointer is touched
    st = L.q8_gemm_skinny_noalloc(a, a, N, K, a, K, M, a, N, None, None)
    assert st == q8.Q8_ERR_WORKSPACE
