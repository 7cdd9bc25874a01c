"""The kernels' failure path, exercised without a fault: a bounded mbarrier
wait that nothing completes gives up after its limit, reports
Q8_DEV_TIMEOUT through the status word, and the context stays usable."""
import numpy as np
import pytest
import torch

import synth
from helpers import check_tol, weights_dev, x_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ms", [1, 5])
def test_bounded_wait_reports_timeout_and_context_survives(oracle, limit_ms):
    from block_quantized_int8_gb300 import q8
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    el = torch.zeros(1, dtype=torch.int64, device="cuda")
    assert q8.lib().q8_selftest_wait_timeout(limit_ms * 1_000_000, q8._p(st), q8._p(el), None) == q8.Q8_OK
    torch.cuda.synchronize()
    assert int(st.item()) & q8.Q8_DEV_TIMEOUT
    waited = int(el.item())
    assert limit_ms * 1_000_000 <= waited < limit_ms * 1_000_000 + 50_000_000
    # the context still runs a matmul correctly
    qn, sn, _ = oracle.quantize_rows(synth.weights(256, 1536, 0, "fail.w"))
    q, s = weights_dev(qn, sn)
    xn = synth.activations(1, 1536, 0, "fail.x")
    y = torch.empty((1, 256), dtype=torch.float32, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    q8.q8_linear_batch([(q, s, x_dev(xn), y)], dev_status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    y_ref, B = oracle.matmul(qn, sn, xn)
    check_tol(y.cpu().numpy(), y_ref, B, "after a timed-out wait")
