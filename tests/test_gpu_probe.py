"""The streaming-read probe reads every byte it is given (its XOR fold
equals the host's) and rejects misaligned arguments."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [16, 4096, 1 << 20, (64 << 20) + 48])
def test_stream_read_folds_every_word(nbytes):
    from block_quantized_int8_gb300 import q8
    rng = np.random.default_rng(nbytes)
    host = rng.integers(0, 2**32, size=nbytes // 4, dtype=np.uint32)
    buf = torch.from_numpy(host.view(np.int32)).cuda()
    out = torch.zeros(int(q8.lib().q8_stream_read_out_words()), dtype=torch.int32, device="cuda")
    assert q8.lib().q8_stream_read(buf.data_ptr(), nbytes, out.data_ptr(), None) == q8.Q8_OK
    torch.cuda.synchronize()
    got = np.bitwise_xor.reduce(out.cpu().numpy().view(np.uint32))
    assert int(got) == int(np.bitwise_xor.reduce(host))
    assert q8.lib().q8_stream_read(buf.data_ptr() + 4, 16, out.data_ptr(), None) == q8.Q8_ERR_ALIGN
    assert q8.lib().q8_stream_read(buf.data_ptr(), 8, out.data_ptr(), None) == q8.Q8_ERR_ALIGN
