"""The in-run read reference (pa_stream_read): every byte is read, checked through the XOR of
all 32-bit words against numpy's, on sizes that exercise the unrolled loop and its tail."""
import numpy as np
import pytest
import torch

from paged_kv_cache_299_gb300 import binding as pa

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [0, 16, 4096 + 48, (3 << 20) + 16 * 7, 64 << 20])
def test_stream_read_xor_matches(nbytes):
    rng = np.random.default_rng(nbytes)
    host = rng.integers(0, 2**32, size=nbytes // 4, dtype=np.uint32)
    buf = torch.from_numpy(host.view(np.int32)).cuda()
    x = torch.full((1,), 12345, dtype=torch.int32, device="cuda")  # XOR accumulates into x
    pa.pa_stream_read(buf, x)
    want = (np.bitwise_xor.reduce(host) if host.size else np.uint32(0)) ^ np.uint32(12345)
    assert int(x.cpu().numpy().view(np.uint32)[0]) == int(want)
