"""Failure detection on the GPU without a fault: a bounded in-kernel wait that
nothing completes expires, is counted in the device counter the host reads,
and the context and stream stay usable for the next launches."""
import numpy as np
import pytest
import torch

import oracle
from paged_sparse_kv_gb300 import ops, synthetic

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_and_is_counted(cuda_device):
    torch.cuda.synchronize(cuda_device)
    before = ops.device_wait_timeouts()
    ops.device_wait_selftest(2_000_000, cuda_device)  # 2 ms
    torch.cuda.synchronize(cuda_device)
    assert ops.device_wait_timeouts() == before + 1
    # the context still runs kernels: a gather after the expiry is exact
    rng = np.random.default_rng(5)
    bs, pages, D = 16, 6, 128
    rec = oracle.fp8_record_bytes(D, 0, True)
    geom = synthetic.CacheGeom(pages, bs, (bs * rec + 15) // 16 * 16)
    host = synthetic.random_cache_bytes(9, geom)
    idx = rng.integers(-1, pages * bs, size=(7, 9)).astype(np.int32)
    out = torch.empty((7, 9, D), dtype=torch.bfloat16, device=cuda_device)
    ops.dequantize_and_gather_k_cache(out, torch.from_numpy(host).to(cuda_device),
                                      torch.from_numpy(idx).to(cuda_device), bs, rope_dim=0)
    want = oracle.dequantize_and_gather_k_cache(host, bs, 0, D, 0, idx)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want)
    torch.cuda.synchronize(cuda_device)
    assert ops.device_wait_timeouts() == before + 1  # the gather's waits all completed
