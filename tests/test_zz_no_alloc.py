"""The allocation-free linear (woq_w4a8_linear_bf16_noalloc) against the regular one.

For callers that cannot allocate device memory (a host application that owns every
allocation, a loop with a fixed memory budget), the library offers a variant of the
int4 bf16 linear that uses its own built-in scratch instead of a caller workspace.
This file is collected last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import to_numpy_u16, to_numpy_u8

pytestmark = pytest.mark.gpu


def test_noalloc_linear_matches_regular_entry_twice():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import weight_only_quantised_gb300 as woq
    dev = "cuda:0"
    torch.cuda.set_device(0)
    M, N, K = 2, 4096, 4096  # several tiles split across CTAs, so the scratch is used
    w, s = synthetic.weights(4, N, K, seed=77)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    x = synthetic.activations(M, K, seed=78)
    xn = to_numpy_u16(x)
    _, S = oracle.linear_bf16(4, wn, sn, N, K, xn)
    bound = oracle.tolerance(S)
    wdev = torch.from_numpy(woq.woq_pack_w4(wn, sn, N, K)).to(dev)
    x_dev = x.to(dev)

    # the existing entry point, with its own zero-filled workspace
    ws = torch.zeros(woq.woq_workspace_bytes(4, M, N, K), dtype=torch.uint8, device=dev)
    y_ref = torch.empty((M, N), dtype=torch.float32, device=dev)
    woq.woq_w4a8_linear_bf16(wdev, x_dev, N, K, y_ref, ws)
    torch.cuda.synchronize()
    yr = y_ref.cpu().numpy().astype(np.float64)

    # two calls in a row through the C ABI, each into a fresh output
    for _ in range(2):
        y = torch.full((M, N), -7.0, dtype=torch.float32, device=dev)
        status = woq.lib.woq_w4a8_linear_bf16_noalloc(wdev.data_ptr(), wdev.numel(), x_dev.data_ptr(), M, N, K,
                                                      y.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert status == woq.WOQ_OK, woq.lib.woq_status_string(status)
        torch.cuda.synchronize()
        err = np.abs(y.cpu().numpy().astype(np.float64) - yr)
        assert (err <= bound).all(), f"max err / tolerance = {float((err / bound).max())}"


def test_noalloc_rejects_oversized_and_bad_arguments():
    import ctypes
    import weight_only_quantised_gb300 as woq
    L = woq.lib
    assert L.woq_w4a8_linear_bf16_noalloc(None, 0, None, 9, 128, 128, None, None) == woq.WOQ_ERR_SHAPE
    assert L.woq_w4a8_linear_bf16_noalloc(None, 0, None, 0, 128, 128, None, None) == woq.WOQ_OK
    y = torch.empty(16, device="cuda:0")
    assert L.woq_w4a8_linear_bf16_noalloc(None, 0, ctypes.c_void_p(0x10000), 1, 128, 128, y.data_ptr(),
                                          None) == woq.WOQ_ERR_NULL
