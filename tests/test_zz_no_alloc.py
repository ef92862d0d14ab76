"""The allocation-free linear (woq_w4a8_linear_bf16_noalloc) against the regular one.

For callers that cannot allocate device memory (a host application that owns every
allocation, a loop with a fixed memory budget), the library offers a variant of the
int4 bf16 linear that uses its own built-in scratch instead of a caller workspace, and
woq_noalloc_read_status to read the device-side error bits kept in that scratch.
This file is collected last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import to_numpy_u16, to_numpy_u8

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SCRATCH_BYTES = 2 << 20  # the built-in scratch array
SENT = -7.0


def _woq():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import weight_only_quantised_gb300 as woq
    torch.cuda.set_device(0)
    return woq


def _noalloc(woq, wdev, x_dev, M, N, K, y):
    """One call through the C ABI on the current stream; returns the status."""
    return woq.lib.woq_w4a8_linear_bf16_noalloc(wdev.data_ptr(), wdev.numel(), x_dev.data_ptr(), M, N, K,
                                                y.data_ptr(), torch.cuda.current_stream().cuda_stream)


# M = 1 .. 4 run the dp4a consumer, 5 and 6 the tensor-core consumer; every one of these
# grids splits tiles across CTAs, so the scratch's split-tile words are used
@pytest.mark.parametrize("M", [1, 2, 4, 5, 6])
def test_noalloc_linear_matches_regular_entry_twice(M):
    woq = _woq()
    N, K = 4096, 4096
    w, s = synthetic.weights(4, N, K, seed=77 + M)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    x = synthetic.activations(M, K, seed=78 + M)
    xn = to_numpy_u16(x)
    _, S = oracle.linear_bf16(4, wn, sn, N, K, xn)
    bound = oracle.tolerance(S)
    wdev = torch.from_numpy(woq.woq_pack_w4(wn, sn, N, K)).to(DEV)
    x_dev = x.to(DEV)
    woq.woq_noalloc_read_status(clear=True)

    # the existing entry point, with its own zero-filled workspace
    ws = torch.zeros(woq.woq_workspace_bytes(4, M, N, K), dtype=torch.uint8, device=DEV)
    y_ref = torch.empty((M, N), dtype=torch.float32, device=DEV)
    woq.woq_w4a8_linear_bf16(wdev, x_dev, N, K, y_ref, ws)
    torch.cuda.synchronize()
    yr = y_ref.cpu().numpy().astype(np.float64)

    # two calls in a row through the C ABI, each into a fresh output
    for _ in range(2):
        y = torch.full((M, N), SENT, dtype=torch.float32, device=DEV)
        status = _noalloc(woq, wdev, x_dev, M, N, K, y)
        assert status == woq.WOQ_OK, woq.lib.woq_status_string(status)
        torch.cuda.synchronize()
        err = np.abs(y.cpu().numpy().astype(np.float64) - yr)
        assert (err <= bound).all(), f"max err / tolerance = {float((err / bound).max())}"
        assert woq.woq_noalloc_read_status() == 0


def test_noalloc_refuses_a_launch_larger_than_its_scratch():
    """A grid whose split-tile words exceed the 2 MiB array is refused before anything is
    enqueued (M = 8 needs 2048 * 8 bytes per CTA: too much for one CTA per SM here)."""
    woq = _woq()
    M, N, K = 8, 7168, 5120
    ctas = woq.woq_plan_launch(4, M, N, K, woq.PLAN_BF16)["ctas"]
    need = 256 + 2048 * M * ctas
    wdev = torch.zeros(woq.woq_packed_bytes(4, N, K), dtype=torch.uint8, device=DEV)
    x_dev = torch.zeros((M, K), dtype=torch.bfloat16, device=DEV)
    y = torch.full((M, N), SENT, dtype=torch.float32, device=DEV)
    status = _noalloc(woq, wdev, x_dev, M, N, K, y)
    torch.cuda.synchronize()
    if need > SCRATCH_BYTES:
        assert status == woq.WOQ_ERR_WORKSPACE
        assert (y.cpu().numpy() == np.float32(SENT)).all()
    else:  # a GPU with few SMs: the launch fits (the zero header is then refused on the device)
        assert status == woq.WOQ_OK
        assert woq.woq_noalloc_read_status(clear=True) & woq.WOQ_DEVERR_HEADER


def test_noalloc_reports_a_header_mismatch_and_recovers():
    """A packed buffer whose header does not match (bits, N, K): the call returns WOQ_OK (the
    check runs on the device), woq_noalloc_read_status reports WOQ_DEVERR_HEADER and y keeps
    its contents; after the clear, a correct call matches the regular entry again."""
    woq = _woq()
    M, N, K = 2, 1024, 2048
    w, s = synthetic.weights(4, N, K, seed=91)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    packed = woq.woq_pack_w4(wn, sn, N, K)
    bad = packed.copy()
    bad[8] = 6  # the header claims int6
    x_dev = synthetic.activations(M, K, seed=92).to(DEV)
    woq.woq_noalloc_read_status(clear=True)

    y = torch.full((M, N), SENT, dtype=torch.float32, device=DEV)
    assert _noalloc(woq, torch.from_numpy(bad).to(DEV), x_dev, M, N, K, y) == woq.WOQ_OK
    torch.cuda.synchronize()
    assert woq.woq_noalloc_read_status(clear=True) & woq.WOQ_DEVERR_HEADER
    assert woq.woq_noalloc_read_status() == 0
    assert (y.cpu().numpy() == np.float32(SENT)).all()

    wdev = torch.from_numpy(packed).to(DEV)
    ws = torch.zeros(woq.woq_workspace_bytes(4, M, N, K), dtype=torch.uint8, device=DEV)
    y_ref = torch.empty((M, N), dtype=torch.float32, device=DEV)
    woq.woq_w4a8_linear_bf16(wdev, x_dev, N, K, y_ref, ws)
    assert _noalloc(woq, wdev, x_dev, M, N, K, y) == woq.WOQ_OK
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ref.cpu().numpy().view(np.uint32))
    assert woq.woq_noalloc_read_status() == 0


def test_noalloc_rejects_oversized_and_bad_arguments():
    woq = _woq()
    L = woq.lib
    assert L.woq_w4a8_linear_bf16_noalloc(None, 0, None, 9, 128, 128, None, None) == woq.WOQ_ERR_SHAPE
    assert L.woq_w4a8_linear_bf16_noalloc(None, 0, None, 0, 128, 128, None, None) == woq.WOQ_OK
    y = torch.empty(16, device=DEV)
    assert L.woq_w4a8_linear_bf16_noalloc(None, 0, ctypes.c_void_p(0x10000), 1, 128, 128, y.data_ptr(),
                                          None) == woq.WOQ_ERR_NULL
    assert L.woq_noalloc_read_status(0, None, None) == woq.WOQ_ERR_NULL
