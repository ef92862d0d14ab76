"""Bounded waits run out without hanging or faulting the GPU.

Every wait of a woq kernel on another CTA of its grid (split-tile partner words, the
SwiGLU prologue's arrival count, the in-place relayout's grid barriers) gives up after a
bound, records WOQ_DEVERR_TIMEOUT (or fails the relayout) and leaves its outputs alone.
These tests make one CTA skip its arrival (a flag nothing else sets) through
woq_tune_fault, with the bound cut to one millisecond, and check the reported status,
that the affected outputs are untouched, and that zero-filling the workspace restores a
working state.  Nothing traps, faults or waits without a bound.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import to_numpy_u16, to_numpy_u8
from tests.test_gpu_parity import DEV, SENT, Guarded, pack_host, tol_ok

pytestmark = pytest.mark.gpu

woq = None
WAIT_US = 1000


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    global woq
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import weight_only_quantised_gb300 as w
    woq = w
    import tests.test_gpu_parity as tp
    tp.woq = w
    torch.cuda.set_device(0)
    yield
    woq.woq_tune_fault(0, 0, 0)


@pytest.fixture()
def fault():
    def inject(kind, cta):
        woq.woq_tune_fault(kind, cta, WAIT_US)
    yield inject
    woq.woq_tune_fault(0, 0, 0)


def _tiles_untouched_or_right(y, y_ref, S, N):
    """Per 128-row tile: either every output still holds the sentinel, or all are within the
    tolerance.  Returns the number of untouched tiles."""
    untouched = 0
    for t in range((N + 127) // 128):
        cols = slice(128 * t, min(N, 128 * t + 128))
        if (y[:, cols] == np.float32(SENT)).all():
            untouched += 1
        else:
            ok, worst = tol_ok(y[:, cols], y_ref[:, cols], S[:, cols])
            assert ok, f"tile {t}: max err / tolerance = {worst}"
    return untouched


@pytest.mark.parametrize("bits,M", [(4, 1), (6, 2)])
def test_split_tile_partner_that_never_publishes(bits, M, fault):
    """N = 1024, K = 4096: 8 tiles of 32 blocks over 64 CTAs of 4 blocks, so every tile is
    shared by 8 CTAs and combined by the first of them (equal parts: ties go to the lowest
    CTA); CTA 1 publishes its part of tile 0 and is made to skip it."""
    N, K = 1024, 4096
    w, s = synthetic.weights(bits, N, K, seed=40 + bits)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    xn = to_numpy_u16(synthetic.activations(M, K, seed=41, outliers=True))
    y_ref, S = oracle.linear_bf16(bits, wn, sn, N, K, xn)
    wdev = pack_host(bits, wn, sn, N, K)
    x_dev = torch.from_numpy(xn.view(np.int16)).to(DEV).view(torch.bfloat16)
    ws = torch.zeros(woq.woq_workspace_bytes(bits, M, N, K), dtype=torch.uint8, device=DEV)
    lin = woq.woq_w4a8_linear_bf16 if bits == 4 else woq.woq_w6a8_linear_bf16
    assert woq.woq_plan_launch(bits, M, N, K, woq.PLAN_BF16)["ctas"] == 64

    fault(1, 1)
    out = Guarded(M, N)
    lin(wdev, x_dev, N, K, out.y, ws)
    torch.cuda.synchronize()
    out.check_guards()
    assert woq.woq_read_status(ws, clear=True) & woq.WOQ_DEVERR_TIMEOUT
    y = out.numpy()
    assert _tiles_untouched_or_right(y, y_ref, S, N) >= 1
    assert (y[:, :128] == np.float32(SENT)).all()  # the combined tile the missing part belongs to

    # without the fault, after the workspace is zero-filled again: the whole result
    woq.woq_tune_fault(0, 0, 0)
    woq.woq_workspace_init(ws)
    out = Guarded(M, N)
    lin(wdev, x_dev, N, K, out.y, ws)
    torch.cuda.synchronize()
    assert woq.woq_read_status(ws) == 0
    ok, worst = tol_ok(out.numpy(), y_ref, S)
    assert ok, f"max err / tolerance = {worst}"
    assert not ws.cpu().numpy()[4:].any()  # every partial word consumed and cleared


def test_swiglu_arrival_that_never_comes(fault):
    """The SwiGLU prologue counts every CTA in before the row maxima are read: one CTA that
    never counts itself in makes every CTA give up, and y stays as it was."""
    bits, M, N, K = 4, 2, 2048, 4096
    w, s = synthetic.weights(bits, N, K, seed=50)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    gu = synthetic.gate_up_output(M, K, 51).numpy().copy()
    y_ref, S = oracle.linear_swiglu(bits, wn, sn, N, K, gu)
    wdev = pack_host(bits, wn, sn, N, K)
    gu_dev = torch.from_numpy(gu).to(DEV)
    ws = torch.zeros(woq.woq_workspace_bytes(bits, M, N, K), dtype=torch.uint8, device=DEV)

    fault(2, 3)
    out = Guarded(M, N)
    woq.woq_w4a8_linear_swiglu_f32(wdev, gu_dev, N, K, out.y, ws)
    torch.cuda.synchronize()
    out.check_guards()
    assert woq.woq_read_status(ws, clear=True) & woq.WOQ_DEVERR_TIMEOUT
    assert (out.numpy() == np.float32(SENT)).all()

    woq.woq_tune_fault(0, 0, 0)
    woq.woq_workspace_init(ws)
    for _ in range(2):  # and the launch after that one (its words were left zero)
        out = Guarded(M, N)
        woq.woq_w4a8_linear_swiglu_f32(wdev, gu_dev, N, K, out.y, ws)
        torch.cuda.synchronize()
        assert woq.woq_read_status(ws) == 0
        ok, worst = tol_ok(out.numpy(), y_ref, S)
        assert ok, f"max err / tolerance = {worst}"


def test_relayout_barrier_arrival_that_never_comes(fault):
    """One CTA of the cooperative relayout leaves before the first grid barrier: the others
    give up, the header is never written and the call returns WOQ_ERR_DEVICE; the next
    relayout of the same buffer (refilled) succeeds."""
    bits, N, K = 4, 4096, 1280
    w, s = synthetic.weights(bits, N, K, seed=60)
    host = woq.woq_pack_w4(to_numpy_u8(w), to_numpy_u16(s), N, K)
    buf = torch.full((woq.woq_packed_bytes(bits, N, K),), 0xA5, dtype=torch.uint8, device=DEV)
    woq.canonical_into_buffer(bits, w.to(DEV), s.to(DEV).view(torch.int16), buf)
    fault(3, 5)
    with pytest.raises(woq.WoqError) as e:
        woq.woq_relayout_inplace(bits, buf, N, K)
    assert e.value.status == woq.WOQ_ERR_DEVICE

    woq.woq_tune_fault(0, 0, 0)
    woq.canonical_into_buffer(bits, w.to(DEV), s.to(DEV).view(torch.int16), buf)
    woq.woq_relayout_inplace(bits, buf, N, K)
    torch.cuda.synchronize()
    assert np.array_equal(buf.cpu().numpy(), host)


def test_fault_knob_rejects_bad_values():
    for args in [(-1, 0, 0), (4, 0, 0), (1, -1, 0), (1, 0, -1), (1, 0, 2000001)]:
        with pytest.raises(woq.WoqError) as e:
            woq.woq_tune_fault(*args)
        assert e.value.status == woq.WOQ_ERR_SHAPE
