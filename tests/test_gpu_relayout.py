"""GPU tests of the in-place relayout (woq_relayout_inplace).

"Doubling LLM token rates in ComfyUI", section "Optimizing the Linear Kernel": the
weights are re-laid out for the kernel in place in VRAM, with no extra memory.  The
buffer starts with the canonical weights and scales at byte 256 and must end up
byte-identical to the host packer's output; the packed buffer must also unpack back to
the canonical inputs and drive the linear to the oracle's result.  Shapes cover ragged
N (a partial last tile), one block, and matrices large enough that the relayout runs in
several batches of tiles (the 27B gate+up and LM head).  Scratch bytes (the header slot
and the slack after the scales) start as garbage.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import to_numpy_u16, to_numpy_u8

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
woq = None


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    global woq
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import weight_only_quantised_gb300 as w
    woq = w
    torch.cuda.set_device(0)
    yield


def _host_pack(bits, wn, sn, N, K):
    return woq.woq_pack_w4(wn, sn, N, K) if bits == 4 else woq.woq_pack_w6(wn, sn, N, K)


def _relaid(bits, w, s, N, K, fill=0xA5):
    buf = torch.full((woq.woq_packed_bytes(bits, N, K),), fill, dtype=torch.uint8, device=DEV)
    woq.canonical_into_buffer(bits, w.to(DEV), s.to(DEV).view(torch.int16), buf)
    woq.woq_relayout_inplace(bits, buf, N, K)
    return buf


@pytest.mark.parametrize("bits", [4, 6])
@pytest.mark.parametrize("N,K", [(1, 128), (127, 256), (129, 384), (1000, 512), (4096, 1280), (7168, 5120)])
def test_relayout_matches_host_pack(bits, N, K):
    w, s = synthetic.weights(bits, N, K, seed=N * 3 + K)
    host = _host_pack(bits, to_numpy_u8(w), to_numpy_u16(s), N, K)
    buf = _relaid(bits, w, s, N, K)
    torch.cuda.synchronize()
    assert np.array_equal(buf.cpu().numpy(), host)


@pytest.mark.parametrize("bits,N,K", [(4, 34816, 5120), (6, 34816, 5120), (4, 5120, 17408), (4, 152064, 5120)])
def test_relayout_in_several_batches(bits, N, K):
    """Large matrices: the tiles move in several batches; the result equals the device packer's."""
    w, s = synthetic.weights(bits, N, K, seed=5, device=DEV)
    ref = torch.empty((woq.woq_packed_bytes(bits, N, K),), dtype=torch.uint8, device=DEV)
    woq.woq_pack_device(bits, w, s.view(torch.int16), N, K, ref)
    buf = _relaid(bits, w, s, N, K, fill=0x3C)
    torch.cuda.synchronize()
    assert torch.equal(buf, ref)


@pytest.mark.parametrize("bits", [4, 6])
def test_relayout_round_trip_and_linear(bits):
    """The relaid buffer unpacks to the canonical inputs and the linear on it meets the oracle."""
    N, K, M = 1500, 1024, 2
    w, s = synthetic.weights(bits, N, K, seed=77)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    buf = _relaid(bits, w, s, N, K)
    q_back, s_back = woq.woq_unpack(bits, buf.cpu().numpy(), N, K)
    assert np.array_equal(q_back, wn) and np.array_equal(s_back, sn)
    x = synthetic.activations(M, K, seed=78)
    xn = to_numpy_u16(x)
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    ws = torch.zeros((woq.woq_workspace_bytes(bits, M, N, K),), dtype=torch.uint8, device=DEV)
    fn = woq.woq_w4a8_linear_bf16 if bits == 4 else woq.woq_w6a8_linear_bf16
    fn(buf, x.to(DEV), N, K, y, ws)
    torch.cuda.synchronize()
    y_ref, S = oracle.linear_bf16(bits, wn, sn, N, K, xn)
    err = np.abs(y.cpu().numpy().astype(np.float64) - y_ref)
    assert (err <= oracle.tolerance(S)).all()


def test_relayout_empty_writes_header_only():
    for bits, N, K in [(4, 0, 256), (6, 5, 0)]:
        buf = torch.full((woq.woq_packed_bytes(bits, N, K),), 0x11, dtype=torch.uint8, device=DEV)
        woq.woq_relayout_inplace(bits, buf, N, K)
        host = _host_pack(bits, np.zeros((N, synthetic.canonical_row_bytes(bits, K)), np.uint8),
                          np.zeros((N, K // 128), np.uint16), N, K)
        assert np.array_equal(buf.cpu().numpy(), host)


def test_relayout_rejects_bad_arguments():
    N, K = 256, 256
    need = woq.woq_packed_bytes(4, N, K)
    buf = torch.zeros((need + 64,), dtype=torch.uint8, device=DEV)
    lib = woq.lib
    assert lib.woq_relayout_inplace(4, None, need, N, K, None) == woq.WOQ_ERR_NULL
    assert lib.woq_relayout_inplace(4, buf.data_ptr() + 8, need, N, K, None) == woq.WOQ_ERR_ALIGN
    assert lib.woq_relayout_inplace(4, buf.data_ptr(), need - 1, N, K, None) == woq.WOQ_ERR_LAYOUT
    assert lib.woq_relayout_inplace(5, buf.data_ptr(), need, N, K, None) == woq.WOQ_ERR_SHAPE
    assert lib.woq_relayout_inplace(4, buf.data_ptr(), need, N, 100, None) == woq.WOQ_ERR_SHAPE
    # more group scales than shared memory can stage: refused before the buffer is touched
    Nb, Kb = 300000, 8192
    big = torch.zeros((woq.woq_packed_bytes(4, Nb, Kb),), dtype=torch.uint8, device=DEV)
    assert lib.woq_relayout_inplace(4, big.data_ptr(), big.numel(), Nb, Kb, None) == woq.WOQ_ERR_SHAPE
    assert int(big[:4096].count_nonzero()) == 0
