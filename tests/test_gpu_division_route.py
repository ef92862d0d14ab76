"""Rows too small for the division-free quantiser take the IEEE division route in every
prologue of the fused linears.

The kernels' codes come from a corrected quotient of x and the reciprocal of the row scale
when that scale is at least 2^-123 (largest |x| at least 2^-116), and from the IEEE division
x / s otherwise ("Optimizing the Linear Kernel": the activations are quantised to int8 per
row inside the linear's own launch).  Rows scaled by 2^-124 are below that bound.  They are
sent through the plain bf16 entry (rows read into registers and rows quantised in rounds),
the RMSNorm entry (a gamma scaled by 2^-126 makes h that small) and the SwiGLU entry (an up
half scaled by 2^-128); each fused linear must be bit-identical to its twin followed by the
int8 GEMV, the twins' q bytes and scales must equal the oracle's, and y must be within the
GEMV tolerance of the oracle.  A normal row rides along in every launch.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import to_numpy_u16, to_numpy_u8
from tests.test_gpu_parity import DEV, Guarded, Workspace, pack_host, tol_ok

pytestmark = pytest.mark.gpu

woq = None
TINY_X, TINY_G, TINY_U = 2.0 ** -124, 2.0 ** -126, 2.0 ** -128


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
    woq.woq_tune_path(0)


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return to_numpy_u16(t.to(torch.bfloat16))


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def _gemv(bits, wdev, q, a, N, K, M):
    out, ws = Guarded(M, N), Workspace(bits, M, N, K)
    (woq.woq_w4a8_gemv if bits == 4 else woq.woq_w6a8_gemv)(wdev, q, a, N, K, out.y, ws.ws)
    torch.cuda.synchronize()
    out.check_guards()
    ws.check()
    return out.numpy()


def _weights(bits, N, K, seed):
    w, s = synthetic.weights(bits, N, K, seed=seed)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    return wn, sn, pack_host(bits, wn, sn, N, K)


def _tiny_rows(M, K, seed):
    """bf16 bits [M, K]: even rows scaled by 2^-124 (largest |x| below 2^-116), odd rows as drawn."""
    x = synthetic.activations(M, K, seed=seed, outliers=True).float()
    x[0::2] *= TINY_X
    xn = _bf16_bits(x)
    amax = np.abs((xn.astype(np.uint32) << 16).view(np.float32)).max(axis=1)
    assert (amax[0::2] < 2.0 ** -116).all() and (amax[0::2] > 0).all()
    return xn


@pytest.mark.parametrize("bits,path", [(4, 1), (4, 2), (6, 1)])
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("K", [1024, 17408])
def test_fused_bf16_linear_on_tiny_rows(bits, path, M, K):
    """K = 1024 keeps every row in registers; 17408 quantises in rounds from M = 2 on."""
    if K > woq.woq_max_k(bits, M, True):
        pytest.skip("beyond the fused entry's shared-memory limit for these rows")
    woq.woq_tune_path(path)
    N = 384
    wn, sn, wdev = _weights(bits, N, K, seed=11 * M + K + bits)
    xn = _tiny_rows(M, K, seed=5 * M + K)
    q_ref, s_ref = oracle.act_quant(xn)
    y_ref, S = oracle.linear_bf16(bits, wn, sn, N, K, xn)
    out, ws = Guarded(M, N), Workspace(bits, M, N, K)
    (woq.woq_w4a8_linear_bf16 if bits == 4 else woq.woq_w6a8_linear_bf16)(wdev, _dev_bf16(xn), N, K, out.y, ws.ws)
    torch.cuda.synchronize()
    out.check_guards()
    ws.check()
    y = out.numpy()
    ok, worst = tol_ok(y, y_ref, S)
    assert ok, f"max err / tolerance = {worst}"
    q = torch.from_numpy(q_ref).to(DEV)
    a = torch.from_numpy(s_ref).to(DEV)
    assert np.array_equal(y.view(np.uint32), _gemv(bits, wdev, q, a, N, K, M).view(np.uint32))


@pytest.mark.parametrize("bits,path", [(4, 1), (4, 2), (6, 1)])
@pytest.mark.parametrize("M", [1, 3, 4])
@pytest.mark.parametrize("K", [1024, 5120])
def test_fused_rmsnorm_linear_on_a_tiny_gamma(bits, path, M, K):
    if K > woq.woq_max_k(bits, M, True):
        pytest.skip("beyond the fused entry's shared-memory limit for these rows")
    woq.woq_tune_path(path)
    N = 384
    wn, sn, wdev = _weights(bits, N, K, seed=13 * M + K + bits)
    xn = _bf16_bits(synthetic.activations(M, K, seed=7 * M + K, outliers=True).float())
    g = _bf16_bits(synthetic.rmsnorm_weight(K, K + M).float() * TINY_G)
    eps = 1e-6
    h = oracle.rmsnorm(xn, g, eps)
    q_ref, s_ref = oracle.act_quant(h)
    assert (s_ref < 2.0 ** -123).all()  # every row takes the division route
    q = torch.full((M, K), 99, dtype=torch.int8, device=DEV)
    a = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    woq.woq_rmsnorm_act_quant_int8(_dev_bf16(xn), _dev_bf16(g), eps, q, a)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(a.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    out, ws = Guarded(M, N), Workspace(bits, M, N, K)
    fn = woq.woq_w4a8_linear_rmsnorm_bf16 if bits == 4 else woq.woq_w6a8_linear_rmsnorm_bf16
    fn(wdev, _dev_bf16(xn), _dev_bf16(g), eps, N, K, out.y, ws.ws)
    torch.cuda.synchronize()
    out.check_guards()
    ws.check()
    y = out.numpy()
    y_ref, S = oracle.linear_rmsnorm(bits, wn, sn, N, K, xn, g, eps)
    ok, worst = tol_ok(y, y_ref, S)
    assert ok, f"max err / tolerance = {worst}"
    assert np.array_equal(y.view(np.uint32), _gemv(bits, wdev, q, a, N, K, M).view(np.uint32))


@pytest.mark.parametrize("bits,path", [(4, 1), (4, 2), (6, 1)])
@pytest.mark.parametrize("M", [1, 3, 4])
@pytest.mark.parametrize("K", [1024, 17408])
def test_fused_swiglu_linear_on_a_tiny_up_half(bits, path, M, K):
    if K > woq.woq_max_k(bits, M, True):
        pytest.skip("beyond the fused entry's shared-memory limit for these rows")
    woq.woq_tune_path(path)
    N = 384
    wn, sn, wdev = _weights(bits, N, K, seed=17 * M + K + bits)
    gu = synthetic.gate_up_output(M, K, seed=3 * M + K).numpy().copy()
    gu[:, K:] *= np.float32(TINY_U)
    q_ref, s_ref = oracle.act_quant(oracle.swiglu(gu))
    assert (s_ref < 2.0 ** -123).all()
    gu_dev = torch.from_numpy(gu).to(DEV)
    q = torch.full((M, K), 99, dtype=torch.int8, device=DEV)
    a = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    woq.woq_swiglu_act_quant_int8(gu_dev, q, a)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(a.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    out, ws = Guarded(M, N), Workspace(bits, M, N, K)
    fn = woq.woq_w4a8_linear_swiglu_f32 if bits == 4 else woq.woq_w6a8_linear_swiglu_f32
    fn(wdev, gu_dev, N, K, out.y, ws.ws)
    torch.cuda.synchronize()
    out.check_guards()
    ws.check()
    y = out.numpy()
    y_ref, S = oracle.linear_swiglu(bits, wn, sn, N, K, gu)
    ok, worst = tol_ok(y, y_ref, S)
    assert ok, f"max err / tolerance = {worst}"
    assert np.array_equal(y.view(np.uint32), _gemv(bits, wdev, q, a, N, K, M).view(np.uint32))
