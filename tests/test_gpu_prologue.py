"""GPU parity of the prologue fusions (RMSNorm or SwiGLU absorbed by the activation
quantisation): the standalone twins against the oracle bit for bit (q bytes and scale
bits), the fused linears against the oracle within the GEMV tolerance and bit-identical to
twin + GEMV, for int4 on both consumers and for int6."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import to_numpy_u16, to_numpy_u8
from tests.test_gpu_parity import DEV, Guarded, Workspace, pack_host, tol_ok

pytestmark = pytest.mark.gpu

woq = None


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


def _rms_inputs(M, K, seed):
    x = synthetic.activations(M, K, seed=seed, outliers=True)
    xn = to_numpy_u16(x)
    if M >= 2:
        xn[1] = 0  # an all-zero row
    g = to_numpy_u16(synthetic.rmsnorm_weight(K, seed))
    return xn, g


def _dev_bf16(a):
    return torch.from_numpy(a.view(np.int16)).to(DEV).view(torch.bfloat16)


def _gu_inputs(M, K, seed):
    gu = synthetic.gate_up_output(M, K, seed).numpy().copy()
    gu[0, :6] = [0.0, 100.0, -100.0, 50.0, -87.5, 88.8]  # exp underflow / overflow edges
    gu[0, 6:10] = [-88.5, -88.7, -88.4, 87.3]  # e^-g with n = 128 in the scaling by 2^n, and near the top
    return gu


@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("K", [1024, 5120, 17408])
@pytest.mark.parametrize("eps", [1e-6, 0.0])
def test_rmsnorm_act_quant_bit_exact(M, K, eps):
    xn, g = _rms_inputs(M, K, seed=M * 11 + K)
    q_ref, s_ref = oracle.act_quant(oracle.rmsnorm(xn, g, eps))
    q = torch.full((M, K), 99, dtype=torch.int8, device=DEV)
    s = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    woq.woq_rmsnorm_act_quant_int8(_dev_bf16(xn), _dev_bf16(g), eps, q, s)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("M", [1, 4, 8])
@pytest.mark.parametrize("K", [1024, 5120, 17408])
def test_swiglu_act_quant_bit_exact(M, K):
    gu = _gu_inputs(M, K, seed=M * 13 + K)
    q_ref, s_ref = oracle.act_quant(oracle.swiglu(gu))
    q = torch.full((M, K), 99, dtype=torch.int8, device=DEV)
    s = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    woq.woq_swiglu_act_quant_int8(torch.from_numpy(gu).to(DEV), q, s)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


BITS_PATHS = [(4, 1), (4, 2), (6, 1)]


def _run(fn, *args):
    fn(*args)
    torch.cuda.synchronize()


@pytest.mark.parametrize("bits,path", BITS_PATHS)
@pytest.mark.parametrize("M", [1, 3, 4])
@pytest.mark.parametrize("N,K", [(1000, 1024), (300, 384), (2048, 5120), (700, 6144), (700, 6272), (64, 256)])
def test_fused_rmsnorm_linear(bits, path, M, N, K):
    """K = 6144 is the largest row the fused RMSNorm keeps in registers (M <= 4); 6272 takes
    the shared-memory passes."""
    woq.woq_tune_path(path)
    w, s = synthetic.weights(bits, N, K, seed=3 * N + K + bits)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    xn, g = _rms_inputs(M, K, seed=N + M)
    eps = 1e-6
    y_ref, S = oracle.linear_rmsnorm(bits, wn, sn, N, K, xn, g, eps)
    wdev = pack_host(bits, wn, sn, N, K)
    out, ws = Guarded(M, N), Workspace(bits, M, N, K)
    fn = woq.woq_w4a8_linear_rmsnorm_bf16 if bits == 4 else woq.woq_w6a8_linear_rmsnorm_bf16
    _run(fn, wdev, _dev_bf16(xn), _dev_bf16(g), eps, N, K, out.y, ws.ws)
    out.check_guards()
    ws.check()
    y = out.numpy()
    ok, worst = tol_ok(y, y_ref, S)
    assert ok, f"max err / tolerance = {worst}"
    # bit-identical to the unfused twin followed by the GEMV
    q = torch.empty((M, K), dtype=torch.int8, device=DEV)
    a = torch.empty((M,), dtype=torch.float32, device=DEV)
    woq.woq_rmsnorm_act_quant_int8(_dev_bf16(xn), _dev_bf16(g), eps, q, a)
    out2, ws2 = Guarded(M, N), Workspace(bits, M, N, K)
    gemv = woq.woq_w4a8_gemv if bits == 4 else woq.woq_w6a8_gemv
    _run(gemv, wdev, q, a, N, K, out2.y, ws2.ws)
    assert np.array_equal(y.view(np.uint32), out2.numpy().view(np.uint32))


@pytest.mark.parametrize("bits,path", BITS_PATHS)
@pytest.mark.parametrize("M", [1, 3, 4])
@pytest.mark.parametrize("N,K", [(1000, 1024), (300, 384), (640, 5120), (64, 256)])
def test_fused_swiglu_linear(bits, path, M, N, K):
    """(64, 256) is two blocks: a grid of one CTA, whose grid-wide maximum is its own."""
    woq.woq_tune_path(path)
    w, s = synthetic.weights(bits, N, K, seed=5 * N + K + bits)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    gu = _gu_inputs(M, K, seed=N + 7 * M)
    y_ref, S = oracle.linear_swiglu(bits, wn, sn, N, K, gu)
    wdev = pack_host(bits, wn, sn, N, K)
    out, ws = Guarded(M, N), Workspace(bits, M, N, K)
    fn = woq.woq_w4a8_linear_swiglu_f32 if bits == 4 else woq.woq_w6a8_linear_swiglu_f32
    gu_dev = torch.from_numpy(gu).to(DEV)
    _run(fn, wdev, gu_dev, N, K, out.y, ws.ws)
    out.check_guards()
    ws.check()
    y = out.numpy()
    ok, worst = tol_ok(y, y_ref, S)
    assert ok, f"max err / tolerance = {worst}"
    q = torch.empty((M, K), dtype=torch.int8, device=DEV)
    a = torch.empty((M,), dtype=torch.float32, device=DEV)
    woq.woq_swiglu_act_quant_int8(gu_dev, q, a)
    out2, ws2 = Guarded(M, N), Workspace(bits, M, N, K)
    gemv = woq.woq_w4a8_gemv if bits == 4 else woq.woq_w6a8_gemv
    _run(gemv, wdev, q, a, N, K, out2.y, ws2.ws)
    assert np.array_equal(y.view(np.uint32), out2.numpy().view(np.uint32))


@pytest.mark.parametrize("M", [5, 8])
def test_fused_prologues_wide_m(M):
    N, K = 640, 2048
    w, s = synthetic.weights(4, N, K, seed=M)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    wdev = pack_host(4, wn, sn, N, K)
    xn, g = _rms_inputs(M, K, seed=M + 1)
    y_ref, S = oracle.linear_rmsnorm(4, wn, sn, N, K, xn, g, 1e-5)
    out, ws = Guarded(M, N), Workspace(4, M, N, K)
    _run(woq.woq_w4a8_linear_rmsnorm_bf16, wdev, _dev_bf16(xn), _dev_bf16(g), 1e-5, N, K, out.y, ws.ws)
    assert tol_ok(out.numpy(), y_ref, S)[0]
    gu = _gu_inputs(M, K, seed=M + 2)
    y_ref, S = oracle.linear_swiglu(4, wn, sn, N, K, gu)
    out, ws = Guarded(M, N), Workspace(4, M, N, K)
    _run(woq.woq_w4a8_linear_swiglu_f32, wdev, torch.from_numpy(gu).to(DEV), N, K, out.y, ws.ws)
    assert tol_ok(out.numpy(), y_ref, S)[0]


@pytest.mark.parametrize("M,K,N", [(1, 17408, 5120), (4, 17408, 5120), (2, 5120, 1000)])
def test_fused_swiglu_repeated_launches(M, K, N):
    """The fused SwiGLU linear splits the SwiGLU over the grid (slices in the workspace
    scratch rows, a grid-wide maximum): repeated launches on one workspace give identical
    y, equal to twin + GEMV, and leave every word but the scratch rows zero.  The shapes
    take the register route (M = 1) and the shared-memory route (M = 4) of the prologue."""
    w, s = synthetic.weights(4, N, K, seed=K + M)
    wdev = pack_host(4, to_numpy_u8(w), to_numpy_u16(s), N, K)
    gu_dev = torch.from_numpy(_gu_inputs(M, K, seed=M + 5)).to(DEV)
    nbytes = woq.woq_workspace_bytes(4, M, N, K)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    ys = []
    for _ in range(3):
        y = torch.empty((M, N), dtype=torch.float32, device=DEV)
        woq.woq_w4a8_linear_swiglu_f32(wdev, gu_dev, N, K, y, ws)
        ys.append(y)
    torch.cuda.synchronize()
    assert woq.woq_read_status(ws) == 0
    assert not ws[: nbytes - M * K * 2].cpu().numpy().any()
    q = torch.empty((M, K), dtype=torch.int8, device=DEV)
    a = torch.empty((M,), dtype=torch.float32, device=DEV)
    woq.woq_swiglu_act_quant_int8(gu_dev, q, a)
    y2 = torch.empty((M, N), dtype=torch.float32, device=DEV)
    woq.woq_w4a8_gemv(wdev, q, a, N, K, y2, ws)
    torch.cuda.synchronize()
    for y in ys:
        assert torch.equal(y.view(torch.int32), y2.view(torch.int32))


def _sampled_rows(N, n_rand, seed):
    rng = np.random.default_rng(seed)
    rows = set([0, 1, 127, 128, N - 1]) | set(rng.integers(0, N, size=n_rand).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < N))


@pytest.mark.parametrize("kind,M,K,N", [
    ("swiglu", 1, 17408, 5120),   # 27B down projection after SwiGLU of the gate+up output
    ("swiglu", 4, 17408, 5120),
    ("rmsnorm", 4, 5120, 7168),   # 27B QKV after the input RMSNorm
])
def test_full_size_prologue_sampled_rows(kind, M, K, N):
    seed = 300 + M
    w, s = synthetic.weights(4, N, K, seed, device=DEV)
    wdev = torch.empty(woq.woq_packed_bytes(4, N, K), dtype=torch.uint8, device=DEV)
    woq.woq_pack_device(4, w, s.view(torch.int16), N, K, wdev)
    out, ws = Guarded(M, N), Workspace(4, M, N, K)
    if kind == "swiglu":
        gu = _gu_inputs(M, K, seed)
        _run(woq.woq_w4a8_linear_swiglu_f32, wdev, torch.from_numpy(gu).to(DEV), N, K, out.y, ws.ws)
        h = oracle.swiglu(gu)
    else:
        xn, g = _rms_inputs(M, K, seed)
        _run(woq.woq_w4a8_linear_rmsnorm_bf16, wdev, _dev_bf16(xn), _dev_bf16(g), 1e-6, N, K, out.y, ws.ws)
        h = oracle.rmsnorm(xn, g, 1e-6)
    rows = _sampled_rows(N, 40, seed)
    idx = torch.from_numpy(rows).to(DEV)
    wn = to_numpy_u8(w.index_select(0, idx))
    sn = to_numpy_u16(s.index_select(0, idx))
    y_ref, S = oracle.linear_bf16(4, wn, sn, len(rows), K, h)
    ok, worst = tol_ok(out.numpy()[:, rows], y_ref, S)
    assert ok, f"max err / tolerance = {worst}"


def test_prologue_argument_errors():
    N, K, M = 128, 256, 1
    w = torch.zeros(woq.woq_packed_bytes(4, N, K), dtype=torch.uint8, device=DEV)
    x = torch.zeros((M, K), dtype=torch.bfloat16, device=DEV)
    g = torch.zeros((K + 8,), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((M, N), device=DEV)
    ws = torch.zeros(woq.woq_workspace_bytes(4, M, N, K), dtype=torch.uint8, device=DEV)
    with pytest.raises(woq.WoqError) as e:
        woq.woq_w4a8_linear_rmsnorm_bf16(w, x, g[1:], 1e-6, N, K, y, ws)  # gamma not 16-byte aligned
    assert e.value.status == woq.WOQ_ERR_ALIGN
    with pytest.raises(woq.WoqError) as e:
        woq.woq_w4a8_linear_rmsnorm_bf16(w, x, g, -1.0, N, K, y, ws)
    assert e.value.status == woq.WOQ_ERR_SHAPE
    q = torch.empty((M, 100), dtype=torch.int8, device=DEV)
    a = torch.empty((M,), device=DEV)
    with pytest.raises(woq.WoqError) as e:
        woq.woq_swiglu_act_quant_int8(torch.zeros((M, 200), device=DEV), q, a)  # K = 100 is not a multiple of 8
    assert e.value.status == woq.WOQ_ERR_SHAPE
