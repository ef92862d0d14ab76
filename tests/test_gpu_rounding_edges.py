"""GPU parity at the quantiser's rounding edge: activations whose quotients x / s are exact
half-integers, or fp32 quotients within 3e-5 of one.

The activation quantiser rounds half to even ("Optimizing the Linear Kernel" quantises the
activation to int8; the rounding rule is the reading of the pages used throughout).  The
kernels reach that rounding by multiplying with the reciprocal of the row scale and fall
back to the IEEE division for quotients this close to a tie, so these rows exercise the
fallback.  Rows are built here from known values:
  - power-of-two rows: amax = 127 * 2^j and x = (k + 1/2) 2^j, so s = 2^j and every x / s is
    a half-integer;
  - near-tie rows: amax = (1 + f/128) 2^e for every f; the x are the bf16 values whose
    IEEE fp32 quotient x / s is within 3e-5 of a half-integer (or lands on one), found by
    enumerating every bf16 value below amax.
They run through woq_act_quant_int8 (q bytes and scale bits against the oracle), the fused
bf16 linears (int4 dp4a, int4 tensor-core MMA, int6; rows that fit registers and rows that
do not: bit-identical to act_quant + GEMV and within the tolerance of the oracle), and the
RMSNorm and SwiGLU twins and fused linears, whose h is made to equal such a row exactly
(RMSNorm: x = +-1, eps = 0, so r = 1 and h = +-gamma; SwiGLU: gate 32, so the sigmoid is 1
in fp32 and h = 32 up).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import to_numpy_u16, to_numpy_u8
from tests.test_gpu_parity import DEV, Workspace, pack_host, run_gemv, run_linear, tol_ok

pytestmark = pytest.mark.gpu

woq = None
DP4A, MMA = 1, 2


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


# ----------------------------------------------------------------------------- tie rows

_POS_BF16 = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)  # every positive finite bf16


def _bits(v: np.ndarray) -> np.ndarray:
    """fp32 values that are bf16-exact -> bf16 bit patterns."""
    b = np.asarray(v, dtype=np.float32).view(np.uint32)
    assert not (b & 0xFFFF).any(), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def _near_tie_values(A: np.float32):
    """bf16 values x in (0, A] whose fp32 quotient x / s, s = fp32(A) / 127, is within 3e-5 of
    a half-integer (or on one)."""
    s = np.float32(A) / np.float32(127)
    xs = _POS_BF16[_POS_BF16 <= A]
    t = xs / s  # IEEE fp32 division
    d = np.abs(t - np.floor(t) - np.float32(0.5))
    return xs[d < 3e-5]


def tie_rows(M: int, K: int, seed: int) -> np.ndarray:
    """bf16 bit patterns [M, K]: row m is a power-of-two tie row for even m and a near-tie
    row for odd m; about half the entries are (near-)ties with random signs, the rest random
    bf16 values in [amax 2^-20, amax), and the amax sits at a random position."""
    rng = np.random.default_rng(seed)
    out = np.zeros((M, K), dtype=np.float32)
    for m in range(M):
        if m % 2 == 0:
            j = int(rng.integers(-6, 7))
            A = np.float32(127.0 * 2.0 ** j)
            ties = ((np.arange(127) + 0.5) * 2.0 ** j).astype(np.float32)
        else:
            e = int(rng.integers(-4, 5))
            while True:
                f = int(rng.integers(0, 128))
                A0 = np.float32(1 + f / 128)
                ties = _near_tie_values(A0)
                if len(ties):
                    break
            A = np.float32(A0 * np.float32(2.0 ** e))
            ties = (ties * np.float32(2.0 ** e)).astype(np.float32)
        others = _POS_BF16[(_POS_BF16 < A) & (_POS_BF16 >= A * np.float32(2.0 ** -20))]
        pick_tie = rng.random(K) < 0.5
        row = np.where(pick_tie, ties[rng.integers(0, len(ties), K)], others[rng.integers(0, len(others), K)])
        row = row * np.where(rng.random(K) < 0.5, -1.0, 1.0).astype(np.float32)
        row[int(rng.integers(0, K))] = A * (1 if rng.random() < 0.5 else -1)
        out[m] = row
    return _bits(out)


def _quotient_tie_count(xn: np.ndarray, s: np.ndarray) -> int:
    x = (xn.astype(np.uint32) << 16).view(np.float32)
    t = np.abs(x / s[:, None].astype(np.float32))
    d = np.abs(t - np.floor(t) - np.float32(0.5))
    return int((d < 3e-5).sum())


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def test_tie_rows_are_ties():
    """The builder's rows really put many quotients on or within 3e-5 of a tie (as the oracle
    scales them)."""
    xn = tie_rows(4, 4096, seed=1)
    _, s = oracle.act_quant(xn)
    assert _quotient_tie_count(xn, s) > 4 * 4096 * 0.4


# ----------------------------------------------------------------------------- act_quant

@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("K", [128, 5120, 17408])
def test_act_quant_on_ties_bit_exact(M, K):
    xn = tie_rows(M, K, seed=10 * M + K)
    q_ref, s_ref = oracle.act_quant(xn)
    q = torch.full((M, K), 99, dtype=torch.int8, device=DEV)
    s = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    woq.woq_act_quant_int8(_dev_bf16(xn), q, s)
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)


# ----------------------------------------------------------------------------- fused bf16 linear

# rows read into registers (M <= 3, M K within the register budget) and rows copied into shared
# memory (longer rows, and every M = 4 row), for each consumer
@pytest.mark.parametrize("bits,path", [(4, DP4A), (4, MMA), (6, DP4A)])
@pytest.mark.parametrize("M,K", [(1, 5120), (1, 24704), (2, 12288), (2, 12416), (3, 8192), (3, 8320),
                                 (4, 1024), (4, 6272)])
def test_fused_linear_on_ties(bits, path, M, K):
    woq.woq_tune_path(path)
    N = 384
    w, s = synthetic.weights(bits, N, K, seed=K + M + bits)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    xn = tie_rows(M, K, seed=3 * K + M)
    y_ref, S = oracle.linear_bf16(bits, wn, sn, N, K, xn)
    wdev = pack_host(bits, wn, sn, N, K)
    x_dev = _dev_bf16(xn)
    y = run_linear(bits, wdev, x_dev, N, K, M)
    ok, worst = tol_ok(y, y_ref, S)
    assert ok, f"max err / tolerance = {worst}"
    q = torch.empty((M, K), dtype=torch.int8, device=DEV)
    a = torch.empty((M,), dtype=torch.float32, device=DEV)
    woq.woq_act_quant_int8(x_dev, q, a)
    y2 = run_gemv(bits, wdev, q, a, N, K, M)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


# ----------------------------------------------------------------------------- RMSNorm and SwiGLU

def _rms_tie_inputs(M, K, seed):
    """x = +-1 (mean of squares exactly 1) and eps = 0 give r = 1, so h = +-gamma: gamma is a
    tie row."""
    rng = np.random.default_rng(seed)
    x = _bits(np.where(rng.random((M, K)) < 0.5, -1.0, 1.0).astype(np.float32))
    gamma = tie_rows(2, K, seed)[seed % 2]  # a power-of-two or a near-tie row
    return x, gamma


def _swiglu_tie_inputs(M, K, seed):
    """gate = 32: e^-32 vanishes next to 1 in fp32, so the sigmoid is exactly 1 and h = 32 up
    exactly; up = row / 32 makes h a tie row."""
    h = (tie_rows(M, K, seed).astype(np.uint32) << 16).view(np.float32)
    gu = np.concatenate([np.full((M, K), 32.0, np.float32), h / np.float32(32)], axis=1)
    return np.ascontiguousarray(gu), _bits(h)


@pytest.mark.parametrize("M", [1, 3, 4])
@pytest.mark.parametrize("K", [1024, 6144, 17408])
def test_prologue_twins_on_ties(M, K):
    x, gamma = _rms_tie_inputs(M, K, seed=K + M)
    h = oracle.rmsnorm(x, gamma, 0.0)
    assert np.array_equal(h, np.where(x >> 15, gamma ^ 0x8000, gamma))  # h = +-gamma exactly
    q_ref, s_ref = oracle.act_quant(h)
    assert _quotient_tie_count(h, s_ref) > M * K * 0.4
    q = torch.full((M, K), 99, dtype=torch.int8, device=DEV)
    s = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    woq.woq_rmsnorm_act_quant_int8(_dev_bf16(x), _dev_bf16(gamma), 0.0, q, s)
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)

    gu, h_want = _swiglu_tie_inputs(M, K, seed=K + 7 * M)
    h = oracle.swiglu(gu)
    assert np.array_equal(h, h_want)
    q_ref, s_ref = oracle.act_quant(h)
    q.fill_(99)
    s.fill_(-1.0)
    woq.woq_swiglu_act_quant_int8(torch.from_numpy(gu).to(DEV), q, s)
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)


@pytest.mark.parametrize("bits,path", [(4, DP4A), (4, MMA), (6, DP4A)])
@pytest.mark.parametrize("M,K", [(1, 5120), (4, 5120), (2, 12288), (4, 17408)])
def test_fused_prologue_linears_on_ties(bits, path, M, K):
    """RMSNorm (rows in registers for K <= 6144, else shared memory) and SwiGLU (split over the
    grid) fused linears: within the tolerance of the oracle and bit-identical to twin + GEMV."""
    if K > woq.woq_max_k(bits, M, True):
        pytest.skip("beyond the fused entry's activation tile")
    woq.woq_tune_path(path)
    N = 256
    w, s = synthetic.weights(bits, N, K, seed=5 * K + M + bits)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    wdev = pack_host(bits, wn, sn, N, K)
    q = torch.empty((M, K), dtype=torch.int8, device=DEV)
    a = torch.empty((M,), dtype=torch.float32, device=DEV)

    x, gamma = _rms_tie_inputs(M, K, seed=K + 3 * M)
    y_ref, S = oracle.linear_rmsnorm(bits, wn, sn, N, K, x, gamma, 0.0)
    ws = Workspace(bits, M, N, K)
    y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    fn = woq.woq_w4a8_linear_rmsnorm_bf16 if bits == 4 else woq.woq_w6a8_linear_rmsnorm_bf16
    fn(wdev, _dev_bf16(x), _dev_bf16(gamma), 0.0, N, K, y, ws.ws)
    torch.cuda.synchronize()
    ws.check()
    yn = y.cpu().numpy()
    ok, worst = tol_ok(yn, y_ref, S)
    assert ok, f"RMSNorm: max err / tolerance = {worst}"
    woq.woq_rmsnorm_act_quant_int8(_dev_bf16(x), _dev_bf16(gamma), 0.0, q, a)
    assert np.array_equal(yn.view(np.uint32), run_gemv(bits, wdev, q, a, N, K, M).view(np.uint32))

    gu, _ = _swiglu_tie_inputs(M, K, seed=K + 5 * M)
    y_ref, S = oracle.linear_swiglu(bits, wn, sn, N, K, gu)
    ws = Workspace(bits, M, N, K)
    fn = woq.woq_w4a8_linear_swiglu_f32 if bits == 4 else woq.woq_w6a8_linear_swiglu_f32
    gu_dev = torch.from_numpy(gu).to(DEV)
    fn(wdev, gu_dev, N, K, y, ws.ws)
    torch.cuda.synchronize()
    ws.check()
    yn = y.cpu().numpy()
    ok, worst = tol_ok(yn, y_ref, S)
    assert ok, f"SwiGLU: max err / tolerance = {worst}"
    woq.woq_swiglu_act_quant_int8(gu_dev, q, a)
    assert np.array_equal(yn.view(np.uint32), run_gemv(bits, wdev, q, a, N, K, M).view(np.uint32))
