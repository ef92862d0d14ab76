"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Bars: act_quant (q bytes and scale bits) and the per-group dot products are
bit-exact; y is within |y_gpu - y_ref| <= 1e-5 * sum_g |term_g| + 1e-6 per
element; the fused bf16 entry is bit-identical to act_quant followed by the
GEMV; repeated launches are bit-identical.  The int4 GEMV / linear tests run
with each consumer forced (dp4a, and the tensor-core MMA); int6 always uses dp4a.  Inputs are the seeded synthetic
workloads (synthetic.py).  Guard regions around outputs and workspace catch
writes out of bounds.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from synthetic import to_numpy_u16, to_numpy_u8

pytestmark = pytest.mark.gpu

woq = None


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    global woq
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import weight_only_quantised_gb300 as w
    woq = w
    torch.cuda.set_device(0)
    yield
    woq.woq_tune_override(0, 0, -1)
    woq.woq_tune_path(0)


DP4A, MMA = 1, 2
BITS_PATHS = [(4, DP4A), (4, MMA), (6, DP4A)]


@pytest.fixture()
def consumer():
    """Force the int4 consumer for one test: consumer(path)."""
    def set_path(path):
        woq.woq_tune_path(path)
    yield set_path
    woq.woq_tune_path(0)


DEV = "cuda:0"
GUARD = 64  # guard elements on each side of an output
SENT = -12345.678


def tol_ok(y, y_ref, S):
    err = np.abs(y.astype(np.float64) - y_ref.astype(np.float64))
    bound = oracle.tolerance(S)
    return bool((err <= bound).all()), float((err / bound).max()) if err.size else 0.0


class Guarded:
    """A device fp32 output [M, N] with sentinel guard regions on both sides."""

    def __init__(self, M, N):
        self.M, self.N = M, N
        self.buf = torch.full((M * N + 2 * GUARD,), SENT, dtype=torch.float32, device=DEV)
        self.y = self.buf[GUARD: GUARD + M * N].view(M, N)

    def check_guards(self):
        b = self.buf.cpu().numpy()
        assert (b[:GUARD] == np.float32(SENT)).all() and (b[GUARD + self.M * self.N:] == np.float32(SENT)).all()

    def numpy(self):
        return self.y.cpu().numpy()


class Workspace:
    def __init__(self, bits, M, N, K):
        self.n = woq.woq_workspace_bytes(bits, M, N, K)
        self.buf = torch.full((self.n + 4096,), 0xA5, dtype=torch.uint8, device=DEV)
        self.ws = self.buf[: self.n]
        woq.woq_workspace_init(self.ws)

    def check(self):
        tail = self.buf[self.n:].cpu().numpy()
        assert (tail == 0xA5).all(), "write past the end of the workspace"
        assert woq.woq_read_status(self.ws) == 0


def make_weights(bits, N, K, seed, device="cpu"):
    w, s = synthetic.weights(bits, N, K, seed, device=device)
    return w, s


def pack_host(bits, wn, sn, N, K):
    fn = woq.woq_pack_w4 if bits == 4 else woq.woq_pack_w6
    return torch.from_numpy(fn(wn, sn, N, K)).to(DEV)


def run_gemv(bits, wdev, q_dev, as_dev, N, K, M):
    out = Guarded(M, N)
    ws = Workspace(bits, M, N, K)
    fn = woq.woq_w4a8_gemv if bits == 4 else woq.woq_w6a8_gemv
    fn(wdev, q_dev, as_dev, N, K, out.y, ws.ws)
    torch.cuda.synchronize()
    out.check_guards()
    ws.check()
    return out.numpy()


def run_linear(bits, wdev, x_dev, N, K, M, ws=None):
    out = Guarded(M, N)
    own = ws is None
    if own:
        ws = Workspace(bits, M, N, K)
    fn = woq.woq_w4a8_linear_bf16 if bits == 4 else woq.woq_w6a8_linear_bf16
    fn(wdev, x_dev, N, K, out.y, ws.ws)
    torch.cuda.synchronize()
    out.check_guards()
    if own:
        ws.check()
    return out.numpy()


# --------------------------------------------------------------------------- act_quant

@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("K", [128, 1000, 5120, 17408])
def test_act_quant_bit_exact(M, K):
    x = synthetic.activations(M, K, seed=1000 + M * 7 + K, outliers=True)
    xn = to_numpy_u16(x)
    if M >= 2:
        xn[1] = 0  # an all-zero row: scale 0, q 0
    if M >= 3:
        xn[2] = (xn[2] & 0x8000) | 0x0080  # tiny values (smallest normal bf16 magnitude)
    q_ref, s_ref = oracle.act_quant(xn)
    x_dev = torch.from_numpy(xn.view(np.int16)).to(DEV).view(torch.bfloat16)
    q = torch.full((M, K), 99, dtype=torch.int8, device=DEV)
    s = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    woq.woq_act_quant_int8(x_dev, q, s)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


# --------------------------------------------------------------------------- group dots

@pytest.mark.parametrize("bits,M", [(4, 1), (4, 4), (4, 8), (6, 1), (6, 4)])
@pytest.mark.parametrize("N,K", [(1000, 1024), (300, 384), (129, 128)])
def test_group_dots_bit_exact(bits, M, N, K):
    w, s = make_weights(bits, N, K, seed=N + K + bits)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    x = synthetic.activations(M, K, seed=N * 3 + M, outliers=True)
    q_ref, _ = oracle.act_quant(to_numpy_u16(x))
    d_ref = oracle.group_dots(bits, wn, N, K, q_ref)
    wdev = pack_host(bits, wn, sn, N, K)
    q_dev = torch.from_numpy(q_ref).to(DEV)
    dots = torch.zeros((M, N, K // 128), dtype=torch.int32, device=DEV)
    woq.woq_debug_group_dots(bits, wdev, q_dev, N, K, dots)
    torch.cuda.synchronize()
    assert np.array_equal(dots.cpu().numpy(), d_ref)


# --------------------------------------------------------------------------- GEMV / linear

SHAPES = [(1024, 1024), (1000, 1024), (300, 384), (129, 128), (4096, 512), (640, 2048)]


@pytest.mark.parametrize("bits,path", BITS_PATHS)
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", SHAPES)
def test_gemv_matches_oracle(bits, path, M, N, K, consumer):
    consumer(path)
    w, s = make_weights(bits, N, K, seed=7 * N + K + bits)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    x = synthetic.activations(M, K, seed=N + 3 * M, outliers=True)
    q_ref, s_ref = oracle.act_quant(to_numpy_u16(x))
    y_ref, S = oracle.gemv(bits, wn, sn, N, K, q_ref, s_ref)
    wdev = pack_host(bits, wn, sn, N, K)
    y = run_gemv(bits, wdev, torch.from_numpy(q_ref).to(DEV), torch.from_numpy(s_ref).to(DEV), N, K, M)
    ok, worst = tol_ok(y, y_ref, S)
    assert ok, f"max err / tolerance = {worst}"


@pytest.mark.parametrize("bits,path", BITS_PATHS)
@pytest.mark.parametrize("M", [1, 3, 4])
@pytest.mark.parametrize("N,K", [(1000, 1024), (300, 384), (2048, 4096)])
def test_fused_linear_matches_oracle_and_separate_path(bits, path, M, N, K, consumer):
    consumer(path)
    w, s = make_weights(bits, N, K, seed=11 * N + K + bits)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    x = synthetic.activations(M, K, seed=5 * N + M, outliers=True)
    xn = to_numpy_u16(x)
    y_ref, S = oracle.linear_bf16(bits, wn, sn, N, K, xn)
    wdev = pack_host(bits, wn, sn, N, K)
    x_dev = torch.from_numpy(xn.view(np.int16)).to(DEV).view(torch.bfloat16)
    y = run_linear(bits, wdev, x_dev, N, K, M)
    ok, worst = tol_ok(y, y_ref, S)
    assert ok, f"max err / tolerance = {worst}"
    # the fused entry equals act_quant + GEMV bit for bit
    q = torch.empty((M, K), dtype=torch.int8, device=DEV)
    a = torch.empty((M,), dtype=torch.float32, device=DEV)
    woq.woq_act_quant_int8(x_dev, q, a)
    y2 = run_gemv(bits, wdev, q, a, N, K, M)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


# The fused entry reads rows that fit registers (up to 12 vectors of 8 values per thread over the
# M rows) straight from global memory for M <= 3, and copies longer rows (and every M = 4 row) into
# shared memory first: both sides of each limit, against the oracle and the separate path.
@pytest.mark.parametrize("bits", [4, 6])
@pytest.mark.parametrize("M,K", [(1, 24576), (1, 24704), (2, 12288), (2, 12416), (3, 8192), (3, 8320),
                                 (4, 6144), (4, 6272)])
def test_fused_linear_register_limit(bits, M, K):
    N = 300
    w, s = make_weights(bits, N, K, seed=17 * K + M + bits)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    x = synthetic.activations(M, K, seed=3 * K + M, outliers=True)
    xn = to_numpy_u16(x)
    y_ref, S = oracle.linear_bf16(bits, wn, sn, N, K, xn)
    wdev = pack_host(bits, wn, sn, N, K)
    x_dev = torch.from_numpy(xn.view(np.int16)).to(DEV).view(torch.bfloat16)
    y = run_linear(bits, wdev, x_dev, N, K, M)
    ok, worst = tol_ok(y, y_ref, S)
    assert ok, f"max err / tolerance = {worst}"
    q = torch.empty((M, K), dtype=torch.int8, device=DEV)
    a = torch.empty((M,), dtype=torch.float32, device=DEV)
    woq.woq_act_quant_int8(x_dev, q, a)
    y2 = run_gemv(bits, wdev, q, a, N, K, M)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


# M = 5 .. 8 (int4 only): the launch table runs the tensor-core consumer
@pytest.mark.parametrize("M", [5, 6, 7, 8])
@pytest.mark.parametrize("N,K", [(1000, 1024), (300, 384), (129, 128), (640, 2048)])
def test_gemv_wide_m_matches_oracle(M, N, K):
    bits = 4
    w, s = make_weights(bits, N, K, seed=13 * N + K + M)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    x = synthetic.activations(M, K, seed=N + 5 * M, outliers=True)
    q_ref, s_ref = oracle.act_quant(to_numpy_u16(x))
    y_ref, S = oracle.gemv(bits, wn, sn, N, K, q_ref, s_ref)
    wdev = pack_host(bits, wn, sn, N, K)
    y = run_gemv(bits, wdev, torch.from_numpy(q_ref).to(DEV), torch.from_numpy(s_ref).to(DEV), N, K, M)
    ok, worst = tol_ok(y, y_ref, S)
    assert ok, f"max err / tolerance = {worst}"


@pytest.mark.parametrize("M", [5, 8])
@pytest.mark.parametrize("N,K", [(1000, 1024), (2048, 4096), (300, 5120)])
def test_fused_linear_wide_m(M, N, K):
    bits = 4
    w, s = make_weights(bits, N, K, seed=17 * N + K + M)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    xn = to_numpy_u16(synthetic.activations(M, K, seed=7 * N + M, outliers=True))
    xn[M - 2] = 0  # an all-zero row
    y_ref, S = oracle.linear_bf16(bits, wn, sn, N, K, xn)
    wdev = pack_host(bits, wn, sn, N, K)
    x_dev = torch.from_numpy(xn.view(np.int16)).to(DEV).view(torch.bfloat16)
    y = run_linear(bits, wdev, x_dev, N, K, M)
    ok, worst = tol_ok(y, y_ref, S)
    assert ok, f"max err / tolerance = {worst}"
    assert not y[M - 2].any()
    q = torch.empty((M, K), dtype=torch.int8, device=DEV)
    a = torch.empty((M,), dtype=torch.float32, device=DEV)
    woq.woq_act_quant_int8(x_dev, q, a)
    y2 = run_gemv(bits, wdev, q, a, N, K, M)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


def test_int6_refuses_more_than_four_rows():
    N, K, M = 128, 256, 5
    w = torch.empty(woq.woq_packed_bytes(6, N, K), dtype=torch.uint8, device=DEV)
    x = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((M, N), device=DEV)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    with pytest.raises(woq.WoqError) as e:
        woq.woq_w6a8_linear_bf16(w, x, N, K, y, ws)
    assert e.value.status == woq.WOQ_ERR_SHAPE
    assert woq.woq_workspace_bytes(6, M, N, K) == 0 and woq.woq_max_k(6, M, 1) == 0


@pytest.mark.parametrize("path", [DP4A, MMA])
def test_repeated_launches_are_bit_identical(path, consumer):
    consumer(path)
    bits, M, N, K = 4, 3, 4096, 4096
    w, s = make_weights(bits, N, K, seed=3)
    wdev = pack_host(bits, to_numpy_u8(w), to_numpy_u16(s), N, K)
    x_dev = synthetic.activations(M, K, seed=4).to(DEV)
    ws = Workspace(bits, M, N, K)
    ys = [run_linear(bits, wdev, x_dev, N, K, M, ws=ws) for _ in range(3)]
    ws.check()
    assert all(np.array_equal(ys[0].view(np.uint32), y.view(np.uint32)) for y in ys[1:])
    # every split-tile partial word was consumed and cleared: the workspace is zero again
    assert not ws.ws.cpu().numpy().any()


@pytest.mark.parametrize("bits", [4, 6])
@pytest.mark.parametrize("N,K", [(1000, 1024), (300, 384), (129, 128)])
def test_device_pack_matches_host_pack(bits, N, K):
    w, s = make_weights(bits, N, K, seed=N + 17)
    host = woq.woq_pack_w4(to_numpy_u8(w), to_numpy_u16(s), N, K) if bits == 4 else \
        woq.woq_pack_w6(to_numpy_u8(w), to_numpy_u16(s), N, K)
    dst = torch.full((host.nbytes,), 0x5A, dtype=torch.uint8, device=DEV)
    woq.woq_pack_device(bits, w.to(DEV), s.to(DEV).view(torch.int16), N, K, dst)
    torch.cuda.synchronize()
    assert np.array_equal(dst.cpu().numpy(), host)


@pytest.mark.parametrize("path", [DP4A, MMA])
@pytest.mark.parametrize("cps,stages,pf", [(1, 2, 0), (1, 3, -1), (1, 4, 1024), (2, 2, -1), (2, 3, 64), (1, 8, -1)])
def test_launch_configurations_agree(cps, stages, pf, path, consumer):
    consumer(path)
    bits, M, N, K = 4, 2, 2048, 2048
    w, s = make_weights(bits, N, K, seed=21)
    wn, sn = to_numpy_u8(w), to_numpy_u16(s)
    x = synthetic.activations(M, K, seed=22)
    xn = to_numpy_u16(x)
    y_ref, S = oracle.linear_bf16(bits, wn, sn, N, K, xn)
    wdev = pack_host(bits, wn, sn, N, K)
    x_dev = torch.from_numpy(xn.view(np.int16)).to(DEV).view(torch.bfloat16)
    woq.woq_tune_override(cps, stages, pf)
    try:
        y = run_linear(bits, wdev, x_dev, N, K, M)
    finally:
        woq.woq_tune_override(0, 0, -1)
    ok, worst = tol_ok(y, y_ref, S)
    assert ok, f"max err / tolerance = {worst}"


def test_max_k_bounds():
    for bits in (4, 6):
        for M in range(1, 9 if bits == 4 else 5):
            k8, kb = woq.woq_max_k(bits, M, False), woq.woq_max_k(bits, M, True)
            assert k8 % 128 == 0 and kb % 128 == 0 and 0 < kb <= k8 and M * k8 <= 98304
    # the decode shapes of the 27B and 9B workloads fit the fused entry at M = 4
    assert woq.woq_max_k(4, 4, True) >= 17408 and woq.woq_max_k(6, 4, True) >= 12288
    # beyond the bound the call is refused on the host
    K = woq.woq_max_k(4, 4, True) + 128
    y = torch.empty((4, 128), device=DEV)
    x = torch.empty((4, K), dtype=torch.bfloat16, device=DEV)
    w = torch.empty(woq.woq_packed_bytes(4, 128, K), dtype=torch.uint8, device=DEV)
    ws = torch.zeros(woq.woq_workspace_bytes(4, 4, 128, K), dtype=torch.uint8, device=DEV)
    with pytest.raises(woq.WoqError) as e:
        woq.woq_w4a8_linear_bf16(w, x, 128, K, y, ws)
    assert e.value.status == woq.WOQ_ERR_SHAPE


def test_binding_refuses_bad_tensors_before_any_launch():
    """Undersized, non-contiguous or wrongly typed tensors are refused by the Python entries
    (the library takes bare pointers without sizes); nothing is launched, y keeps its guards."""
    bits, M, N, K = 4, 2, 256, 256
    w, s = make_weights(bits, N, K, seed=3)
    wdev = pack_host(bits, to_numpy_u8(w), to_numpy_u16(s), N, K)
    x = torch.zeros((M, K), dtype=torch.bfloat16, device=DEV)
    out = Guarded(M, N)
    ws = Workspace(bits, M, N, K)
    small_y = out.buf[GUARD: GUARD + M * N - 1]
    with pytest.raises(ValueError, match="elements"):
        woq.woq_w4a8_linear_bf16(wdev, x, N, K, small_y, ws.ws)
    with pytest.raises(ValueError, match="elements"):
        woq.woq_w4a8_linear_bf16(wdev, torch.zeros((M, K - 8), dtype=torch.bfloat16, device=DEV), N, K, out.y, ws.ws)
    with pytest.raises(ValueError, match="contiguous"):
        woq.woq_w4a8_linear_bf16(wdev, torch.zeros((K, M), dtype=torch.bfloat16, device=DEV).t(), N, K, out.y, ws.ws)
    with pytest.raises(ValueError, match="byte elements"):
        woq.woq_w4a8_linear_bf16(wdev, x.float(), N, K, out.y, ws.ws)
    q = torch.zeros((M, K), dtype=torch.int8, device=DEV)
    with pytest.raises(ValueError, match="elements"):
        woq.woq_w4a8_gemv(wdev, q, torch.zeros((M - 1,), device=DEV), N, K, out.y, ws.ws)
    torch.cuda.synchronize()
    out.check_guards()
    assert (out.y.cpu().numpy() == np.float32(SENT)).all()
    ws.check()


def test_header_mismatch_sets_status_and_leaves_y():
    bits, M, N, K = 4, 1, 256, 256
    w, s = make_weights(bits, N, K, seed=1)
    packed = woq.woq_pack_w4(to_numpy_u8(w), to_numpy_u16(s), N, K).copy()
    packed[8] = 6  # header claims int6
    wdev = torch.from_numpy(packed).to(DEV)
    x_dev = synthetic.activations(M, K, seed=2).to(DEV)
    out = Guarded(M, N)
    ws = Workspace(bits, M, N, K)
    woq.woq_w4a8_linear_bf16(wdev, x_dev, N, K, out.y, ws.ws)
    torch.cuda.synchronize()
    assert woq.woq_read_status(ws.ws, clear=True) & woq.WOQ_DEVERR_HEADER
    assert woq.woq_read_status(ws.ws) == 0
    assert (out.numpy() == np.float32(SENT)).all()
    out.check_guards()


def test_empty_and_degenerate_shapes():
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    y = torch.full((2, 5), 3.0, device=DEV)
    wdev = torch.from_numpy(woq.woq_pack_w4(np.zeros((5, 0), np.uint8), np.zeros((5, 0), np.uint16), 5, 0)).to(DEV)
    x = torch.zeros((2, 0), dtype=torch.bfloat16, device=DEV)
    woq.lib.woq_w4a8_linear_bf16(wdev.data_ptr(), wdev.numel(), x.data_ptr(), 2, 5, 0, y.data_ptr(), ws.data_ptr(),
                                 256, None)
    torch.cuda.synchronize()
    assert not y.cpu().numpy().any()  # K = 0: empty sums
    y0 = torch.full((1, 8), 7.0, device=DEV)
    assert woq.lib.woq_w4a8_linear_bf16(None, 0, None, 0, 8, 128, y0.data_ptr(), None, 0, None) == 0
    torch.cuda.synchronize()
    assert (y0.cpu().numpy() == 7.0).all()
    # zero weights give exactly +0, with either int4 consumer
    N, K, M = 200, 256, 2
    packed = woq.woq_pack_w4(np.zeros((N, K // 2), np.uint8), np.full((N, 2), 0x3C00, np.uint16), N, K)
    x = synthetic.activations(M, K, seed=9).to(DEV)
    for path in (DP4A, MMA):
        woq.woq_tune_path(path)
        try:
            y = run_linear(4, torch.from_numpy(packed).to(DEV), x, N, K, M)
        finally:
            woq.woq_tune_path(0)
        assert not y.any() and not np.signbit(y).any()


@pytest.mark.parametrize("path", [DP4A, MMA])
def test_cuda_graph_replay_matches_eager(path, consumer):
    consumer(path)
    bits, M, N, K = 4, 1, 4096, 4096
    w, s = make_weights(bits, N, K, seed=31)
    wdev = pack_host(bits, to_numpy_u8(w), to_numpy_u16(s), N, K)
    x_dev = synthetic.activations(M, K, seed=32).to(DEV)
    eager = run_linear(bits, wdev, x_dev, N, K, M)
    ws = Workspace(bits, M, N, K)
    y = torch.zeros((M, N), dtype=torch.float32, device=DEV)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        woq.woq_w4a8_linear_bf16(wdev, x_dev, N, K, y, ws.ws)  # warm-up outside capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(3):
            woq.woq_w4a8_linear_bf16(wdev, x_dev, N, K, y, ws.ws)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint32), eager.view(np.uint32))
    ws.check()


# --------------------------------------------------------------------------- full sizes, sampled rows

def _sampled_rows(N, n_rand, seed):
    rng = np.random.default_rng(seed)
    rows = set([0, 1, 127, 128, N - 1, N - 2]) | set(rng.integers(0, N, size=n_rand).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < N))


@pytest.mark.parametrize("bits,M,K,N,fused,path", [
    (4, 1, 5120, 152064, True, DP4A),   # 27B LM head, decode
    (4, 1, 5120, 152064, True, MMA),
    (4, 4, 17408, 5120, True, MMA),     # 27B down projection, MTP verification rows
    (4, 4, 17408, 5120, True, DP4A),
    (4, 3, 5120, 34816, False, MMA),    # 27B gate+up, int8 entry
    (4, 2, 17408, 5120, False, MMA),    # 27B down, int8 entry (padded activation rows)
    (6, 4, 4096, 24576, True, DP4A),    # 9B gate+up in W6
    (6, 2, 12288, 4096, True, DP4A),    # 9B down in W6
])
def test_full_size_sampled_rows(bits, M, K, N, fused, path, consumer):
    consumer(path)
    seed = 100 + bits + M
    w, s = make_weights(bits, N, K, seed, device=DEV)
    wdev = torch.empty(woq.woq_packed_bytes(bits, N, K), dtype=torch.uint8, device=DEV)
    woq.woq_pack_device(bits, w, s.view(torch.int16), N, K, wdev)
    x = synthetic.activations(M, K, seed=seed + 1, outliers=True)
    xn = to_numpy_u16(x)
    x_dev = x.to(DEV)
    if fused:
        y = run_linear(bits, wdev, x_dev, N, K, M)
    else:
        q_ref, s_ref = oracle.act_quant(xn)
        y = run_gemv(bits, wdev, torch.from_numpy(q_ref).to(DEV), torch.from_numpy(s_ref).to(DEV), N, K, M)
    rows = _sampled_rows(N, 48, seed)
    idx = torch.from_numpy(rows).to(DEV)
    wn = to_numpy_u8(w.index_select(0, idx))
    sn = to_numpy_u16(s.index_select(0, idx))
    y_ref, S = oracle.linear_bf16(bits, wn, sn, len(rows), K, xn)
    ok, worst = tol_ok(y[:, rows], y_ref, S)
    assert ok, f"max err / tolerance = {worst}"
