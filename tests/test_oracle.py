"""Pins for the CPU oracle: it is checked against facts fixed outside itself.

* a hand-derived worked example (tests/golden/worked_example.txt);
* the IEEE fp16 / bf16 decoders over all 65,536 bit patterns against torch;
* every int4 / int6 code;
* round half to even at every half-integer quotient (closed form: Python round);
* fp64 dequantise-then-matmul brute force on tiny random shapes, starting
  from known integer weights encoded by the test's own encoder;
* invariants: max |q| = 127, odd symmetry, power-of-two scaling, zero
  weights give zero, doubling the scales doubles y, int4 weights written in
  the int6 format give the same result.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import bf16_bits, bf16_values, encode_w4, encode_w6, f16_bits, f16_values, read_golden


# --------------------------------------------------------------------------
# worked example
# --------------------------------------------------------------------------

def _example_arrays(g, fmt):
    K = int(g["K"])
    M, N = 2, 2
    x = np.zeros((M, K), dtype=np.float64)
    for m in range(M):
        v = [float(t) for t in g[("x", m)]]
        x[m, : len(v)] = v
    wvals = np.zeros((N, K), dtype=np.int64)
    for n in range(N):
        v = [int(t) for t in g[(fmt, n)]]
        wvals[n, : len(v)] = v
    nb = K // 2 if fmt == "w4" else K // 4 * 3
    wbytes = np.zeros((N, nb), dtype=np.uint8)
    for n in range(N):
        b = [int(t, 16) for t in g[(fmt + "bytes", n)]]
        wbytes[n, : len(b)] = b
    scales = np.array([[float(g[(fmt + "scale", n)][0])] for n in range(N)])
    return K, x, wvals, wbytes, scales


@pytest.mark.parametrize("fmt,bits", [("w4", 4), ("w6", 6)])
def test_worked_example(fmt, bits):
    g = read_golden("worked_example.txt")
    K, x, wvals, wbytes, scales = _example_arrays(g, fmt)
    xb = bf16_bits(x)
    assert np.array_equal(bf16_values(xb), x), "example activations must be exact in bf16"
    # the hand-packed bytes decode to the listed weights
    assert np.array_equal(oracle.unpack_weights(bits, wbytes, 2, K), wvals.astype(np.int8))
    # and the test's encoder produces the same bytes
    enc = encode_w4(wvals) if bits == 4 else encode_w6(wvals)
    assert np.array_equal(enc, wbytes)
    q, s = oracle.act_quant(xb)
    for m in range(2):
        exp_q = [int(t) for t in g[("q", m)]]
        assert q[m, : len(exp_q)].tolist() == exp_q
        assert not q[m, len(exp_q):].any()
        assert s[m] == np.float32(float(g[("ascale", m)][0]))
    sb = f16_bits(scales)
    d = oracle.group_dots(bits, wbytes, 2, K, q)
    y, S = oracle.gemv(bits, wbytes, sb, 2, K, q, s)
    y2, S2 = oracle.linear_bf16(bits, wbytes, sb, 2, K, xb)
    for m in range(2):
        assert d[m, :, 0].tolist() == [int(t) for t in g[(fmt + "dots", m)]]
        assert y[m].tolist() == [float(t) for t in g[(fmt + "y", m)]]
    assert np.array_equal(y, y2) and np.array_equal(S, S2)
    assert np.array_equal(S, np.abs(y).astype(np.float64))  # one group: S = |term| = |y|


# --------------------------------------------------------------------------
# exhaustive small domains
# --------------------------------------------------------------------------

def test_f16_decoder_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = f16_values(bits)
    got = np.array([oracle.f16_to_f32(b) for b in bits.tolist()], dtype=np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # the sign of zero survives
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_decoder_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bf16_values(bits)
    got = np.array([oracle.bf16_to_f32(b) for b in bits.tolist()], dtype=np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_int4_every_code():
    K = 128
    for code in range(16):
        expected = code - 16 if code >= 8 else code
        row = np.zeros((1, K // 2), dtype=np.uint8)
        row[0, 3] = code | (((code + 5) % 16) << 4)  # k = 6 (low), k = 7 (high)
        vals = oracle.unpack_weights(4, row, 1, K)
        hi = (code + 5) % 16
        assert vals[0, 6] == expected
        assert vals[0, 7] == (hi - 16 if hi >= 8 else hi)
        assert np.count_nonzero(vals) == (expected != 0) + (hi != 0)


def test_int6_every_code_every_slot():
    K = 128
    for slot in range(4):
        for code in range(64):
            expected = code - 64 if code >= 32 else code
            word = code << (6 * slot)
            row = np.zeros((1, K // 4 * 3), dtype=np.uint8)
            row[0, 6:9] = [word & 0xFF, (word >> 8) & 0xFF, (word >> 16) & 0xFF]  # k = 8 .. 11
            vals = oracle.unpack_weights(6, row, 1, K)
            assert vals[0, 8 + slot] == expected
            assert np.count_nonzero(vals) == (expected != 0)


# --------------------------------------------------------------------------
# activation quantisation
# --------------------------------------------------------------------------

def test_round_half_even_at_every_half_integer():
    # amax = 127 gives a scale of exactly 1, so x / scale = x and the rounding is visible
    halves = np.arange(-127, 127, dtype=np.float64) + 0.5  # -126.5 .. 126.5
    x = np.concatenate([[127.0], halves])[None, :]
    xb = bf16_bits(x)
    assert np.array_equal(bf16_values(xb), x)
    q, s = oracle.act_quant(xb)
    assert s[0] == np.float32(1.0)
    assert q[0, 0] == 127
    expected = [round(v) for v in halves.tolist()]  # Python rounds ties to even
    assert q[0, 1:].tolist() == expected


def test_act_quant_invariants():
    gen = torch.Generator().manual_seed(123)
    M, K = 4, 1000
    x = torch.randn(M, K, generator=gen, dtype=torch.float64) * torch.tensor([[1.0], [1e-3], [40.0], [3.0]])
    x[3, 17] = 200.0  # an outlier dominates row 3
    xb = bf16_bits(x.numpy())
    q, s = oracle.act_quant(xb)
    assert np.abs(q.astype(np.int32)).max() <= 127
    assert (np.abs(q.astype(np.int32)).max(axis=1) == 127).all()
    # odd symmetry: x -> -x flips q, keeps the scale
    qn, sn = oracle.act_quant(xb ^ np.uint16(0x8000))
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)
    # scaling by a power of two leaves q and scales the scale exactly
    for j in (-3, 5):
        xs = bf16_bits(bf16_values(xb) * 2.0 ** j)
        assert np.array_equal(bf16_values(xs), bf16_values(xb) * 2.0 ** j)
        q2, s2 = oracle.act_quant(xs)
        assert np.array_equal(q2, q)
        assert np.array_equal(s2.astype(np.float64), s.astype(np.float64) * 2.0 ** j)
    # quantisation error: |q * scale - x| <= scale / 2 (plus fp32 slack)
    xv = bf16_values(xb)
    err = np.abs(q.astype(np.float64) * s[:, None].astype(np.float64) - xv)
    assert (err <= s[:, None] * (0.5 + 1e-5)).all()
    # the scale is amax / 127 to within one fp32 ulp of the exact quotient
    amax = np.abs(xv).max(axis=1)
    assert np.allclose(s.astype(np.float64), amax / 127.0, rtol=2 ** -23, atol=0)


def test_act_quant_matches_numpy_ieee_division():
    # library check: numpy float32 division is IEEE, np.rint rounds ties to even
    gen = torch.Generator().manual_seed(7)
    x = torch.randn(3, 4096, generator=gen, dtype=torch.float64) * 7.3
    xb = bf16_bits(x.numpy())
    q, s = oracle.act_quant(xb)
    xv = bf16_values(xb).astype(np.float32)
    amax = np.abs(xv).max(axis=1)
    s_ref = amax / np.float32(127.0)
    assert np.array_equal(s, s_ref)
    q_ref = np.clip(np.rint(xv / s_ref[:, None]), -127, 127).astype(np.int8)
    assert np.array_equal(q, q_ref)


def test_zero_row_and_nonfinite():
    x = np.zeros((2, 256), dtype=np.float64)
    x[1, 5] = 3.0
    q, s = oracle.act_quant(bf16_bits(x))
    assert s[0] == 0.0 and not q[0].any()
    assert s[1] == np.float32(3.0) / np.float32(127.0) and q[1, 5] == 127
    for bad in (np.inf, -np.inf, np.nan):
        xb = bf16_bits(x)
        xb[1, 7] = bf16_bits([bad])[0]
        with pytest.raises(oracle.OracleError):
            oracle.act_quant(xb)


# --------------------------------------------------------------------------
# brute force: fp64 dequantise-then-matmul on tiny shapes
# --------------------------------------------------------------------------

def _random_case(rng, bits, M, N, K):
    lo, hi = (-8, 7) if bits == 4 else (-32, 31)
    wv = rng.integers(lo, hi + 1, size=(N, K))
    wb = encode_w4(wv) if bits == 4 else encode_w6(wv)
    sb = f16_bits(np.abs(rng.standard_normal((N, K // 128))) * 0.02 + 1e-3)
    q = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    s = (np.abs(rng.standard_normal(M)) * 0.05 + 1e-4).astype(np.float32)
    return wv, wb, sb, q, s


@pytest.mark.parametrize("bits", [4, 6])
def test_brute_force_tiny_shapes(bits):
    rng = np.random.default_rng(2024 + bits)
    for M, N, K in [(1, 1, 128), (2, 3, 256), (3, 17, 384), (4, 33, 512), (4, 8, 128), (1, 31, 640)]:
        wv, wb, sb, q, s = _random_case(rng, bits, M, N, K)
        assert np.array_equal(oracle.unpack_weights(bits, wb, N, K), wv.astype(np.int8))
        # exact integer group dots
        d = oracle.group_dots(bits, wb, N, K, q)
        G = K // 128
        d_ref = np.einsum("ngk,mgk->mng", wv.reshape(N, G, 128).astype(np.int64),
                          q.astype(np.int64).reshape(M, G, 128))
        assert np.array_equal(d.astype(np.int64), d_ref)
        # fp64 dequantise then matmul: W = q_w * ws, A = q_a * as
        ws = f16_values(sb)  # [N, G]
        Wd = wv.astype(np.float64) * np.repeat(ws, 128, axis=1)
        Ad = q.astype(np.float64) * s.astype(np.float64)[:, None]
        y_ref = Ad @ Wd.T
        y, S = oracle.gemv(bits, wb, sb, N, K, q, s)
        # each fp32 term carries two roundings, the fp64 sum one final fp32 rounding
        bound = 3e-7 * S + 6e-8 * np.abs(y_ref) + 1e-37
        assert (np.abs(y.astype(np.float64) - y_ref) <= bound).all()
        terms = np.abs(d_ref.astype(np.float64) * ws[None, :, :] * s.astype(np.float64)[:, None, None]).sum(-1)
        assert np.allclose(S, terms, rtol=3e-7, atol=0)


# --------------------------------------------------------------------------
# invariants of the linear
# --------------------------------------------------------------------------

def test_linear_invariants():
    rng = np.random.default_rng(99)
    M, N, K = 3, 20, 384
    wv, wb, sb, q, s = _random_case(rng, 4, M, N, K)
    y, S = oracle.gemv(4, wb, sb, N, K, q, s)
    # zero weights -> +0 everywhere
    yz, Sz = oracle.gemv(4, np.zeros_like(wb), sb, N, K, q, s)
    assert not yz.any() and not np.signbit(yz).any() and not Sz.any()
    # doubling every scale doubles y exactly
    sb2 = f16_bits(f16_values(sb) * 2.0)
    y2, _ = oracle.gemv(4, wb, sb2, N, K, q, s)
    assert np.array_equal(y2.astype(np.float64), 2.0 * y.astype(np.float64))
    # the same integer weights in the int6 format give identical dots and outputs
    wb6 = encode_w6(wv)
    assert np.array_equal(oracle.group_dots(4, wb, N, K, q), oracle.group_dots(6, wb6, N, K, q))
    y6, S6 = oracle.gemv(6, wb6, sb, N, K, q, s)
    assert np.array_equal(y6, y) and np.array_equal(S6, S)
    # negating the activation negates y exactly
    yn, _ = oracle.gemv(4, wb, sb, N, K, (-q.astype(np.int16)).astype(np.int8), s)
    assert np.array_equal(yn, -y)
    # S bounds |y|
    assert (np.abs(y) <= S * (1 + 1e-6) + 1e-30).all()


def test_shape_errors():
    wb = np.zeros((2, 64), dtype=np.uint8)
    sb = np.zeros((2, 1), dtype=np.uint16)
    q = np.zeros((1, 100), dtype=np.int8)
    with pytest.raises(oracle.OracleError):
        oracle.gemv(4, wb, sb, 2, 100, q, np.zeros(1, np.float32))
    with pytest.raises(oracle.OracleError):
        oracle.gemv(5, wb, sb, 2, 128, np.zeros((1, 128), np.int8), np.zeros(1, np.float32))


def test_empty_shapes():
    q, s = oracle.act_quant(np.zeros((0, 128), dtype=np.uint16))
    assert q.shape == (0, 128) and s.shape == (0,)
    y, S = oracle.gemv(4, np.zeros((0, 64), np.uint8), np.zeros((0, 1), np.uint16), 0, 128,
                       np.zeros((2, 128), np.int8), np.ones(2, np.float32))
    assert y.shape == (2, 0)
    # K = 0: no groups, y = 0
    y, S = oracle.gemv(4, np.zeros((3, 0), np.uint8), np.zeros((3, 0), np.uint16), 3, 0,
                       np.zeros((1, 0), np.int8), np.ones(1, np.float32))
    assert y.shape == (1, 3) and not y.any()


# --------------------------------------------------------------------------- prologue fusions (R11 - R13)

def _bf16_bits(t):
    import torch
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bf16_value(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_f32_to_bf16_is_round_to_nearest_even():
    import torch
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    # exact ties: low 16 bits 0x8000 with even and odd kept parts
    ties = (np.arange(2000, dtype=np.uint32) * 0x10000 + 0x3F808000).view(np.float32)
    for x in np.concatenate([v, ties]):
        assert oracle.f32_to_bf16(float(x)) == int(_bf16_bits(torch.tensor([x]))[0])


def test_exp_cw_within_two_ulp_of_exp():
    import math
    xs = np.concatenate([np.linspace(-86.9, 88.6, 40001, dtype=np.float32),
                         np.float32([0.0, 1e-8, -1e-8, 0.5, -0.5, 0.6931472, -0.6931472])])
    worst = 0.0
    for x in xs:
        e = oracle.exp_cw(float(x))
        ref = math.exp(float(x))
        ulp = float(np.spacing(np.float32(ref)))  # fp32 spacing at the result
        worst = max(worst, abs(e - ref) / ulp)
    assert worst <= 2.0, worst
    assert oracle.exp_cw(0.0) == 1.0
    assert oracle.exp_cw(88.72) == float("inf") and oracle.exp_cw(-87.0) == 0.0


def test_swiglu_matches_fp64_within_one_bf16_step():
    rng = np.random.default_rng(5)
    M, K = 3, 2048
    gu = (rng.standard_normal((M, 2 * K)) * 3).astype(np.float32)
    gu[0, :8] = [0.0, -0.0, 50.0, -50.0, 100.0, -100.0, 1e-30, -1e-30]
    h = oracle.swiglu(gu)
    g = gu[:, :K].astype(np.float64)
    u = gu[:, K:].astype(np.float64)
    ref = g / (1.0 + np.exp(-g)) * u
    hv = _bf16_value(h)
    step = np.maximum(np.abs(ref), 1e-38) * 2.0 ** -7  # one bf16 step at the value
    assert (np.abs(hv - ref) <= step).all()
    assert hv[0, 0] == 0 and hv[0, 5] == 0  # silu(0) = 0, silu(-100) = -0
    assert abs(hv[0, 4] - 100.0 * u[0, 4]) <= abs(100.0 * u[0, 4]) * 2.0 ** -8


def test_rmsnorm_matches_fp64_and_its_invariants():
    import torch
    rng = np.random.default_rng(6)
    M, K = 4, 5120
    x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32))
    x[:, ::97] *= 20.0
    xb = _bf16_bits(x)
    gamma = _bf16_bits(torch.from_numpy((1.0 + 0.1 * rng.standard_normal(K)).astype(np.float32)))
    eps = 1e-6
    h = oracle.rmsnorm(xb, gamma, eps)
    xv, gv = _bf16_value(xb), _bf16_value(gamma)
    ref = xv / np.sqrt((xv ** 2).mean(axis=1, keepdims=True) + eps) * gv
    assert (np.abs(_bf16_value(h) - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30).all()
    # scaling x by a power of two leaves h unchanged (eps = 0): the squares are exact
    h0 = oracle.rmsnorm(xb, gamma, 0.0)
    for j in (-9, 3, 11):
        xs = _bf16_bits(torch.from_numpy((xv * 2.0 ** j).astype(np.float32)))
        assert np.array_equal(oracle.rmsnorm(xs, gamma, 0.0), h0)
    # all-zero row gives zeros; a constant row with gamma = 1 gives +-1
    z = np.zeros((1, 256), np.uint16)
    assert not oracle.rmsnorm(z, np.full(256, 0x3F80, np.uint16), 1e-6).any()
    c = np.full((1, 256), 0xC040, np.uint16)  # -3.0
    assert (oracle.rmsnorm(c, np.full(256, 0x3F80, np.uint16), 0.0) == 0xBF80).all()  # -1.0


def test_rmsnorm_eps_enters_under_the_square_root():
    """eps is added to the mean of squares, under the square root, and nowhere else.
    Rows of +-1 have mean of squares exactly 1: eps = 3 gives r = 1/sqrt(4) = 1/2 exactly, so
    h = +-gamma / 2 (a dropped eps gives +-gamma, an eps added after the square root
    +-gamma / 4).  The same at another scale: x = +-2^-10 (mean 2^-20) with eps = 3 2^-20 gives
    r = 2^9 and h = +-gamma / 2 again.  eps = 1 gives h within one bf16 step of
    +-gamma / sqrt(2)."""
    import torch
    rng = np.random.default_rng(8)
    M, K = 3, 1024
    sign = rng.random((M, K)) < 0.5
    gv = (1.0 + rng.standard_normal(K)).astype(np.float32)
    gamma = _bf16_bits(torch.from_numpy(gv))
    gval = _bf16_value(gamma)
    for xmag, eps, factor in [(1.0, 3.0, 0.5), (2.0 ** -10, 3.0 * 2.0 ** -20, 0.5), (1.0, 0.0, 1.0)]:
        x = _bf16_bits(torch.from_numpy(np.where(sign, -xmag, xmag).astype(np.float32)))
        h = _bf16_value(oracle.rmsnorm(x, gamma, eps))
        assert np.array_equal(h, np.where(sign, -1.0, 1.0) * gval * factor), (xmag, eps)
    x = _bf16_bits(torch.from_numpy(np.where(sign, -1.0, 1.0).astype(np.float32)))
    ref = np.where(sign, -1.0, 1.0) * gval / np.sqrt(2.0)
    h = _bf16_value(oracle.rmsnorm(x, gamma, 1.0))
    assert (np.abs(h - ref) <= np.abs(ref) * 2.0 ** -7).all()


def test_rmsnorm_matches_fp64_where_eps_is_large():
    """Small activations (mean of squares about 1e-4) with eps from 1e-5 to 1e-2: eps changes r
    by up to a factor of ten, and h stays within one bf16 step of the fp64 RMSNorm."""
    import torch
    rng = np.random.default_rng(9)
    M, K = 4, 4096
    x = torch.from_numpy((rng.standard_normal((M, K)) * 0.01).astype(np.float32))
    xb = _bf16_bits(x)
    gamma = _bf16_bits(torch.from_numpy((1.0 + 0.1 * rng.standard_normal(K)).astype(np.float32)))
    xv, gv = _bf16_value(xb), _bf16_value(gamma)
    for eps in (1e-5, 1e-4, 1e-3, 1e-2):
        e32 = float(np.float32(eps))
        ref = xv / np.sqrt((xv ** 2).mean(axis=1, keepdims=True) + e32) * gv
        h = _bf16_value(oracle.rmsnorm(xb, gamma, eps))
        assert (np.abs(h - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30).all(), eps


def test_fused_linear_oracles_compose_the_steps():
    rng = np.random.default_rng(7)
    N, K, M = 64, 256, 2
    wv = rng.integers(-8, 8, size=(N, K))
    w = encode_w4(wv)
    s = (np.abs(rng.standard_normal((N, K // 128))) * 0.02 + 1e-3).astype(np.float16).view(np.uint16)
    gu = rng.standard_normal((M, 2 * K)).astype(np.float32)
    y, S = oracle.linear_swiglu(4, w, s, N, K, gu)
    y2, _ = oracle.linear_bf16(4, w, s, N, K, oracle.swiglu(gu))
    assert np.array_equal(y, y2)
    x = rng.integers(0, 1 << 16, size=(M, K), dtype=np.uint16) & 0xBFFF  # finite values
    g = np.full(K, 0x3F80, np.uint16)
    y3, _ = oracle.linear_rmsnorm(4, w, s, N, K, x, g, 1e-5)
    y4, _ = oracle.linear_bf16(4, w, s, N, K, oracle.rmsnorm(x, g, 1e-5))
    assert np.array_equal(y3, y4)
