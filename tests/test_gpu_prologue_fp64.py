"""The RMSNorm and SwiGLU prologues on the GPU against a plain fp64 restatement.

"Optimizing the Linear Kernel" folds the RMSNorm (or the SwiGLU) before a linear into its
input quantisation.  The oracle's RMSNorm and SwiGLU follow the kernels' own fp32 recipe
operation for operation, so here the kernels are also checked against the textbook
definitions computed in fp64, independently of that recipe:

    RMSNorm  h = x gamma / sqrt(mean(x^2) + eps)        SwiGLU  h = g u / (1 + e^-g)

h64 is rounded to bf16 (round half to even, on the fp64 value) and quantised as the oracle
quantises a bf16 row (scale = fp32(amax) / 127, q = rne(fp32 h / scale)).  The kernels'
fp32 recipe is within a relative error bound of h64 (derived below); where h64 lies that
close to a bf16 rounding boundary, the kernel may round to either neighbour, so q there may
be either neighbour's quotient; everywhere else q must match exactly, and the row scale must
be the scale of one of the possible row maxima.  The twins (woq_rmsnorm_act_quant_int8,
woq_swiglu_act_quant_int8) are compared; the fused linears are bit-identical to twin +
GEMV (test_gpu_prologue.py).

Error bounds (u = 2^-24, relative):
  RMSNorm: the mean of squares is summed at a fixed point that drops less than 2^-30 of the
    largest square per term (at most K 2^-30 max(x^2) / sum(x^2) in all), then RN(S), / K,
    + eps, sqrt, 1 /, x r, * gamma: at most that / 2 + 6 u; the test allows twice.
  SwiGLU: e^-g within 2 fp32 ulps (4 u), then 1 + e, 1 /, g sg, * u: at most 8 u; allowed 16 u.
"""
import numpy as np
import pytest
import torch

import synthetic
from synthetic import to_numpy_u16

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
U = 2.0 ** -24
woq = None


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    global woq
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import weight_only_quantised_gb300 as w
    woq = w
    torch.cuda.set_device(0)
    yield


def _bf16_f64(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_candidates(h64, rel_margin):
    """Round fp64 values to bf16 (half to even, on the fp64 value; normal range) and give the
    two neighbours around each value that lies within rel_margin |h| of a rounding boundary.
    Returns (ref, alt, ambiguous) as float64 arrays: alt = the other neighbour where ambiguous,
    else ref."""
    m, e = np.frexp(h64)  # h = m 2^e, 0.5 <= |m| < 1
    a = np.abs(m) * 256.0  # 8 significant bits: bf16 keeps floor or ceil of a
    sign = np.sign(m)
    ref = sign * np.ldexp(np.rint(a), e - 8)
    fl = np.floor(a)
    amb = (np.abs(a - fl - 0.5) <= rel_margin[..., None] * a if np.ndim(rel_margin) else
           np.abs(a - fl - 0.5) <= rel_margin * a) & (h64 != 0)
    other = np.where(np.rint(a) == fl, fl + 1.0, fl)
    alt = np.where(amb, sign * np.ldexp(other, e - 8), ref)
    return ref, alt, amb


def _rne_q(h, s):
    """The oracle's quantisation of bf16 values h (float64 holding bf16-exact values) by the
    fp32 scale s: q = rne(fp32(h) / s) (IEEE fp32 division), clamped to [-127, 127]."""
    t = np.float32(h) / np.float32(s) if np.ndim(h) == 0 else h.astype(np.float32) / np.float32(s)
    return np.clip(np.rint(t), -127, 127).astype(np.int64)


def _check_rows(q_k, s_k, ref, alt, amb):
    """q_k, s_k from the kernel; ref / alt / amb from _bf16_candidates, per row."""
    M = ref.shape[0]
    n_amb = 0
    for m in range(M):
        lo_mag = np.minimum(np.abs(ref[m]), np.abs(alt[m]))
        hi_mag = np.maximum(np.abs(ref[m]), np.abs(alt[m]))
        amax_lo, amax_hi = lo_mag.max(), hi_mag.max()
        cands = np.unique(np.concatenate([lo_mag, hi_mag]))
        cands = cands[(cands >= amax_lo) & (cands <= amax_hi)]
        scales = {np.float32(c) / np.float32(127): c for c in cands}
        s = np.float32(s_k[m])
        assert s in scales, f"row {m}: scale {s} is none of {sorted(scales)}"
        q_ref = _rne_q(ref[m], s)
        q_alt = _rne_q(alt[m], s)
        qk = q_k[m].astype(np.int64)
        assert ((qk == q_ref) | (amb[m] & (qk == q_alt))).all(), f"row {m}: q differs where h64 is unambiguous"
        n_amb += int(amb[m].sum())
    return n_amb


@pytest.mark.parametrize("M", [1, 3, 4])
@pytest.mark.parametrize("K", [1024, 5120, 17408])
@pytest.mark.parametrize("eps,xscale", [(1e-6, 1.0), (0.5, 0.3), (1e-2, 0.05)])
def test_rmsnorm_twin_against_fp64(M, K, eps, xscale):
    x = synthetic.activations(M, K, seed=M * 31 + K, outliers=True) * xscale
    xn = to_numpy_u16(x.to(torch.bfloat16))
    gn = to_numpy_u16(synthetic.rmsnorm_weight(K, K + M))
    xv, gv = _bf16_f64(xn), _bf16_f64(gn)
    e32 = float(np.float32(eps))
    ms = (xv ** 2).mean(axis=1, keepdims=True)
    h64 = xv * gv / np.sqrt(ms + e32)
    trunc = K * 2.0 ** -30 * (xv ** 2).max(axis=1) / (xv ** 2).sum(axis=1)
    ref, alt, amb = _bf16_candidates(h64, 2 * (trunc / 2 + 6 * U))
    q = torch.full((M, K), 99, dtype=torch.int8, device=DEV)
    s = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    woq.woq_rmsnorm_act_quant_int8(torch.from_numpy(xn.view(np.int16)).to(DEV).view(torch.bfloat16),
                                   torch.from_numpy(gn.view(np.int16)).to(DEV).view(torch.bfloat16), eps, q, s)
    torch.cuda.synchronize()
    n_amb = _check_rows(q.cpu().numpy(), s.cpu().numpy(), ref, alt, amb)
    assert n_amb <= 0.01 * M * K  # the bound leaves almost every value decided


@pytest.mark.parametrize("M", [1, 4, 8])
@pytest.mark.parametrize("K", [1024, 5120, 17408])
def test_swiglu_twin_against_fp64(M, K):
    gu = synthetic.gate_up_output(M, K, seed=M * 37 + K).numpy().astype(np.float32)
    g, u = gu[:, :K].astype(np.float64), gu[:, K:].astype(np.float64)
    h64 = g * u / (1.0 + np.exp(-g))
    ref, alt, amb = _bf16_candidates(h64, 16 * U)
    q = torch.full((M, K), 99, dtype=torch.int8, device=DEV)
    s = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    woq.woq_swiglu_act_quant_int8(torch.from_numpy(gu).to(DEV), q, s)
    torch.cuda.synchronize()
    n_amb = _check_rows(q.cpu().numpy(), s.cpu().numpy(), ref, alt, amb)
    assert n_amb <= 0.01 * M * K


def test_candidate_rounding_is_round_half_even_on_fp64():
    """The helper's bf16 rounding of fp64 values (no GPU involved): exact bf16 values stay, a
    value just above a midpoint rounds up, an exact midpoint goes to the even neighbour."""
    one_ulp = 2.0 ** -7  # bf16 spacing in [1, 2)
    v = np.array([1.0, 1.0 + one_ulp, 1.0 + 0.5 * one_ulp, 1.0 + 1.5 * one_ulp, 1.0 + 0.5 * one_ulp + 1e-12,
                  -(1.0 + 1.5 * one_ulp)])
    ref, alt, amb = _bf16_candidates(v, 1e-9)
    assert list(ref) == [1.0, 1.0 + one_ulp, 1.0, 1.0 + 2 * one_ulp, 1.0 + one_ulp, -(1.0 + 2 * one_ulp)]
    assert list(amb) == [False, False, True, True, True, True]
    assert alt[2] == 1.0 + one_ulp and alt[3] == 1.0 + one_ulp and alt[4] == 1.0
