"""CPU oracle for the weight-only-quantised skinny linear (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It compiles ``oracle.c`` (plain C11,
no fast-math, no FP contraction) with gcc into ``oracle/_build/liboracle.so``
and wraps its entry points for numpy arrays.  It never imports the CUDA
library and shares no code with it.

Every function restates "Doubling LLM token rates in ComfyUI" (blog.comfy.org),
sections "What is the bottleneck?" and "Optimizing the Linear Kernel"; the
readings the pages leave open are listed at the top of ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_SHAPE = 1
ERR_NONFINITE = 2
ERR_RANGE = 3
ERR_BITS = 4


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile oracle.c if the shared object is missing or older than the source."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f32.restype = ctypes.c_float
            lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f32.restype = ctypes.c_float
            lib.oracle_w4_at.argtypes = [P, I, I, I]
            lib.oracle_w4_at.restype = I
            lib.oracle_w6_at.argtypes = [P, I, I, I]
            lib.oracle_w6_at.restype = I
            lib.oracle_unpack_weights.argtypes = [I, P, I, I, P]
            lib.oracle_unpack_weights.restype = I
            lib.oracle_act_quant.argtypes = [P, I, I, P, P]
            lib.oracle_act_quant.restype = I
            lib.oracle_group_dots.argtypes = [I, P, I, I, P, I, P]
            lib.oracle_group_dots.restype = I
            lib.oracle_gemv.argtypes = [I, P, P, I, I, P, P, I, P, P]
            lib.oracle_gemv.restype = I
            lib.oracle_linear_bf16.argtypes = [I, P, P, I, I, P, I, P, P]
            lib.oracle_linear_bf16.restype = I
            lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
            lib.oracle_exp_cw.argtypes = [ctypes.c_float]
            lib.oracle_exp_cw.restype = ctypes.c_float
            lib.oracle_rmsnorm_bf16.argtypes = [P, P, ctypes.c_float, I, I, P]
            lib.oracle_rmsnorm_bf16.restype = I
            lib.oracle_swiglu_bf16.argtypes = [P, I, I, P]
            lib.oracle_swiglu_bf16.restype = I
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _check(rc: int, what: str):
    if rc != OK:
        raise OracleError(f"{what}: oracle status {rc}")


def f16_to_f32(bits: int) -> float:
    """IEEE binary16 bit pattern -> value (as fp32)."""
    return float(_load().oracle_f16_to_f32(int(bits)))


def bf16_to_f32(bits: int) -> float:
    """bfloat16 bit pattern -> value (as fp32)."""
    return float(_load().oracle_bf16_to_f32(int(bits)))


def unpack_weights(bits: int, w: np.ndarray, N: int, K: int) -> np.ndarray:
    """Canonical int4/int6 bytes -> int8 [N, K] weight values."""
    w = _c(w, np.uint8)
    out = np.zeros((N, K), dtype=np.int8)
    _check(_load().oracle_unpack_weights(bits, _ptr(w), N, K, _ptr(out)), "unpack_weights")
    return out


def act_quant(x_bf16: np.ndarray):
    """bf16 bit patterns [M, K] (uint16) -> (q int8 [M, K], ascale fp32 [M])."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    q = np.zeros((M, K), dtype=np.int8)
    s = np.zeros((M,), dtype=np.float32)
    _check(_load().oracle_act_quant(_ptr(x), M, K, _ptr(q), _ptr(s)), "act_quant")
    return q, s


def group_dots(bits: int, w: np.ndarray, N: int, K: int, q: np.ndarray) -> np.ndarray:
    """Exact per-group dot products, int32 [M, N, K/128]."""
    w = _c(w, np.uint8)
    q = _c(q, np.int8)
    M = q.shape[0]
    out = np.zeros((M, N, K // 128), dtype=np.int32)
    _check(_load().oracle_group_dots(bits, _ptr(w), N, K, _ptr(q), M, _ptr(out)), "group_dots")
    return out


def gemv(bits: int, w: np.ndarray, wscale_f16: np.ndarray, N: int, K: int, q: np.ndarray, ascale: np.ndarray):
    """y fp32 [M, N] and S = sum_g |term_g| fp64 [M, N] from int8 activations."""
    w = _c(w, np.uint8)
    ws = _c(wscale_f16, np.uint16)
    q = _c(q, np.int8)
    a = _c(ascale, np.float32)
    M = q.shape[0]
    y = np.zeros((M, N), dtype=np.float32)
    S = np.zeros((M, N), dtype=np.float64)
    _check(_load().oracle_gemv(bits, _ptr(w), _ptr(ws), N, K, _ptr(q), _ptr(a), M, _ptr(y), _ptr(S)), "gemv")
    return y, S


def linear_bf16(bits: int, w: np.ndarray, wscale_f16: np.ndarray, N: int, K: int, x_bf16: np.ndarray):
    """The whole op from bf16 activations: y fp32 [M, N] and S fp64 [M, N]."""
    w = _c(w, np.uint8)
    ws = _c(wscale_f16, np.uint16)
    x = _c(x_bf16, np.uint16)
    M = x.shape[0]
    y = np.zeros((M, N), dtype=np.float32)
    S = np.zeros((M, N), dtype=np.float64)
    _check(_load().oracle_linear_bf16(bits, _ptr(w), _ptr(ws), N, K, _ptr(x), M, _ptr(y), _ptr(S)), "linear_bf16")
    return y, S


def tolerance(S: np.ndarray) -> np.ndarray:
    """Allowed |y_gpu - y_ref| per element: 1e-5 * sum_g |term_g| + 1e-6."""
    return 1e-5 * np.asarray(S, dtype=np.float64) + 1e-6


# ----------------------------------------------------------------------------- prologue fusions (R11 - R13)

def f32_to_bf16(v: float) -> int:
    """fp32 -> bf16 bit pattern, round to nearest even."""
    return int(_load().oracle_f32_to_bf16(float(v)))


def exp_cw(a: float) -> float:
    """e^a in fp32 by the Cody-Waite method with a degree-7 Taylor polynomial (R12)."""
    return float(_load().oracle_exp_cw(float(a)))


def rmsnorm(x_bf16: np.ndarray, gamma_bf16: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm (R11) of bf16 rows [M, K] with bf16 weights [K] -> bf16 bit patterns [M, K]."""
    x = _c(x_bf16, np.uint16)
    g = _c(gamma_bf16, np.uint16)
    M, K = x.shape
    h = np.zeros((M, K), dtype=np.uint16)
    _check(_load().oracle_rmsnorm_bf16(_ptr(x), _ptr(g), float(eps), M, K, _ptr(h)), "rmsnorm")
    return h


def swiglu(gate_up_f32: np.ndarray) -> np.ndarray:
    """SwiGLU (R12) of fp32 rows [M, 2K] (gate, then up) -> bf16 bit patterns [M, K]."""
    gu = _c(gate_up_f32, np.float32)
    M, K2 = gu.shape
    h = np.zeros((M, K2 // 2), dtype=np.uint16)
    _check(_load().oracle_swiglu_bf16(_ptr(gu), M, K2 // 2, _ptr(h)), "swiglu")
    return h


def linear_rmsnorm(bits, w, wscale_f16, N, K, x_bf16, gamma_bf16, eps):
    """RMSNorm, act_quant and the linear (R11, R13, R5, R6): y fp32 [M, N], S fp64 [M, N]."""
    return linear_bf16(bits, w, wscale_f16, N, K, rmsnorm(x_bf16, gamma_bf16, eps))


def linear_swiglu(bits, w, wscale_f16, N, K, gate_up_f32):
    """SwiGLU, act_quant and the linear (R12, R13, R5, R6): y fp32 [M, N], S fp64 [M, N]."""
    return linear_bf16(bits, w, wscale_f16, N, K, swiglu(gate_up_f32))
