"""Python binding of libwoq.so, the weight-only-quantised skinny linear for GB300.

Argument marshalling only: every function forwards to the C ABI of the same
name declared in include/woq.h, passing raw pointers (torch tensors'
``data_ptr()`` for device buffers, numpy arrays for host buffers), sizes and the
current CUDA stream.  Every step of the computation runs in the library's CUDA
kernels; there is no Python or CPU fallback.  Importing this package loads the
in-tree ``libwoq.so`` and raises if it has not been built
(``python -m weight_only_quantised_gb300._build`` or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# WOQ_LIB selects another build of the same ABI (e.g. the trace build libwoq_trace.so)
LIB_PATH = os.environ.get("WOQ_LIB") or os.path.join(_PKG, "libwoq.so")

WOQ_OK = 0
WOQ_ERR_NULL = 1
WOQ_ERR_ALIGN = 2
WOQ_ERR_SHAPE = 3
WOQ_ERR_WORKSPACE = 4
WOQ_ERR_LAYOUT = 5
WOQ_ERR_CUDA = 6
WOQ_ERR_DEVICE = 7
WOQ_DEVERR_HEADER = 0x1
WOQ_DEVERR_TIMEOUT = 0x2
GROUP = 128
TILE_ROWS = 128

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it first (python -m weight_only_quantised_gb300._build)")

lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t
_SIGS = {
    "woq_version": ([], _I),
    "woq_status_string": ([_I], ctypes.c_char_p),
    "woq_max_m": ([], _I),
    "woq_max_k": ([_I, _I, _I], _I),
    "woq_packed_bytes": ([_I, _I, _I], _Z),
    "woq_pack_w4": ([_P, _P, _I, _I, _P, _Z], _I),
    "woq_pack_w6": ([_P, _P, _I, _I, _P, _Z], _I),
    "woq_unpack": ([_I, _P, _Z, _I, _I, _P, _P], _I),
    "woq_pack_device": ([_I, _P, _P, _I, _I, _P, _Z, _P], _I),
    "woq_relayout_inplace": ([_I, _P, _Z, _I, _I, _P], _I),
    "woq_workspace_bytes": ([_I, _I, _I, _I], _Z),
    "woq_workspace_init": ([_P, _Z, _P], _I),
    "woq_read_status": ([_P, _Z, _I, ctypes.POINTER(ctypes.c_uint32), _P], _I),
    "woq_act_quant_int8": ([_P, _I, _I, _P, _P, _P], _I),
    "woq_w4a8_gemv": ([_P, _Z, _P, _P, _I, _I, _I, _P, _P, _Z, _P], _I),
    "woq_w6a8_gemv": ([_P, _Z, _P, _P, _I, _I, _I, _P, _P, _Z, _P], _I),
    "woq_w4a8_linear_bf16": ([_P, _Z, _P, _I, _I, _I, _P, _P, _Z, _P], _I),
    "woq_w6a8_linear_bf16": ([_P, _Z, _P, _I, _I, _I, _P, _P, _Z, _P], _I),
    "woq_debug_group_dots": ([_I, _P, _Z, _P, _I, _I, _I, _P, _P], _I),
    "woq_w4a8_linear_bf16_noalloc": ([_P, _Z, _P, _I, _I, _I, _P, _P], _I),
    "woq_noalloc_read_status": ([_I, ctypes.POINTER(ctypes.c_uint32), _P], _I),
    "woq_tune_override": ([_I, _I, _I], _I),
    "woq_tune_path": ([_I], _I),
    "woq_tune_fault": ([_I, _I, _I], _I),
    "woq_prefetch_next": ([_P, _Z, _I, _I, _I, _I], _I),
    "woq_last_cuda_error": ([], _I),
    "woq_cuda_error_name": ([_I], ctypes.c_char_p),
    "woq_w4a8_linear_rmsnorm_bf16": ([_P, _Z, _P, _P, ctypes.c_float, _I, _I, _I, _P, _P, _Z, _P], _I),
    "woq_w6a8_linear_rmsnorm_bf16": ([_P, _Z, _P, _P, ctypes.c_float, _I, _I, _I, _P, _P, _Z, _P], _I),
    "woq_w4a8_linear_swiglu_f32": ([_P, _Z, _P, _I, _I, _I, _P, _P, _Z, _P], _I),
    "woq_w6a8_linear_swiglu_f32": ([_P, _Z, _P, _I, _I, _I, _P, _P, _Z, _P], _I),
    "woq_rmsnorm_act_quant_int8": ([_P, _P, ctypes.c_float, _I, _I, _P, _P, _P], _I),
    "woq_swiglu_act_quant_int8": ([_P, _I, _I, _P, _P, _P], _I),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = _res


class WoqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {lib.woq_status_string(status).decode()} (status {status})"
        if status == WOQ_ERR_CUDA:
            code = lib.woq_last_cuda_error()
            msg += f" [{lib.woq_cuda_error_name(code).decode()}]"
        super().__init__(msg)


def _check(status: int, what: str) -> None:
    if status != WOQ_OK:
        raise WoqError(status, what)


def _dptr(t, name: str = "tensor", itemsize: int = 0, numel: int = -1):
    """Device pointer of a tensor (None -> NULL).  The C entries take bare pointers (most with
    no size), so the tensor is checked here: a contiguous CUDA tensor on the current device,
    elements of itemsize bytes (when given) and at least numel of them (when given)."""
    if t is None:
        return None
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{name}: expected a CUDA tensor")
    import torch
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name}: tensor is on {t.device}, the current device is cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if itemsize and t.element_size() != itemsize:
        raise ValueError(f"{name}: expected {itemsize}-byte elements, got {t.dtype}")
    if numel >= 0 and t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements, the call needs {numel}")
    return ctypes.c_void_p(t.data_ptr())


def _rows(t, name: str) -> int:
    """Row count M of a 2-D activation tensor."""
    if t is None or t.dim() != 2:
        raise ValueError(f"{name}: expected a 2-D [M, K] tensor")
    return t.shape[0]


def _nbytes(t) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _hptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


# ----------------------------------------------------------------------------- info

def woq_version() -> int:
    return lib.woq_version()


def woq_max_m() -> int:
    return lib.woq_max_m()


def woq_max_k(bits: int, M: int, fused: bool) -> int:
    return lib.woq_max_k(bits, M, int(fused))


def woq_packed_bytes(bits: int, N: int, K: int) -> int:
    return lib.woq_packed_bytes(bits, N, K)


def woq_workspace_bytes(bits: int, M: int, N: int, K: int) -> int:
    return lib.woq_workspace_bytes(bits, M, N, K)


# ----------------------------------------------------------------------------- packing

def _pack_host(fn, bits: int, q: np.ndarray, scales_f16: np.ndarray, N: int, K: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(scales_f16).view(np.uint16)
    out = np.empty(max(lib.woq_packed_bytes(bits, N, K), 1), dtype=np.uint8)
    _check(fn(_hptr(q), _hptr(s), N, K, _hptr(out), out.nbytes), fn.__name__)
    return out[: lib.woq_packed_bytes(bits, N, K)]


def woq_pack_w4(q4: np.ndarray, scales_f16: np.ndarray, N: int, K: int) -> np.ndarray:
    """Host pack: canonical int4 bytes [N, K/2] + fp16 scale bits [N, K/128] -> packed bytes."""
    return _pack_host(lib.woq_pack_w4, 4, q4, scales_f16, N, K)


def woq_pack_w6(q6: np.ndarray, scales_f16: np.ndarray, N: int, K: int) -> np.ndarray:
    """Host pack: canonical int6 bytes [N, 3K/4] + fp16 scale bits [N, K/128] -> packed bytes."""
    return _pack_host(lib.woq_pack_w6, 6, q6, scales_f16, N, K)


def woq_unpack(bits: int, packed: np.ndarray, N: int, K: int):
    """Host unpack: packed bytes -> (canonical bytes [N, row bytes], fp16 scale bits [N, K/128])."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    row = K // 2 if bits == 4 else K // 4 * 3
    q = np.zeros((N, row), dtype=np.uint8)
    s = np.zeros((N, K // GROUP), dtype=np.uint16)
    _check(lib.woq_unpack(bits, _hptr(packed), packed.nbytes, N, K, _hptr(q), _hptr(s)), "woq_unpack")
    return q, s


def woq_pack_device(bits: int, q_dev, scales_dev, N: int, K: int, dst_dev, stream=None) -> None:
    """Device pack into dst_dev (uint8 tensor of woq_packed_bytes(bits, N, K) bytes)."""
    row = K // 2 if bits == 4 else K // 4 * 3
    _check(lib.woq_pack_device(bits, _dptr(q_dev, "q_dev", 1, N * row), _dptr(scales_dev, "scales_dev", 2, N * (K // GROUP)),
                               N, K, _dptr(dst_dev, "dst_dev", 1), _nbytes(dst_dev), _stream(stream)), "woq_pack_device")


def woq_relayout_inplace(bits: int, buf, N: int, K: int, stream=None) -> None:
    """In-place relayout of buf (uint8 device tensor of woq_packed_bytes(bits, N, K)
    bytes): canonical weights from byte 256 on, then the fp16 scales; packed on return."""
    _check(lib.woq_relayout_inplace(bits, _dptr(buf, "buf", 1), _nbytes(buf), N, K, _stream(stream)),
           "woq_relayout_inplace")


def canonical_into_buffer(bits: int, q_dev, scales_dev, buf) -> None:
    """Place canonical weights and scales (device tensors) where woq_relayout_inplace expects them."""
    import torch

    qb = q_dev.reshape(-1).view(torch.uint8)
    sb = scales_dev.reshape(-1).view(torch.uint8)
    buf[256:256 + qb.numel()].copy_(qb)
    buf[256 + qb.numel():256 + qb.numel() + sb.numel()].copy_(sb)


# ----------------------------------------------------------------------------- workspace

def woq_workspace_init(ws, stream=None) -> None:
    _check(lib.woq_workspace_init(_dptr(ws, "ws", 1), _nbytes(ws), _stream(stream)), "woq_workspace_init")


def woq_read_status(ws, clear: bool = False, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(lib.woq_read_status(_dptr(ws, "ws", 1), _nbytes(ws), int(clear), ctypes.byref(v), _stream(stream)),
           "woq_read_status")
    return int(v.value)


# ----------------------------------------------------------------------------- compute

def woq_act_quant_int8(x_bf16, q, ascale, stream=None) -> None:
    """x_bf16 [M, K] bf16 -> q [M, K] int8, ascale [M] fp32 (device tensors)."""
    M = _rows(x_bf16, "x_bf16")
    K = x_bf16.shape[1]
    _check(lib.woq_act_quant_int8(_dptr(x_bf16, "x_bf16", 2), M, K, _dptr(q, "q", 1, M * K),
                                  _dptr(ascale, "ascale", 4, M), _stream(stream)), "woq_act_quant_int8")


def _gemv(fn, name, wpacked, q, ascale, N, K, y, ws, stream):
    M = _rows(q, "q")
    _check(fn(_dptr(wpacked, "wpacked", 1), _nbytes(wpacked), _dptr(q, "q", 1, M * K), _dptr(ascale, "ascale", 4, M),
              M, N, K, _dptr(y, "y", 4, M * N), _dptr(ws, "ws", 1), _nbytes(ws), _stream(stream)), name)


def woq_w4a8_gemv(wpacked, q, ascale, N: int, K: int, y, ws, stream=None) -> None:
    _gemv(lib.woq_w4a8_gemv, "woq_w4a8_gemv", wpacked, q, ascale, N, K, y, ws, stream)


def woq_w6a8_gemv(wpacked, q, ascale, N: int, K: int, y, ws, stream=None) -> None:
    _gemv(lib.woq_w6a8_gemv, "woq_w6a8_gemv", wpacked, q, ascale, N, K, y, ws, stream)


def _linear(fn, name, wpacked, x_bf16, N, K, y, ws, stream):
    M = _rows(x_bf16, "x_bf16")
    _check(fn(_dptr(wpacked, "wpacked", 1), _nbytes(wpacked), _dptr(x_bf16, "x_bf16", 2, M * K), M, N, K,
              _dptr(y, "y", 4, M * N), _dptr(ws, "ws", 1), _nbytes(ws), _stream(stream)), name)


def woq_w4a8_linear_bf16(wpacked, x_bf16, N: int, K: int, y, ws, stream=None) -> None:
    _linear(lib.woq_w4a8_linear_bf16, "woq_w4a8_linear_bf16", wpacked, x_bf16, N, K, y, ws, stream)


def woq_w6a8_linear_bf16(wpacked, x_bf16, N: int, K: int, y, ws, stream=None) -> None:
    _linear(lib.woq_w6a8_linear_bf16, "woq_w6a8_linear_bf16", wpacked, x_bf16, N, K, y, ws, stream)


def _linear_rmsnorm(fn, name, wpacked, x_bf16, gamma_bf16, eps, N, K, y, ws, stream):
    M = _rows(x_bf16, "x_bf16")
    _check(fn(_dptr(wpacked, "wpacked", 1), _nbytes(wpacked), _dptr(x_bf16, "x_bf16", 2, M * K),
              _dptr(gamma_bf16, "gamma_bf16", 2, K), float(eps), M, N, K, _dptr(y, "y", 4, M * N),
              _dptr(ws, "ws", 1), _nbytes(ws), _stream(stream)), name)


def woq_w4a8_linear_rmsnorm_bf16(wpacked, x_bf16, gamma_bf16, eps: float, N: int, K: int, y, ws, stream=None) -> None:
    """RMSNorm(x) with gamma, quantised and run through the int4 linear, in one launch."""
    _linear_rmsnorm(lib.woq_w4a8_linear_rmsnorm_bf16, "woq_w4a8_linear_rmsnorm_bf16", wpacked, x_bf16, gamma_bf16, eps,
                    N, K, y, ws, stream)


def woq_w6a8_linear_rmsnorm_bf16(wpacked, x_bf16, gamma_bf16, eps: float, N: int, K: int, y, ws, stream=None) -> None:
    _linear_rmsnorm(lib.woq_w6a8_linear_rmsnorm_bf16, "woq_w6a8_linear_rmsnorm_bf16", wpacked, x_bf16, gamma_bf16, eps,
                    N, K, y, ws, stream)


def _linear_swiglu(fn, name, wpacked, gate_up, N, K, y, ws, stream):
    M = _rows(gate_up, "gate_up")
    _check(fn(_dptr(wpacked, "wpacked", 1), _nbytes(wpacked), _dptr(gate_up, "gate_up", 4, M * 2 * K), M, N, K,
              _dptr(y, "y", 4, M * N), _dptr(ws, "ws", 1), _nbytes(ws), _stream(stream)), name)


def woq_w4a8_linear_swiglu_f32(wpacked, gate_up, N: int, K: int, y, ws, stream=None) -> None:
    """SwiGLU of an fp32 gate+up output [M, 2K], quantised and run through the int4 linear, in one launch."""
    _linear_swiglu(lib.woq_w4a8_linear_swiglu_f32, "woq_w4a8_linear_swiglu_f32", wpacked, gate_up, N, K, y, ws, stream)


def woq_w6a8_linear_swiglu_f32(wpacked, gate_up, N: int, K: int, y, ws, stream=None) -> None:
    _linear_swiglu(lib.woq_w6a8_linear_swiglu_f32, "woq_w6a8_linear_swiglu_f32", wpacked, gate_up, N, K, y, ws, stream)


def woq_rmsnorm_act_quant_int8(x_bf16, gamma_bf16, eps: float, q, ascale, stream=None) -> None:
    M = _rows(x_bf16, "x_bf16")
    K = x_bf16.shape[1]
    _check(lib.woq_rmsnorm_act_quant_int8(_dptr(x_bf16, "x_bf16", 2), _dptr(gamma_bf16, "gamma_bf16", 2, K), float(eps),
                                          M, K, _dptr(q, "q", 1, M * K), _dptr(ascale, "ascale", 4, M),
                                          _stream(stream)), "woq_rmsnorm_act_quant_int8")


def woq_swiglu_act_quant_int8(gate_up, q, ascale, stream=None) -> None:
    M = _rows(gate_up, "gate_up")
    K = gate_up.shape[1] // 2
    _check(lib.woq_swiglu_act_quant_int8(_dptr(gate_up, "gate_up", 4), M, K, _dptr(q, "q", 1, M * K),
                                         _dptr(ascale, "ascale", 4, M), _stream(stream)), "woq_swiglu_act_quant_int8")


def woq_w4a8_linear_bf16_noalloc(wpacked, x_bf16, N: int, K: int, y, stream=None) -> None:
    """woq_w4a8_linear_bf16 for callers that cannot allocate a workspace (the library's own
    2 MiB scratch is used; calls that overlap on the GPU race)."""
    M = _rows(x_bf16, "x_bf16")
    _check(lib.woq_w4a8_linear_bf16_noalloc(_dptr(wpacked, "wpacked", 1), _nbytes(wpacked),
                                            _dptr(x_bf16, "x_bf16", 2, M * K), M, N, K, _dptr(y, "y", 4, M * N),
                                            _stream(stream)), "woq_w4a8_linear_bf16_noalloc")


def woq_noalloc_read_status(clear: bool = False, stream=None) -> int:
    """Status word (WOQ_DEVERR_* bits) of the allocation-free linear's built-in scratch."""
    v = ctypes.c_uint32(0)
    _check(lib.woq_noalloc_read_status(int(clear), ctypes.byref(v), _stream(stream)), "woq_noalloc_read_status")
    return int(v.value)


def woq_debug_group_dots(bits: int, wpacked, q, N: int, K: int, dots, stream=None) -> None:
    M = _rows(q, "q")
    _check(lib.woq_debug_group_dots(bits, _dptr(wpacked, "wpacked", 1), _nbytes(wpacked), _dptr(q, "q", 1, M * K), M, N,
                                    K, _dptr(dots, "dots", 4, M * N * (K // GROUP)), _stream(stream)),
           "woq_debug_group_dots")


class LaunchPlan(ctypes.Structure):
    """woq_launch_plan of include/woq.h."""
    _fields_ = [("ctas", ctypes.c_int), ("stages", ctypes.c_int), ("prefetch_stages", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("consumer", ctypes.c_int)]


lib.woq_plan_launch.argtypes = [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(LaunchPlan)]
lib.woq_plan_launch.restype = _I

PLAN_INT8, PLAN_BF16, PLAN_SWIGLU = 0, 1, 2  # entry kinds of woq_plan_launch


def woq_plan_launch(bits: int, M: int, N: int, K: int, entry: int = PLAN_BF16, sms: int = 0,
                    smem_max: int = 0) -> dict:
    """The launch table's choice (grid, ring stages, L2 prefetch stages, shared memory, consumer)
    for one launch, on the current device or on one with sms SMs and smem_max bytes of opt-in
    shared memory per block; nothing is launched."""
    plan = LaunchPlan()
    _check(lib.woq_plan_launch(bits, M, N, K, entry, sms, smem_max, ctypes.byref(plan)), "woq_plan_launch")
    return {name: getattr(plan, name) for name, _ in LaunchPlan._fields_}


def woq_prefetch_next(next_wpacked, bits: int, N: int, K: int, budget_kb: int = 0) -> None:
    """Hint for the next GEMV / linear call of this thread: the linear that runs after it
    (packed weights next_wpacked of (bits, N, K)); None clears the hint."""
    if next_wpacked is None:
        _check(lib.woq_prefetch_next(None, 0, bits, N, K, 0), "woq_prefetch_next")
        return
    _check(lib.woq_prefetch_next(_dptr(next_wpacked, "next_wpacked", 1), _nbytes(next_wpacked), bits, N, K, budget_kb),
           "woq_prefetch_next")


def woq_tune_override(ctas_per_sm: int = 0, stages: int = 0, prefetch_kb: int = -1) -> None:
    _check(lib.woq_tune_override(ctas_per_sm, stages, prefetch_kb), "woq_tune_override")


def woq_tune_fault(kind: int = 0, cta: int = 0, wait_limit_us: int = 0) -> None:
    """Tests of the bounded waits: inject one CTA's missing arrival (include/woq.h)."""
    _check(lib.woq_tune_fault(kind, cta, wait_limit_us), "woq_tune_fault")


def woq_tune_path(path: int = 0) -> None:
    """int4 consumer of later launches: 0 launch table, 1 dp4a, 2 tensor-core MMA."""
    _check(lib.woq_tune_path(path), "woq_tune_path")


# ----------------------------------------------------------------------------- draft-tree planner
# (include/woq_tree.h; host code in the same library)

_TREE_ROWS, _TREE_BINS, TREE_SHAPES = 7, 8, 64


class TreePlannerState(ctypes.Structure):
    _fields_ = [("counts", (ctypes.c_double * _TREE_BINS) * _TREE_ROWS),
                ("draft_ms", ctypes.c_double), ("verify_ms", ctypes.c_double),
                ("decay", ctypes.c_double), ("hysteresis", ctypes.c_double),
                ("replan_every", ctypes.c_int), ("steps", ctypes.c_int), ("times_seen", ctypes.c_int),
                ("widths", ctypes.c_int * _TREE_ROWS), ("depth", ctypes.c_int)]


_TP = ctypes.POINTER(TreePlannerState)
_IP = ctypes.POINTER(ctypes.c_int)
_DP = ctypes.POINTER(ctypes.c_double)
for _name, (_args, _res) in {
    "woq_tree_init": ([_TP, ctypes.c_double, ctypes.c_double, _I], _I),
    "woq_tree_shape": ([_I, _IP, _IP], _I),
    "woq_tree_score": ([_TP, _IP, _I, _DP, _DP], _I),
    "woq_tree_observe": ([_TP, _I, _IP, ctypes.c_double, ctypes.c_double, _IP], _I),
    "woq_tree_replan": ([_TP, _IP, _DP, _IP], _I),
}.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = _res


def woq_tree_shape(index: int) -> tuple:
    w = (ctypes.c_int * _TREE_ROWS)()
    d = ctypes.c_int()
    _check(lib.woq_tree_shape(index, w, ctypes.byref(d)), "woq_tree_shape")
    return tuple(w[: d.value])


class TreePlanner:
    """The draft-tree planner of include/woq_tree.h (argument marshalling only)."""

    def __init__(self, decay: float = 0.0, hysteresis: float = -1.0, replan_every: int = 0):
        self.state = TreePlannerState()
        _check(lib.woq_tree_init(ctypes.byref(self.state), decay, hysteresis, replan_every), "woq_tree_init")

    @property
    def shape(self) -> tuple:
        return tuple(self.state.widths[: self.state.depth])

    def score(self, widths) -> tuple:
        w = (ctypes.c_int * _TREE_ROWS)(*widths)
        e, s = ctypes.c_double(), ctypes.c_double()
        _check(lib.woq_tree_score(ctypes.byref(self.state), w, len(widths), ctypes.byref(e), ctypes.byref(s)),
               "woq_tree_score")
        return e.value, s.value

    def observe(self, ranks, draft_ms: float = -1.0, verify_ms: float = -1.0) -> bool:
        r = (ctypes.c_int * _TREE_ROWS)(*ranks)
        sw = ctypes.c_int()
        _check(lib.woq_tree_observe(ctypes.byref(self.state), len(ranks), r, draft_ms, verify_ms, ctypes.byref(sw)),
               "woq_tree_observe")
        return bool(sw.value)

    def replan(self) -> tuple:
        i, s, sw = ctypes.c_int(), ctypes.c_double(), ctypes.c_int()
        _check(lib.woq_tree_replan(ctypes.byref(self.state), ctypes.byref(i), ctypes.byref(s), ctypes.byref(sw)),
               "woq_tree_replan")
        return i.value, s.value, bool(sw.value)

    def counts(self) -> np.ndarray:
        return np.array([[self.state.counts[d][b] for b in range(_TREE_BINS)] for d in range(_TREE_ROWS)])
