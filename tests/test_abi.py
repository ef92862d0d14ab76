"""The C ABI library builds, loads without a GPU, exports every symbol that
include/*.h declares, and rejects invalid arguments on the host (these
checks run before any CUDA call, so no GPU is needed)."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def woq():
    from weight_only_quantised_gb300 import _build
    _build.build()
    import weight_only_quantised_gb300 as w
    return w


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for h in sorted(os.listdir(inc)):
        if h.endswith(".h"):
            with open(os.path.join(inc, h)) as f:
                names |= set(re.findall(r"^WOQ_API\s+[\w\s\*]+?\b(woq_\w+)\s*\(", f.read(), flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["woq_pack_w4", "woq_pack_w6", "woq_act_quant_int8", "woq_w4a8_gemv", "woq_w6a8_gemv",
                     "woq_w4a8_linear_bf16", "woq_w6a8_linear_bf16", "woq_debug_group_dots"]:
        assert required in names


def test_library_exports_every_declared_symbol(woq):
    names = declared_functions()
    assert len(names) >= 19
    for n in names:
        assert hasattr(woq.lib, n), n
    # and nothing else leaks out (the CUDA runtime is linked statically and kept local)
    out = subprocess.run(["nm", "-D", "--defined-only", woq.LIB_PATH], capture_output=True, text=True).stdout
    exported = sorted(line.split()[-1] for line in out.splitlines() if line.strip())
    assert exported == names


def test_status_strings(woq):
    for s in range(8):
        assert woq.lib.woq_status_string(s)
    assert woq.lib.woq_status_string(99) == b"unknown status"
    assert woq.woq_max_m() == 8
    assert woq.woq_version() >= 100


def test_packed_bytes_formula(woq):
    for bits, per_block in ((4, 256 + 128 * 64), (6, 256 + 128 * 96)):
        for N, K in [(1, 128), (128, 128), (129, 256), (4096, 4096), (152064, 5120), (0, 128), (5, 0)]:
            tiles = (N + 127) // 128
            assert woq.woq_packed_bytes(bits, N, K) == 256 + tiles * (K // 128) * per_block
    assert woq.woq_packed_bytes(4, 10, 100) == 0
    assert woq.woq_packed_bytes(5, 10, 128) == 0
    assert woq.woq_packed_bytes(4, -1, 128) == 0


FAKE = 0x10000  # an aligned, never-dereferenced address: host validation fails first


def test_gemv_host_validation(woq):
    L = woq.lib
    P = ctypes.c_void_p
    good = dict(w=P(FAKE), wb=10 ** 9, q=P(FAKE), a=P(FAKE), M=1, N=128, K=128, y=P(FAKE), ws=P(FAKE), wsb=10 ** 9)

    def call(fn=L.woq_w4a8_gemv, **kw):
        a = dict(good, **kw)
        return fn(a["w"], a["wb"], a["q"], a["a"], a["M"], a["N"], a["K"], a["y"], a["ws"], a["wsb"], None)

    assert call(M=5) == woq.WOQ_ERR_SHAPE
    assert call(M=-1) == woq.WOQ_ERR_SHAPE
    assert call(K=100) == woq.WOQ_ERR_SHAPE
    assert call(M=4, K=128 * 200) == woq.WOQ_ERR_SHAPE  # M * K beyond the shared-memory bound
    assert call(M=0) == woq.WOQ_OK  # empty: nothing launched
    assert call(N=0) == woq.WOQ_OK
    assert call(w=None) == woq.WOQ_ERR_NULL
    assert call(q=None) == woq.WOQ_ERR_NULL
    assert call(y=None) == woq.WOQ_ERR_NULL
    assert call(w=P(FAKE + 8)) == woq.WOQ_ERR_ALIGN
    assert call(q=P(FAKE + 4)) == woq.WOQ_ERR_ALIGN
    assert call(y=P(FAKE + 2)) == woq.WOQ_ERR_ALIGN
    assert call(ws=P(FAKE + 8)) == woq.WOQ_ERR_ALIGN
    assert call(wb=woq.woq_packed_bytes(4, 128, 128) - 1) == woq.WOQ_ERR_LAYOUT
    assert call(fn=L.woq_w6a8_gemv, wb=woq.woq_packed_bytes(4, 128, 128)) == woq.WOQ_ERR_LAYOUT


def test_linear_and_act_quant_host_validation(woq):
    L = woq.lib
    P = ctypes.c_void_p
    assert L.woq_w4a8_linear_bf16(P(FAKE), 10 ** 9, None, 1, 128, 128, P(FAKE), P(FAKE), 10 ** 9, None) == \
        woq.WOQ_ERR_NULL
    assert L.woq_w4a8_linear_bf16(P(FAKE), 10 ** 9, P(FAKE + 2), 1, 128, 128, P(FAKE), P(FAKE), 10 ** 9, None) == \
        woq.WOQ_ERR_ALIGN
    assert L.woq_act_quant_int8(P(FAKE), 9, 128, P(FAKE), P(FAKE), None) == woq.WOQ_ERR_SHAPE
    assert L.woq_act_quant_int8(P(FAKE), 0, 128, None, None, None) == woq.WOQ_OK
    assert L.woq_act_quant_int8(None, 1, 128, P(FAKE), P(FAKE), None) == woq.WOQ_ERR_NULL
    assert L.woq_act_quant_int8(P(FAKE + 1), 1, 128, P(FAKE), P(FAKE), None) == woq.WOQ_ERR_ALIGN
    assert L.woq_debug_group_dots(5, P(FAKE), 10 ** 9, P(FAKE), 1, 128, 128, P(FAKE), None) == woq.WOQ_ERR_SHAPE
    assert L.woq_debug_group_dots(4, None, 10 ** 9, P(FAKE), 1, 128, 128, P(FAKE), None) == woq.WOQ_ERR_NULL
    assert L.woq_tune_override(3, 0, -1) == woq.WOQ_ERR_SHAPE
    assert L.woq_tune_override(0, 1, -1) == woq.WOQ_ERR_SHAPE
    assert L.woq_tune_override(0, 0, -2) == woq.WOQ_ERR_SHAPE
    assert L.woq_tune_override(0, 0, -1) == woq.WOQ_OK


def test_cuda_failure_is_reported_and_cleared(woq):
    """Without a GPU every CUDA runtime call fails: the entry returns WOQ_ERR_CUDA, the failing
    code is kept for woq_last_cuda_error (and named by woq_cuda_error_name), and the binding's
    exception carries the name.  Skipped where a GPU is present (no invalid pointer ever reaches
    a device)."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU")
    L = woq.lib
    P = ctypes.c_void_p
    assert L.woq_cuda_error_name(0) == b"cudaSuccess"
    assert L.woq_workspace_init(P(FAKE), 256, None) == woq.WOQ_ERR_CUDA
    code = L.woq_last_cuda_error()
    assert code != 0
    assert L.woq_cuda_error_name(code).startswith(b"cudaError")
    # host-side validation still answers first and leaves the recorded code alone
    assert L.woq_workspace_init(None, 256, None) == woq.WOQ_ERR_NULL
    assert L.woq_last_cuda_error() == code
    with pytest.raises(woq.WoqError, match=r"\[cudaError\w+\]"):
        woq._check(L.woq_workspace_init(P(FAKE), 256, None), "woq_workspace_init")


def test_binding_refuses_host_tensors(woq):
    """The Python entries hand bare pointers to the library: a tensor that is not on the GPU is
    refused before any call (checked on the CPU; the size, layout and element checks need device
    tensors and are covered by the GPU tests)."""
    torch = pytest.importorskip("torch")
    N, K, M = 128, 256, 1
    w = torch.zeros(woq.woq_packed_bytes(4, N, K), dtype=torch.uint8)
    x = torch.zeros((M, K), dtype=torch.bfloat16)
    y = torch.zeros((M, N), dtype=torch.float32)
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        woq.woq_w4a8_linear_bf16(w, x, N, K, y, ws)
    with pytest.raises(ValueError, match="CUDA tensor"):
        woq.woq_act_quant_int8(x, torch.zeros((M, K), dtype=torch.int8), torch.zeros((M,)))
    with pytest.raises(ValueError, match="2-D"):
        woq.woq_w4a8_linear_bf16(w, x.reshape(-1), N, K, y, ws)
