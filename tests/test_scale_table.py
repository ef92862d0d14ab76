"""The fused prologue's row-scale tables against IEEE fp32 division.

The GEMV's fused activation prologue looks the scale s = RN(amax / 127) and its
reciprocal rc = RN(1 / s) up by the bf16 significand of amax and shifts the
exponent.  Here numpy's correctly rounded fp32 division recomputes both for every
bf16 amax in the table's range (every significand, every exponent from 2^-119 to
the top of the range), and the committed header must equal the generator's output.
"""
import os
import re

import numpy as np

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "weight_only_quantised_gb300", "csrc")


def _tables():
    text = open(os.path.join(CSRC, "woq_scale_table.h")).read()
    words = [int(v, 16) for v in re.findall(r"0x([0-9A-F]{8})u", text)]
    assert len(words) == 256
    return np.array(words[:128], dtype=np.uint32), np.array(words[128:], dtype=np.uint32)


def test_table_matches_fp32_division_over_range():
    sig_s, sig_r = _tables()
    f = np.arange(128, dtype=np.uint32)
    for e in range(-119, 128):
        amax = ((np.uint32(e + 127) << np.uint32(23)) | (f << np.uint32(16))).view(np.float32)
        s = (amax / np.float32(127)).astype(np.float32)
        rc = (np.float32(1) / s).astype(np.float32)
        shift = np.int64(e) << 23
        s_tab = ((sig_s.astype(np.int64) + shift) & 0xFFFFFFFF).astype(np.uint32)
        r_tab = ((sig_r.astype(np.int64) - shift) & 0xFFFFFFFF).astype(np.uint32)
        np.testing.assert_array_equal(s_tab, s.view(np.uint32), err_msg=f"scale, exponent {e}")
        np.testing.assert_array_equal(r_tab, rc.view(np.uint32), err_msg=f"reciprocal, exponent {e}")


def test_header_is_generator_output():
    import importlib.util
    spec = importlib.util.spec_from_file_location("gen_scale_table", os.path.join(CSRC, "gen_scale_table.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    assert open(os.path.join(CSRC, "woq_scale_table.h")).read() == gen.render()
