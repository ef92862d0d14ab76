"""Shared test helpers: the golden-file parser and canonical-layout encoders.

The encoders go from integer weight values to the canonical checkpoint bytes
(the inverse of what the oracle and the packer read).  They are written here,
independently of both, so a test can start from known integer weights.
"""
from __future__ import annotations

import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str) -> dict:
    """Parse 'key idx : v v v' lines into {(key, idx): [tokens]}; 'K 128' lines into {key: value}."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                head, vals = line.split(":", 1)
                key, idx = head.split()
                out[(key, int(idx))] = vals.split()
            else:
                key, val = line.split()
                out[key] = val
    return out


def encode_w4(vals: np.ndarray) -> np.ndarray:
    """int values in [-8, 7], shape [N, K] -> canonical bytes [N, K/2] (low nibble = even k)."""
    v = np.asarray(vals, dtype=np.int64)
    assert v.size == 0 or (v.min() >= -8 and v.max() <= 7)
    u = (v & 0xF).astype(np.uint8)
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def encode_w6(vals: np.ndarray) -> np.ndarray:
    """int values in [-32, 31], shape [N, K] -> canonical bytes [N, 3K/4] (24-bit LE words of 4 fields)."""
    v = np.asarray(vals, dtype=np.int64)
    assert v.size == 0 or (v.min() >= -32 and v.max() <= 31)
    N, K = v.shape
    f = (v & 0x3F).reshape(N, K // 4, 4)
    word = f[..., 0] | (f[..., 1] << 6) | (f[..., 2] << 12) | (f[..., 3] << 18)
    b = np.stack([word & 0xFF, (word >> 8) & 0xFF, (word >> 16) & 0xFF], axis=-1)
    return b.reshape(N, K // 4 * 3).astype(np.uint8)


def f16_bits(vals) -> np.ndarray:
    """Values -> fp16 bit patterns (round to nearest even by torch)."""
    t = torch.tensor(np.asarray(vals, dtype=np.float64), dtype=torch.float64).to(torch.float16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits(vals) -> np.ndarray:
    """Values -> bf16 bit patterns (round to nearest even by torch)."""
    t = torch.tensor(np.asarray(vals, dtype=np.float64), dtype=torch.float64).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values (via torch)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def f16_values(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.float16)
    return t.to(torch.float64).numpy()
