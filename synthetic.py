"""Seeded synthetic inputs for the skinny linear (shared by tests, smoke and bench).

This module only draws random numbers; it holds none of the method's
arithmetic, so the CPU oracle and the CUDA library can both be fed from it
without sharing any code with each other.

Recipe (the workloads of the decode linears of 9B- and 27B-class decoders):
  * int4 weights: uniform random bytes in the canonical layout (two weights per
    byte along K), i.e. each weight uniform over the 16 codes [-8, 7];
  * int6 weights: uniform random bytes in the canonical layout (four weights per
    three bytes along K), i.e. each weight uniform over [-32, 31];
  * group scales (one per row and 128 consecutive k): |N(0,1)| * c + eps drawn in
    fp32, then rounded to fp16 (round to nearest even);
    c, eps = 0.02, 1e-3 for int4 and 0.005, 1e-4 for int6;
  * activations: N(0,1) in fp32; optionally round(0.01 * K) outlier channels,
    picked once per matrix by a seeded permutation and shared by all rows,
    are multiplied by 20; then rounded once to bf16;
  * RMSNorm weights: 1 + 0.1 N(0,1) in fp32, rounded to bf16;
  * gate+up outputs (the SwiGLU prologue's input): 2 N(0,1) in fp32.

All draws use torch generators, so the same call gives the same bits for a
given device type; tests generate once and hand the same arrays to both sides.
"""
from __future__ import annotations

import hashlib

import numpy as np
import torch

GROUP = 128


def sub_seed(seed: int, *tags) -> int:
    """A 63-bit seed derived from a base seed and labels (deterministic everywhere)."""
    h = hashlib.sha256(repr((int(seed),) + tuple(tags)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def canonical_row_bytes(bits: int, K: int) -> int:
    """Bytes of one canonical row: K/2 for int4, 3K/4 for int6."""
    if bits == 4:
        return K // 2
    if bits == 6:
        return K // 4 * 3
    raise ValueError("bits must be 4 or 6")


def weights(bits: int, N: int, K: int, seed: int, device="cpu"):
    """Canonical weights (uint8 [N, row bytes]) and fp16 group scales ([N, K/128])."""
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    dev = torch.device(device)
    gw = _gen(sub_seed(seed, "w", bits, N, K), dev)
    w = torch.randint(0, 256, (N, canonical_row_bytes(bits, K)), dtype=torch.uint8, generator=gw, device=dev)
    c, eps = (0.02, 1e-3) if bits == 4 else (0.005, 1e-4)
    gs = _gen(sub_seed(seed, "s", bits, N, K), dev)
    s = torch.randn((N, K // GROUP), dtype=torch.float32, generator=gs, device=dev).abs_().mul_(c).add_(eps)
    return w, s.to(torch.float16)


def activations(M: int, K: int, seed: int, outliers: bool = True, device="cpu") -> torch.Tensor:
    """bf16 activations [M, K]: N(0,1), 1% outlier channels x20 when asked."""
    dev = torch.device(device)
    gx = _gen(sub_seed(seed, "x", M, K), dev)
    x = torch.randn((M, K), dtype=torch.float32, generator=gx, device=dev)
    if outliers and K > 0:
        n_out = int(round(0.01 * K))
        gp = _gen(sub_seed(seed, "outlier-channels", K), "cpu")
        idx = torch.randperm(K, generator=gp)[:n_out].to(dev)
        x[:, idx] *= 20.0
    return x.to(torch.bfloat16)


def rmsnorm_weight(K: int, seed: int, device="cpu") -> torch.Tensor:
    """bf16 RMSNorm weights [K]: 1 + 0.1 N(0,1)."""
    dev = torch.device(device)
    g = _gen(sub_seed(seed, "gamma", K), dev)
    return (1.0 + 0.1 * torch.randn((K,), dtype=torch.float32, generator=g, device=dev)).to(torch.bfloat16)


def gate_up_output(M: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """fp32 [M, 2K] stand-in for a gate+up linear's output (gate, then up): N(0,1) * 2."""
    dev = torch.device(device)
    g = _gen(sub_seed(seed, "gate_up", M, K), dev)
    return 2.0 * torch.randn((M, 2 * K), dtype=torch.float32, generator=g, device=dev)


def to_numpy_u16(t: torch.Tensor) -> np.ndarray:
    """Bit patterns of a 16-bit float tensor as a numpy uint16 array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def to_numpy_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


# Shapes of the decode linears (K -> N), named by what they are.
LINEARS_9B = {  # hidden 4096, 32 q heads + 8 kv heads of 128, MLP 12288
    "qkv": (4096, 6144),
    "o": (4096, 4096),
    "gate_up": (4096, 24576),
    "down": (12288, 4096),
}
LINEARS_27B = {  # hidden 5120, 40 q heads + 8 kv heads of 128, MLP 17408, 64 layers
    "qkv": (5120, 7168),
    "o": (5120, 5120),
    "gate_up": (5120, 34816),
    "down": (17408, 5120),
}
LM_HEAD_27B = (5120, 152064)
LAYERS_27B = 64


def step_27b():
    """The 27B-class decode step: 64 x (qkv, o, gate_up, down) then the LM head, as (name, K, N)."""
    out = []
    for layer in range(LAYERS_27B):
        for name, (K, N) in LINEARS_27B.items():
            out.append((f"L{layer}.{name}", K, N))
    out.append(("lm_head", LM_HEAD_27B[0], LM_HEAD_27B[1]))
    return out
