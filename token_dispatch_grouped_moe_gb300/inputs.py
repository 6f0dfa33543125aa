"""Seeded synthetic inputs for the MoE layer (shared by the CUDA path's tests,
the benchmark and the oracle's tests).

This module draws random numbers and nothing else: it holds none of the
layer's arithmetic. Every tensor comes from its own CPU ``torch.Generator``
seeded with ``seed + offset`` (x: +0, Wg: +1, W1: +2, W3: +3, W2: +4,
shared W1s/W3s/W2s: +5/+6/+7), as ``randn * sigma`` in fp32, rounded to
nearest-even bf16. x has sigma 1; every weight has sigma 0.02 (a standard
deviation, not a variance).

Layouts (row-major, contiguous): x[T,H], Wg[H,E], W1/W3[E,H,F], W2[E,F,H],
W1s/W3s[H,Fs], W2s[Fs,H].
"""
from __future__ import annotations

import numpy as np
import torch

SIGMA_X = 1.0
SIGMA_W = 0.02

SEED_OFFSETS = dict(x=0, Wg=1, W1=2, W3=3, W2=4, W1s=5, W3s=6, W2s=7)


def _randn_bf16(shape, seed: int, sigma: float) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    if sigma != 1.0:
        t.mul_(sigma)
    return t.to(torch.bfloat16)


def make_inputs(T: int, H: int, F: int, E: int, Fs: int = 0, seed: int = 0,
                only: tuple[str, ...] | None = None) -> dict[str, torch.Tensor]:
    """CPU bf16 tensors for one layer. ``only`` restricts which are drawn."""
    shapes = dict(x=(T, H), Wg=(H, E), W1=(E, H, F), W3=(E, H, F), W2=(E, F, H))
    if Fs > 0:
        shapes.update(W1s=(H, Fs), W3s=(H, Fs), W2s=(Fs, H))
    out = {}
    for name, shape in shapes.items():
        if only is not None and name not in only:
            continue
        sigma = SIGMA_X if name == "x" else SIGMA_W
        out[name] = _randn_bf16(shape, seed + SEED_OFFSETS[name], sigma)
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bits of a CPU bf16 tensor as a uint16 numpy array (no copy)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    """Inverse of :func:`bf16_bits`."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
