"""Seeded synthetic inputs shared by the tests, ``smoke()`` and ``bench.py``.

This module only draws random numbers and moves bit patterns around; it
holds none of the tensor-parallel arithmetic.  Both the CUDA path and the
CPU oracle are fed the same bit patterns produced here.

Recipe: ``torch.Generator(device).manual_seed(seed)`` then ``torch.randn``
in float32, scaled by ``std`` and rounded to bfloat16 by torch's
``.to(torch.bfloat16)``.  Integer-valued variants use ``torch.randint``.
Token ids are uniform on [0, vocab) as int32.  Seeds per tensor follow the
offsets of :data:`SEED_OFFSETS` so that each tensor of a configuration has
its own stream.
"""

from __future__ import annotations

from typing import Sequence

import numpy as np
import torch

SEED_OFFSETS = {"x": 0, "gate": 1, "up": 2, "down": 3, "bias": 4, "ids": 5, "table": 6, "head_x": 7}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape: Sequence[int], std: float, seed: int, device="cpu") -> torch.Tensor:
    """bfloat16 tensor of N(0, std^2) draws."""
    x = torch.randn(tuple(shape), generator=_gen(seed, device), dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def normal_f32(shape: Sequence[int], std: float, seed: int, device="cpu") -> torch.Tensor:
    """float32 tensor of N(0, std^2) draws."""
    x = torch.randn(tuple(shape), generator=_gen(seed, device), dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    return x


def int_valued(shape: Sequence[int], lo: int, hi: int, seed: int, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """Integers drawn uniformly from [lo, hi] stored in a float dtype."""
    x = torch.randint(lo, hi + 1, tuple(shape), generator=_gen(seed, device), device=device)
    return x.to(dtype)


def uniform_ids(n: int, vocab: int, seed: int, device="cpu") -> torch.Tensor:
    """int32 token ids uniform on [0, vocab)."""
    return torch.randint(0, vocab, (n,), generator=_gen(seed, device), device=device, dtype=torch.int64).to(torch.int32)


def bits_u16(t: torch.Tensor) -> np.ndarray:
    """Bit patterns of a bfloat16 tensor as a numpy uint16 array (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits_u32(t: torch.Tensor) -> np.ndarray:
    """Bit patterns of a float32 tensor as a numpy uint32 array (host copy)."""
    assert t.dtype == torch.float32
    return t.detach().contiguous().view(torch.int32).cpu().numpy().view(np.uint32)


def from_bits_u16(bits: np.ndarray, device="cpu") -> torch.Tensor:
    """bfloat16 tensor holding the given uint16 bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).to(device)
