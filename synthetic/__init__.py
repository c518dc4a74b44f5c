"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws numbers; it holds none of the tile pipeline's arithmetic.
Both the CPU oracle and the CUDA path receive the same host bytes from here.

Recipe (the workloads of the tile-copy and row-sum lessons, scaled to the
streaming sizes):

* ``uniform``: ``torch.rand`` in float32 on the CPU, mapped to [-1, 1) by
  ``2u - 1``, then rounded to the storage dtype (round to nearest even).
* ``normal``: ``torch.randn`` in float32 on the CPU, then rounded.
* A generator seeded with ``seed`` is used, so a (shape, dtype, dist, seed)
  tuple always gives the same bits on every machine.
* Pitched storage (``ld > N``): columns ``N .. ld-1`` of every row hold
  ``PAD_BITS[dtype]``, a quiet-NaN bit pattern that must never reach a copy
  destination or a row sum.
"""
from __future__ import annotations

import torch

__all__ = [
    "DTYPES",
    "ESIZE",
    "PAD_BITS",
    "POISON_BITS",
    "pitched_ld",
    "make_matrix",
    "fill_bits",
    "special_values",
]

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
ESIZE = {"f16": 2, "bf16": 2, "f32": 4}

# Quiet NaNs with a payload, written into pad columns of a pitched source.
PAD_BITS = {"f16": 0x7E5A, "bf16": 0x7FA5, "f32": 0x7FC0_5A5A}
# Another payload, written over a destination before a copy so that any byte
# the copy did not write (or wrote where it should not) is detectable.
POISON_BITS = {"f16": 0x7D3C, "bf16": 0x7FB3, "f32": 0x7FB0_3C3C}

_INT_VIEW = {2: torch.int16, 4: torch.int32}


def pitched_ld(N: int, dtype: str) -> int:
    """Smallest row pitch (elements) >= N whose byte size is a multiple of 16."""
    per16 = 16 // ESIZE[dtype]
    return ((N + per16 - 1) // per16) * per16


def _signed(bits: int, nbytes: int) -> int:
    top = 1 << (8 * nbytes)
    return bits - top if bits >= top // 2 else bits


def fill_bits(t: torch.Tensor, bits: int) -> torch.Tensor:
    """Fill tensor ``t`` (in place) with the raw bit pattern ``bits``."""
    es = t.element_size()
    t.view(_INT_VIEW[es]).fill_(_signed(bits, es))
    return t


def make_matrix(M: int, N: int, dtype: str, dist: str, seed: int,
                ld: int | None = None, device: str | None = None,
                draw_on: str = "cpu") -> torch.Tensor:
    """Return a (M, ld) tensor whose first N columns hold the seeded values.

    The logical matrix is ``t[:, :N]``; ``t.stride(0) == ld``.  ``draw_on``
    selects the generator: "cpu" (the bits every test uses) or a CUDA device
    (same distribution, different bits, much faster for GiB-sized inputs).
    The result lives on ``device`` (default: where it was drawn).
    """
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    ld = N if ld is None else ld
    if ld < N:
        raise ValueError("ld must be >= N")
    where = torch.device(draw_on)
    g = torch.Generator(device=where)
    g.manual_seed(seed)
    out = torch.empty(M, ld, dtype=DTYPES[dtype], device=where)
    if ld > N:
        fill_bits(out[:, N:], PAD_BITS[dtype])
    # draw in row blocks of at most 2^26 values to bound the float32 scratch
    rows = max(1, (1 << 26) // max(N, 1))
    for r0 in range(0, M, rows):
        r1 = min(M, r0 + rows)
        if dist == "uniform":
            vals = torch.rand(r1 - r0, N, generator=g, dtype=torch.float32, device=where)
            vals.mul_(2.0).sub_(1.0)
        elif dist == "normal":
            vals = torch.randn(r1 - r0, N, generator=g, dtype=torch.float32, device=where)
        else:
            raise ValueError(f"unknown distribution {dist!r}")
        out[r0:r1, :N].copy_(vals)
        del vals
    if device is not None and torch.device(device) != where:
        out = out.to(device)
    return out


def special_values(dtype: str) -> list[int]:
    """Bit patterns a bit-exact copy must preserve: signed zeros, infinities,
    NaNs with payloads, subnormals and the largest finite values."""
    if dtype == "f16":
        return [0x0000, 0x8000, 0x7C00, 0xFC00, 0x7E00, 0x7C01, 0xFE5A, 0x0001,
                0x8001, 0x03FF, 0x7BFF, 0xFBFF, 0x3C00, 0x0400]
    if dtype == "bf16":
        return [0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x7F81, 0xFFC1, 0x0001,
                0x8001, 0x007F, 0x7F7F, 0xFF7F, 0x3F80, 0x0080]
    if dtype == "f32":
        return [0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000,
                0x7F800001, 0xFFC0ABCD, 0x00000001, 0x80000001, 0x007FFFFF,
                0x7F7FFFFF, 0xFF7FFFFF, 0x3F800000, 0x00800000]
    raise ValueError(dtype)
