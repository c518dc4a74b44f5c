"""Pins for the oracle's exact element widening (binary16, bfloat16, binary32).

The reference values come from a library routine (PyTorch's CPU dtype
conversion) and from closed forms, not from the oracle.
"""
import math
import struct

import numpy as np
import pytest
import torch

import oracle


def _all_16bit(dtype):
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    return bits.view(dtype).to(torch.float32).tolist()


@pytest.mark.parametrize("name,dtype,fn", [
    ("f16", torch.float16, oracle.f16_to_f64),
    ("bf16", torch.bfloat16, oracle.bf16_to_f64),
])
def test_every_16bit_pattern_matches_library(name, dtype, fn):
    ref = _all_16bit(dtype)
    for b in range(1 << 16):
        got = fn(b)
        want = ref[b]
        if math.isnan(want):
            assert math.isnan(got), (name, hex(b))
        else:
            assert got == want, (name, hex(b), got, want)
            # signed zero preserved
            assert math.copysign(1.0, got) == math.copysign(1.0, want)


def test_f16_closed_forms():
    assert oracle.f16_to_f64(0x3C00) == 1.0
    assert oracle.f16_to_f64(0xC000) == -2.0
    assert oracle.f16_to_f64(0x7BFF) == 65504.0           # largest finite
    assert oracle.f16_to_f64(0x0001) == 2.0 ** -24         # smallest subnormal
    assert oracle.f16_to_f64(0x03FF) == 1023 * 2.0 ** -24  # largest subnormal
    assert oracle.f16_to_f64(0x0400) == 2.0 ** -14         # smallest normal
    assert oracle.f16_to_f64(0x7C00) == math.inf
    assert oracle.f16_to_f64(0xFC00) == -math.inf
    assert math.isnan(oracle.f16_to_f64(0x7E00))


def test_bf16_closed_forms():
    assert oracle.bf16_to_f64(0x3F80) == 1.0
    assert oracle.bf16_to_f64(0x4049) == 3.140625
    assert oracle.bf16_to_f64(0x0001) == 2.0 ** -133
    assert oracle.bf16_to_f64(0x7F80) == math.inf


def test_f32_random_patterns_match_numpy():
    rng = np.random.default_rng(7)
    pats = rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    vals = pats.view(np.float32).astype(np.float64)
    for p, v in zip(pats.tolist(), vals.tolist()):
        got = oracle.f32_to_f64(p)
        if math.isnan(v):
            assert math.isnan(got)
        else:
            assert got == v
    assert oracle.f32_to_f64(struct.unpack("<I", struct.pack("<f", 0.1))[0]) == \
        struct.unpack("<f", struct.pack("<f", 0.1))[0]
