"""The seeded input generator: determinism, value ranges and pad sentinels."""
import torch

import synthetic


def test_same_seed_same_bits_and_pitch():
    a = synthetic.make_matrix(7, 13, "f16", "uniform", seed=9, ld=16)
    b = synthetic.make_matrix(7, 13, "f16", "uniform", seed=9, ld=16)
    assert a.stride(0) == 16
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    c = synthetic.make_matrix(7, 13, "f16", "uniform", seed=10, ld=16)
    assert not torch.equal(a[:, :13], c[:, :13])


def test_uniform_range_and_pad_bits():
    x = synthetic.make_matrix(64, 37, "f32", "uniform", seed=1, ld=40)
    v = x[:, :37]
    assert v.min() >= -1.0 and v.max() <= 1.0
    pad = x[:, 37:].contiguous().view(torch.int32)
    assert (pad == synthetic.PAD_BITS["f32"]).all()


def test_normal_is_roughly_standard():
    x = synthetic.make_matrix(256, 256, "bf16", "normal", seed=3).float()
    assert abs(x.mean().item()) < 0.02 and abs(x.std().item() - 1.0) < 0.02


def test_pitched_ld_is_16_byte_multiple():
    assert synthetic.pitched_ld(8191, "f32") == 8192
    assert synthetic.pitched_ld(16383, "f16") == 16384
    assert synthetic.pitched_ld(64, "bf16") == 64
