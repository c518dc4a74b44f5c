"""Pins of oracle.xor_fold (the read-bandwidth reference's checksum) against
what the definition fixes without the oracle: byte order of a word, a lone
word, words that cancel in pairs, and a pure-Python fold of tiny buffers."""
import functools
import operator

import torch

import oracle


def _bytes(values):
    return torch.tensor(values, dtype=torch.uint8)


def test_empty_and_word_byte_order():
    assert oracle.xor_fold(torch.empty(0, dtype=torch.uint8)) == 0
    assert oracle.xor_fold(_bytes([1, 0, 0, 0])) == 1                 # little-endian
    assert oracle.xor_fold(_bytes([0, 0, 0, 1])) == 0x0100_0000
    assert oracle.xor_fold(_bytes([0x78, 0x56, 0x34, 0x12])) == 0x1234_5678


def test_lone_word_anywhere():
    for n in (1, 2, 7, 64):
        for k in range(n):
            buf = torch.zeros(4 * n, dtype=torch.uint8)
            buf[4 * k:4 * k + 4] = _bytes([0xEF, 0xBE, 0xAD, 0xDE])
            assert oracle.xor_fold(buf) == 0xDEAD_BEEF, (n, k)


def test_words_in_pairs_cancel():
    g = torch.Generator().manual_seed(3)
    w = torch.randint(0, 256, (100, 4), dtype=torch.uint8, generator=g)
    buf = torch.cat([w, w.flip(0)]).reshape(-1)
    assert oracle.xor_fold(buf) == 0
    buf2 = buf.clone()
    buf2[5] ^= 0x40                      # one flipped bit in word 1 shows up
    assert oracle.xor_fold(buf2) == 0x40 << 8


def test_matches_a_python_fold_of_tiny_buffers():
    g = torch.Generator().manual_seed(4)
    for n in (1, 3, 16, 257):
        buf = torch.randint(0, 256, (4 * n,), dtype=torch.uint8, generator=g)
        raw = bytes(buf.tolist())
        words = [int.from_bytes(raw[4 * k:4 * k + 4], "little") for k in range(n)]
        assert oracle.xor_fold(buf) == functools.reduce(operator.xor, words, 0), n


def test_any_dtype_view_of_the_same_bytes():
    g = torch.Generator().manual_seed(5)
    buf = torch.randint(0, 256, (4096,), dtype=torch.uint8, generator=g)
    want = oracle.xor_fold(buf)
    for dt in (torch.int16, torch.float32, torch.bfloat16):
        assert oracle.xor_fold(buf.view(dt)) == want
