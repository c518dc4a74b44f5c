"""Pins for the oracle's swizzle restatement and the lessons' size formulas."""
import re

import pytest

from oracle import smem, swizzle
from conftest import read_golden, read_golden_text


def _eval_layout(shape, stride, coord):
    """Evaluate a (nested) shape:stride layout at a nested coordinate."""
    if isinstance(shape, tuple):
        return sum(_eval_layout(s, d, c) for s, d, c in zip(shape, stride, coord))
    return coord * stride


def _parse_printed_layout(text):
    m = re.match(r"Sw<(\d+),(\d+),(\d+)> o smem_ptr\[(\d+)b\]\(unset\) o (.*)$", text)
    B, M, S, bits, layout = int(m[1]), int(m[2]), int(m[3]), int(m[4]), m[5]
    shape_txt, stride_txt = layout.split(":")
    to_tuple = lambda t: eval(t.replace("_", ""))  # noqa: E731  (digits, commas, parens)
    return (B, M, S), bits, to_tuple(shape_txt), to_tuple(stride_txt)


def test_printed_128x64_half_layout_matches_restatement():
    (B, M, S), bits, shape, stride = _parse_printed_layout(
        read_golden_text("smem_layout_128x64_f16.txt")[0])
    assert (B, M, S) == (3, 4, 3) and bits == 16
    esize = bits // 8
    seen = set()
    for r in range(128):
        for c in range(64):
            coord = ((r % 8, r // 8), (c, 0))
            elem = _eval_layout(shape, stride, coord)
            # the unswizzled layout is plain row-major with 64-element rows
            assert elem == r * 64 + c
            phys = swizzle.swizzle(B, M, S, elem * esize)
            assert phys == swizzle.box_offset(r, c, esize)
            seen.add(phys)
    assert len(seen) == 128 * 64


def test_sw128_is_a_bijection_on_a_16k_box():
    img = sorted(swizzle.sw128(o) for o in range(16384))
    assert img == list(range(16384))


def test_sw128_keeps_16_byte_units_and_row0():
    for o in range(16384):
        assert swizzle.sw128(o) & 15 == o & 15
        assert swizzle.sw128(o) >> 7 == o >> 7          # stays in its 128-B row
    assert [swizzle.sw128(o) for o in range(128)] == list(range(128))


def test_sw128_chunks_form_a_latin_square_per_1024_bytes():
    """Within each 8-row atom, a fixed logical chunk lands in 8 different
    physical chunks (so 8 rows read at the same column hit 8 different
    bank groups), and each row's chunks are a permutation."""
    for atom in range(4):
        for c in range(8):
            phys = {(swizzle.sw128(atom * 1024 + r * 128 + c * 16) >> 4) & 7 for r in range(8)}
            assert phys == set(range(8))
        for r in range(8):
            phys = {(swizzle.sw128(atom * 1024 + r * 128 + c * 16) >> 4) & 7 for c in range(8)}
            assert phys == set(range(8))
    # period 1024
    for o in range(4096):
        assert swizzle.sw128(o + 1024) == swizzle.sw128(o) + 1024


def test_smaller_atoms_from_the_lesson_list():
    # Swizzle<1,4,3> (32 B) and <2,4,3> (64 B): XOR one / two address bits
    assert swizzle.swizzle(1, 4, 3, 0x80) == 0x90
    assert swizzle.swizzle(2, 4, 3, 0x180) == 0x1B0
    assert swizzle.swizzle(0, 4, 3, 0x3F0) == 0x3F0       # no swizzle


def test_staged_image_of_a_box():
    rows = 16
    tile = bytes((i * 7 + 3) % 251 for i in range(rows * 128))
    img = swizzle.staged_image(tile, rows, 2)
    assert img[:128] == tile[:128]                        # row 0 unchanged
    assert img[128 + 16:128 + 32] == tile[128:128 + 16]   # row 1 chunk 0 -> chunk 1
    assert sorted(img) == sorted(tile)


@pytest.mark.parametrize("row", read_golden("lesson_sizes.txt"))
def test_lesson_sizes(row):
    q, tm, tn, es, st, value = row[0], *map(int, row[1:])
    if q == "single_tile_smem":
        assert smem.single_tile_smem(tm, tn, es) == value
    elif q == "tx_bytes":
        assert smem.tx_bytes(tm, tn, es) == value
    elif q == "tma_box_inner":
        assert 128 // es == value                        # one 128-byte swizzle row
    elif q == "tma_box_outer":
        assert tm == value
    elif q.startswith("pipeline_"):
        assert smem.pipeline_smem(st, tm, tn, es)[q[len("pipeline_"):]] == value
    else:
        pytest.fail(q)
