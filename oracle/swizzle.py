"""Shared-memory swizzle of bulk-tensor tiles, restated on byte offsets.

Test infrastructure (see ``oracle/__init__.py``).

Source: "cute(11) Hopper TMA copy", §2.2: the staged tile uses the K-major
128-byte swizzle atom, printed by the lesson as ``Sw<3,4,3>`` composed with a
16-bit shared-memory pointer and the layout
``((_8,_16),(_64,_1)):((_64,_512),(_1,_0))`` for a 128 x 64 half tile; the
copy engine needs the swizzle's base parameter M >= 4 (16-byte units); the
32/64/128-byte atoms are Swizzle<1,4,3>, <2,4,3> and <3,4,3>.

Reading: a Swizzle<B, M, S> acting on a byte address keeps the low M bits (one
16-byte unit when M = 4), and XORs the B bits that start S places above the
unit index into the unit index.  For the 128-byte atom that is
``offset ^ (((offset >> 7) & 7) << 4)``: the 16-byte chunk number of a 128-byte
row is XORed with the row number modulo 8, repeating every 1024 bytes.
"""
from __future__ import annotations


def swizzle(B: int, M: int, S: int, offset: int) -> int:
    """Apply Swizzle<B, M, S> to one byte offset."""
    if B < 0 or M < 0 or S < B:
        raise ValueError("bad swizzle parameters")
    source_mask = ((1 << B) - 1) << (M + S)
    return offset ^ ((offset & source_mask) >> S)


def sw128(offset: int) -> int:
    """The 128-byte swizzle used for every staged tile."""
    return swizzle(3, 4, 3, offset)


def box_offset(row: int, col: int, esize: int, row_bytes: int = 128) -> int:
    """Byte offset, inside one 1024-byte-aligned box buffer, of element
    (row, col) of a box whose rows are ``row_bytes`` (128) long."""
    if col * esize >= row_bytes:
        raise ValueError("column outside the box row")
    return sw128(row * row_bytes + col * esize)


def staged_image(tile: bytes, rows: int, esize: int) -> bytes:
    """Raw shared-memory bytes of one box after a swizzled bulk load of
    ``tile`` (``rows`` rows of 128 bytes, row-major, unswizzled)."""
    if len(tile) != rows * 128:
        raise ValueError("tile must be rows x 128 bytes")
    out = bytearray(len(tile))
    for r in range(rows):
        for c in range(128 // esize):
            src = r * 128 + c * esize
            dst = box_offset(r, c, esize)
            out[dst:dst + esize] = tile[src:src + esize]
    return bytes(out)
