"""Shared-memory and transaction-byte formulas of the two lessons.

Test infrastructure (see ``oracle/__init__.py``).

* "cute(11) Hopper TMA copy", §3.3 and the launch in its main program: one
  tile of data followed by one 8-byte mbarrier and 8 more bytes of slack; the
  barrier expects the whole tile's bytes.
* "cute(12) async_pipeline", §5 and §6.4: a structure holding first the
  pipeline's barriers (a full and an empty barrier per stage, 8 bytes each),
  then the stage buffers aligned to 128 bytes; the launch rounds the
  structure's size up to a multiple of 128.
"""
from __future__ import annotations

MBARRIER_BYTES = 8


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def tx_bytes(tile_m: int, tile_n: int, esize: int) -> int:
    """Bytes one tile's bulk load delivers, registered with expect_tx."""
    return tile_m * tile_n * esize


def single_tile_smem(tile_m: int, tile_n: int, esize: int) -> int:
    """Dynamic shared memory of the single-tile copy kernel."""
    return tx_bytes(tile_m, tile_n, esize) + MBARRIER_BYTES + 8


def pipeline_smem(stages: int, tile_m: int, tile_n: int, esize: int) -> dict:
    """Layout of the multi-stage pipeline's shared storage."""
    barriers = 2 * stages * MBARRIER_BYTES
    data_offset = round_up(barriers, 128)
    data = stages * tx_bytes(tile_m, tile_n, esize)
    total = round_up(data_offset + data, 128)
    return {"barriers": barriers, "data_offset": data_offset, "data": data,
            "total": total}
