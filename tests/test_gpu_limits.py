"""Shapes at the coordinate limits: bulk tensor copies take 32-bit element
coordinates, so the library accepts M, N <= 2^31 - 1.  A very wide and a very
tall matrix (8.6 and 34 GB) through copy, row sum and column sum, checked
against the oracle on sampled rows and columns (first, last, around 2^31
elements and the middle).  About 80 GB of device memory at most."""
import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import ROWSUM_RTOL, bits, colsum_errors, rowsum_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


def test_wide_matrix_at_the_column_limit():
    M, N = 2, (1 << 31) - 64                     # bf16, 64 x 256 tiles: 8.4 M column strips
    x = synthetic.make_matrix(M, N, "bf16", "uniform", seed=91, draw_on="cuda:0")
    y = torch.empty_like(x)
    mbt.tile_copy(x, y, 64, 256, 3)
    rows = mbt.tile_rowsum(x, None, 64, 256, 2)
    cols = mbt.tile_colsum(x, None, 64, 256, 2)
    assert mbt.tile_status()[0] == 0
    for c0 in (0, N // 2 - 100, (1 << 30) - 100, N - 300):
        blk = x[:, c0:c0 + 300].cpu()
        assert torch.equal(bits(y[:, c0:c0 + 300].cpu()), bits(blk)), c0
        assert colsum_errors(cols[c0:c0 + 300], blk.contiguous())[0] <= ROWSUM_RTOL, c0
    assert rowsum_errors(rows, x.cpu())[0] <= ROWSUM_RTOL
    del x, y, cols
    torch.cuda.empty_cache()


def test_tall_matrix_at_the_row_limit():
    M, N = (1 << 31) - 1, 8                      # fp16 rows of 16 bytes: one chunk each
    x = synthetic.make_matrix(M, N, "f16", "uniform", seed=92, draw_on="cuda:0")
    y = torch.empty_like(x)
    mbt.tile_copy(x, y, 128, 64, 3)
    rows = mbt.tile_rowsum(x, None, 128, 64, 2, split=False)
    assert mbt.tile_status()[0] == 0
    for r0 in (0, M // 2, (1 << 30) - 500, M - 1000):
        blk = x[r0:r0 + 1000].cpu()
        assert torch.equal(bits(y[r0:r0 + 1000].cpu()), bits(blk)), r0
        assert rowsum_errors(rows[r0:r0 + 1000], blk)[0] <= ROWSUM_RTOL, r0
    del x, y, rows
    torch.cuda.empty_cache()
