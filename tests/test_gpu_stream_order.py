"""Stream order across calls.  The pipeline kernels are launched with
programmatic stream serialization, so a kernel may be launched while the
previous kernel of its stream is still completing; it must read and write
global memory only after that kernel has finished.  These chains on one
stream would give wrong results if it did not: each call reads what the call
before it wrote (read after write), or overwrites what the call before it
was still reading (write after read), with sizes at which one kernel's
launch overlaps the previous one's last tiles."""
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


def test_read_after_write_chain():
    """x -> y (copy) -> z (copy) -> row and column sums of z, and the row sums
    of z's elements read as rows of 8191 (a pitch that is not a multiple of
    16 bytes: the 1-D bulk-copy kernel), all queued before any result is
    looked at, three times over with new data in x each time."""
    M, N, NF = 4096, 8192, 8191
    s = torch.cuda.Stream()
    ws = torch.zeros(8 << 20, dtype=torch.uint8, device="cuda")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    z = torch.empty_like(y)
    zf = z.view(-1)[:M * NF].view(M, NF)
    rows = torch.empty(M, device="cuda")
    rows_f = torch.empty(M, device="cuda")
    cols = torch.empty(N, device="cuda")
    x = torch.empty_like(y)
    torch.cuda.synchronize()
    for seed in (11, 12, 13):
        src = synthetic.make_matrix(M, N, "bf16", "normal", seed)
        with torch.cuda.stream(s):
            x.copy_(src)
            mbt.tile_copy(x, y, 128, 64, 3, stream=s)
            mbt.tile_copy(y, z, 64, 256, 2, stream=s)
            mbt.tile_rowsum(z, rows, 64, 256, 2, workspace=ws, stream=s)
            mbt.tile_colsum(z, cols, 64, 256, 2, workspace=ws, stream=s)
            mbt.tile_rowsum(zf, rows_f, 128, 64, 2, stream=s)
        s.synchronize()
        assert mbt.tile_status(s)[0] == 0
        assert torch.equal(bits(z.cpu()), bits(src))
        assert rowsum_errors(rows, src)[0] <= ROWSUM_RTOL
        assert colsum_errors(cols, src)[0] <= ROWSUM_RTOL
        assert rowsum_errors(rows_f, src.view(-1)[:M * NF].view(M, NF))[0] <= ROWSUM_RTOL


def test_write_after_read_chain():
    """Each call overwrites the buffer the call before it read: the sums and
    the copy must see the old contents, never the new."""
    M, N = 4096, 8192
    s = torch.cuda.Stream()
    ws = torch.zeros(8 << 20, dtype=torch.uint8, device="cuda")
    a_h = synthetic.make_matrix(M, N, "f16", "uniform", 21)
    b_h = synthetic.make_matrix(M, N, "f16", "uniform", 22)
    a = a_h.cuda()
    b = b_h.cuda()
    a2 = a_h.cuda()
    c = torch.empty_like(a)
    rows_a = torch.empty(M, device="cuda")
    rows_b = torch.empty(M, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        mbt.tile_rowsum(a, rows_a, 64, 256, 2, workspace=ws, stream=s)   # reads a
        mbt.tile_copy(b, a, 128, 64, 3, stream=s)                        # then overwrites a
        mbt.tile_copy(a, c, 128, 64, 3, stream=s)                        # reads the new a
        mbt.tile_rowsum(c, rows_b, 64, 256, 2, workspace=ws, stream=s)   # reads c
        mbt.tile_copy(a2, c, 128, 64, 3, stream=s)                       # then overwrites c
    s.synchronize()
    assert mbt.tile_status(s)[0] == 0
    assert rowsum_errors(rows_a, a_h)[0] <= ROWSUM_RTOL
    assert rowsum_errors(rows_b, b_h)[0] <= ROWSUM_RTOL
    assert torch.equal(bits(a.cpu()), bits(b_h))
    assert torch.equal(bits(c.cpu()), bits(a_h))
