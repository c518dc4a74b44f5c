"""The read-bandwidth reference (tile_read_checksum): its XOR checksum of a
device buffer equals the oracle's fold of the same bytes, for sizes below one
vector per thread, ragged against the grid's stride, and above L2; argument
errors are refused on the host."""
import ctypes

import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
from mbarrier_async_tile_gb300 import C

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("nbytes", [16, 48, 4096, 16 * 1000003, 300 << 20])
def test_checksum_matches_oracle(nbytes):
    g = torch.Generator().manual_seed(nbytes % 1000)
    host = torch.randint(-2**31, 2**31 - 1, (nbytes // 4,), dtype=torch.int32, generator=g)
    dev = host.cuda()
    out = mbt.tile_read_checksum(dev)
    torch.cuda.synchronize()
    got = int(out.cpu().view(torch.int32)[0]) & 0xFFFFFFFF
    assert got == oracle.xor_fold(host)
    # twice: out is overwritten, not accumulated
    out = mbt.tile_read_checksum(dev, out)
    assert int(out.cpu()[0]) & 0xFFFFFFFF == got


def test_zero_bytes_and_argument_errors():
    out = torch.full((4,), 7, dtype=torch.int32, device="cuda")
    assert C.tile_read_checksum(None, 0, out.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert int(out[0]) == 0
    buf = torch.zeros(64, dtype=torch.uint8, device="cuda")
    assert C.tile_read_checksum(buf.data_ptr(), 24, out.data_ptr(), None) == -2   # not 16 x k
    assert C.tile_read_checksum(buf.data_ptr() + 8, 16, out.data_ptr(), None) == -2
    assert C.tile_read_checksum(buf.data_ptr(), 16, out.data_ptr() + 2, None) == -1
    assert C.tile_read_checksum(buf.data_ptr(), 16, None, None) == -1
    assert C.tile_read_checksum(None, 16, out.data_ptr(), None) == -1
