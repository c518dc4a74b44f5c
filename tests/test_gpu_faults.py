"""Bounded waits: a pipeline that stalls by construction (the two deadlocks the
lessons describe, injected from the host) must end with MBT_ERR_TIMEOUT in the
status word instead of hanging, and leave the context usable.  No bulk copy is
in flight when these kernels return (the producer drains its own copies)."""
import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
from helpers import bits, copy_case

pytestmark = pytest.mark.gpu

BUDGET_NS = 20_000_000   # 20 ms per wait


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("fault", [1, 2])
@pytest.mark.parametrize("op", ["copy", "copy_bulk", "rowsum"])
def test_stalled_pipeline_reports_timeout(fault, op):
    src, dst, want = copy_case("f16", 512, 1024, seed=3)
    s, d = src.cuda(), dst.cuda()
    if op.startswith("copy"):
        mbt.tile_copy(s, d, 128, 64, 3, max_ctas=4, fault=fault, wait_budget_ns=BUDGET_NS,
                      store_mode=1 if op == "copy_bulk" else 0)
    else:
        mbt.tile_rowsum(s, None, 128, 64, 3, max_ctas=4, fault=fault, wait_budget_ns=BUDGET_NS)
    code, info = mbt.tile_status()
    assert code == mbt.MBT_ERR_TIMEOUT, info
    assert 0 <= info[1] < 4
    # fault 1: the producer's first wait; fault 2: a wait blocked by a missing release
    if fault == 1:
        assert info[3] in (0, 1, 2, 3)
    # the status word was cleared, and the context still works
    assert mbt.tile_status()[0] == 0
    d2 = dst.cuda()
    mbt.tile_copy(s, d2, 128, 64, 3)
    assert mbt.tile_status()[0] == 0
    assert torch.equal(bits(d2.cpu()), bits(want))
    out = mbt.tile_rowsum(s, None, 128, 64, 3)
    assert mbt.tile_status()[0] == 0
