"""Row sums with a full/empty barrier pair per (stage, 128-byte box)
(pipeline=3; the default at up to 2 stages), wherever each consumer warp
reads a single box.  The sums must equal,
bit for bit, those of the stage-wide barrier pairs (pipeline=2) -- the
barrier layout changes when a box may be read, not what is added in which
order -- and match the binary64 oracle; stalls end in MBT_ERR_TIMEOUT."""
import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import DTYPES, ROWSUM_RTOL, copy_case, rowsum_errors
from oracle.pipeline_state import sequence

pytestmark = pytest.mark.gpu

BUDGET_NS = 20_000_000   # 20 ms per wait


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


def box_barriers(M, N, tm, tn, st, torch_dtype, W, ld=0):
    info = mbt.tile_device_info()
    return mbt.tile_plan(mbt.OP_ROWSUM, M, N, tm, tn, st, torch_dtype,
                         num_sms=info["num_sms"], smem_optin=info["smem_optin"], fit_per_sm=1,
                         consumer_warps=W, ld_src=ld, pipeline=3)["box_barriers"]


CASES = [
    # dtype, dist, M, N, tile_m, tile_n, stages, consumer_warps, split
    ("bf16", "normal", 3000, 20000, 64, 256, 2, 8, True),     # 4 boxes, 2 warps each
    ("bf16", "normal", 3000, 20000, 64, 256, 3, 8, False),
    ("bf16", "uniform", 777, 9001, 32, 256, 2, 4, True),      # 4 boxes, 1 warp each
    ("f16", "normal", 1025, 30000, 128, 128, 3, 8, True),     # 2 boxes, 4 warps each
    ("f16", "uniform", 4097, 777, 32, 512, 2, 8, True),       # 8 boxes, 1 warp each
    ("f32", "normal", 500, 12345, 32, 128, 4, 8, True),       # 4 boxes of fp32
    ("bf16", "normal", 64, 256, 64, 256, 1, 8, True),         # one tile, one stage
    ("f16", "uniform", 1, 70000, 128, 128, 2, 8, True),       # one row, ragged tail
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_box_barriers_bitwise_equal_stage_barriers(case):
    dtype, dist, M, N, tm, tn, st, W, split = case
    ld = synthetic.pitched_ld(N, dtype)
    assert box_barriers(M, N, tm, tn, st, DTYPES[dtype], W, ld) == 1
    x = synthetic.make_matrix(M, N, dtype, dist, seed=M ^ N, ld=ld)
    xd = x.cuda()[:, :N]
    a = mbt.tile_rowsum(xd, None, tm, tn, st, consumer_warps=W, split=split, pipeline=3)
    b = mbt.tile_rowsum(xd, None, tm, tn, st, consumer_warps=W, split=split, pipeline=2)
    c = mbt.tile_rowsum(xd, None, tm, tn, st, consumer_warps=W, split=split)
    code, info = mbt.tile_status()
    assert code == 0, info
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(a.view(torch.int32), c.view(torch.int32))
    worst, rel, _ = rowsum_errors(a, x[:, :N])
    assert worst <= ROWSUM_RTOL, (worst, rel)


def test_box_barriers_equal_fused_sums():
    """The fused kernel keeps stage-wide barriers (its store warp reads whole
    stages) and sums in the same order."""
    x = synthetic.make_matrix(2000, 40000, "bf16", "normal", seed=21).cuda()
    y = torch.empty_like(x)
    assert box_barriers(2000, 40000, 64, 256, 2, torch.bfloat16, 8) == 1
    a = mbt.tile_rowsum(x, None, 64, 256, 2, consumer_warps=8, max_ctas=152, pipeline=3)
    b = mbt.tile_copy_rowsum(x, y, None, 64, 256, 2, consumer_warps=8, max_ctas=152)
    assert mbt.tile_status()[0] == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(y.view(torch.int16), x.view(torch.int16))


@pytest.mark.parametrize("fault", [1, 2])
def test_box_barrier_stall_reports_timeout(fault):
    x = synthetic.make_matrix(512, 4096, "bf16", "normal", seed=5)
    xd = x.cuda()
    assert box_barriers(512, 4096, 64, 256, 3, torch.bfloat16, 8) == 1
    mbt.tile_rowsum(xd, None, 64, 256, 3, consumer_warps=8, max_ctas=4, fault=fault,
                    wait_budget_ns=BUDGET_NS, pipeline=3)
    code, info = mbt.tile_status()
    assert code == mbt.MBT_ERR_TIMEOUT, info
    assert 0 <= info[1] < 4
    assert mbt.tile_status()[0] == 0
    out = mbt.tile_rowsum(xd, None, 64, 256, 3, consumer_warps=8)
    assert mbt.tile_status()[0] == 0
    assert rowsum_errors(out, x)[0] <= ROWSUM_RTOL
    src, dst, want = copy_case("f16", 256, 512, seed=6)
    d = dst.cuda()
    mbt.tile_copy(src.cuda(), d, 128, 64, 2)
    assert mbt.tile_status()[0] == 0


def test_log_of_one_cta_box_barrier_pipeline():
    """Both roles still walk (stage, phase) in the pipeline's order: the
    producer starts at phase 1 (free buffers), the consumers at phase 0."""
    x = synthetic.make_matrix(64, 4096, "bf16", "uniform", seed=13)
    log = torch.zeros(2 * 16 * 4, dtype=torch.int32, device="cuda")
    assert box_barriers(64, 4096, 64, 256, 3, torch.bfloat16, 8) == 1
    out = mbt.tile_rowsum(x.cuda(), None, 64, 256, 3, consumer_warps=8, max_ctas=1,
                          split=False, log=log, pipeline=3)
    assert mbt.tile_status()[0] == 0
    assert rowsum_errors(out, x)[0] <= ROWSUM_RTOL
    rec = log.view(2, 16, 4).cpu()
    assert [(s, p) for _, s, p, _ in rec[0].tolist()] == sequence(3, 1, 16)
    assert [(s, p) for _, s, p, _ in rec[1].tolist()] == sequence(3, 0, 16)
    assert [t for *_, t in rec[1].tolist()] == list(range(16))
