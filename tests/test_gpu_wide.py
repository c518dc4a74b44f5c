"""The wide row- and column-sum kernels (more than 8 consumer warps, one CTA
per SM): the row sum's default where only one CTA fits an SM and 8 warps would
give each thread two rounds of a tile row's chunks (fp32 128 x 128 tiles),
else when the caller asks for more than 8 warps, as for the column sum.  GPU
parity against the binary64 oracle on split and unsplit plans, ragged shapes
and explicit warp counts above 8, sums bit-identical from call to call."""
import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import ROWSUM_RTOL, colsum_errors, rowsum_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


def _plan(op, M, N, tm, tn, st, dtype, **opt):
    """The plan the device call makes (tile_plan_device: the real device's
    occupancy; a 4-stage ring of 32 KB tiles leaves room for one CTA per SM)."""
    return mbt.tile_plan_device(op, M, N, tm, tn, st, dtype, **opt)


CASES = [
    # dtype, dist, M, N, tile_m, tile_n, stages, opts
    ("bf16", "normal", 2048, 65536, 64, 256, 4, {"consumer_warps": 16}),
    ("bf16", "normal", 2048, 65536, 64, 256, 4, {"consumer_warps": 16, "split": False}),
    ("f16", "uniform", 1000, 30001, 64, 256, 4, {"consumer_warps": 16}),   # ragged M and N
    ("f32", "uniform", 777, 20000, 128, 128, 3, {}),    # 512-byte rows, 64 KB tiles: the default
    ("bf16", "uniform", 4097, 3000, 32, 512, 5, {"consumer_warps": 16}),   # 1 KB tile rows
    ("f16", "normal", 3000, 9000, 128, 64, 2, {"consumer_warps": 12}),
    ("bf16", "normal", 3000, 9000, 256, 64, 3, {"consumer_warps": 16, "ctas_per_sm": 1}),
    ("bf16", "normal", 3000, 9000, 64, 256, 2, {"consumer_warps": 10}),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c[:7])) +
                         "".join(f"-{k}{v}" for k, v in c[7].items()))
def test_wide_rowsum_matches_oracle(case):
    dtype, dist, M, N, tm, tn, st, opt = case
    ld = synthetic.pitched_ld(N, dtype)           # a 16-byte pitch: the tiled kernels
    x = synthetic.make_matrix(M, N, dtype, dist, seed=M + N, ld=ld)
    xd = x.cuda()[:, :N]
    kw = {k: v for k, v in opt.items() if k != "split"}
    plan = _plan(mbt.OP_ROWSUM, M, N, tm, tn, st, synthetic.DTYPES[dtype], ld_src=ld, **kw)
    assert plan["flat"] == 0
    assert plan["consumer_warps"] == opt.get("consumer_warps", 16)
    a = mbt.tile_rowsum(xd, None, tm, tn, st, **opt)
    b = mbt.tile_rowsum(xd, None, tm, tn, st, **opt)
    assert mbt.tile_status()[0] == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    worst, rel, _ = rowsum_errors(a, x[:, :N])
    assert worst <= ROWSUM_RTOL, (worst, rel)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c[:7])) +
                         "".join(f"-{k}{v}" for k, v in c[7].items()))
def test_wide_colsum_matches_oracle(case):
    """16 consumer warps unless the case names a count (128-byte tile rows with
    more than 8 warps: strips walked one at a time)."""
    dtype, dist, M, N, tm, tn, st, opt = case
    opt = dict(opt)
    opt.setdefault("consumer_warps", 16)
    ld = synthetic.pitched_ld(N, dtype)
    x = synthetic.make_matrix(M, N, dtype, dist, seed=M + N + 1, ld=ld)
    xd = x.cuda()[:, :N]
    a = mbt.tile_colsum(xd, None, tm, tn, st, **opt)
    b = mbt.tile_colsum(xd, None, tm, tn, st, **opt)
    assert mbt.tile_status()[0] == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    worst, rel, _ = colsum_errors(a, x[:, :N])
    assert worst <= ROWSUM_RTOL, (worst, rel)


def test_wide_full_size_colsum_sampled():
    """bf16 8192 x 65536 at 4 stages (the column-sum sweep point): sampled
    column blocks against the oracle."""
    M, N = 8192, 65536
    x = synthetic.make_matrix(M, N, "bf16", "normal", seed=1004, draw_on="cuda:0")
    assert _plan(mbt.OP_COLSUM, M, N, 64, 256, 4, torch.bfloat16,
                 consumer_warps=16)["threads"] == 32 * 18
    out = mbt.tile_colsum(x, None, 64, 256, 4, consumer_warps=16)
    assert mbt.tile_status()[0] == 0
    g = torch.Generator().manual_seed(11)
    for c0 in [0, N - 256] + (torch.randperm(N // 8, generator=g)[:16] * 8).tolist():
        w = 256 if c0 in (0, N - 256) else 8
        block = x[:, c0:c0 + w].cpu().contiguous()
        assert colsum_errors(out[c0:c0 + w], block)[0] <= ROWSUM_RTOL, c0


def test_device_plan_of_the_sweep_points():
    """tile_plan_device on the bench's row-sum tiles: 2 CTAs of 8 consumer
    warps per SM at 2 stages (bands split), one CTA of 8 per SM at 4."""
    sms = mbt.tile_device_info()["num_sms"]
    p2 = _plan(mbt.OP_ROWSUM, 8192, 65536, 64, 256, 2, torch.bfloat16)
    assert p2["grid"] == 2 * sms and p2["consumer_warps"] == 8 and p2["split"] == 1
    p4 = _plan(mbt.OP_ROWSUM, 8192, 65536, 64, 256, 4, torch.bfloat16)
    assert p4["grid"] == sms and p4["consumer_warps"] == 8
    whole = _plan(mbt.OP_ROWSUM, 8192, 65536, 64, 256, 2, torch.bfloat16, no_split=1)
    assert whole["split"] == 0 and whole["grid"] == 128
