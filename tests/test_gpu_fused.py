"""GPU parity of tile_copy_rowsum (copy and row sums in one pass) against the
CPU oracle's copy (bit-exact) and binary64 row sums (1e-5 scaled), through
the C ABI: ragged edges, pitched buffers with untouched pads, 1-4 stages,
split and whole-band plans, the full-size ragged configurations."""
import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import ROWSUM_RTOL, bits, copy_case, rowsum_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


CASES = [
    # dtype, dist, M, N, tile_m, tile_n, stages, split
    ("f16", "uniform", 1, 1, 128, 64, 1, True),
    ("f16", "uniform", 300, 200, 128, 64, 3, True),
    ("bf16", "normal", 129, 1000, 64, 256, 2, True),
    ("bf16", "normal", 129, 1000, 64, 256, 2, False),
    ("f32", "uniform", 257, 33, 128, 32, 4, True),
    ("f32", "normal", 1000, 8191, 128, 32, 3, True),
    ("f16", "uniform", 1000, 700, 128, 64, 1, True),
    ("f16", "normal", 65, 20000, 8, 512, 2, True),
    ("bf16", "uniform", 4097, 300, 256, 64, 3, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_fused_matches_oracle(case):
    dtype, dist, M, N, tm, tn, st, split = case
    es = synthetic.ESIZE[dtype]
    src, dst, want = copy_case(dtype, M, N, seed=M * 3 + N, src_pad=16 // es,
                               dst_pad=32 // es, dist=dist)
    s, d = src.cuda(), dst.cuda()
    out = mbt.tile_copy_rowsum(s[:, :N], d[:, :N], None, tm, tn, st, split=split)
    code, info = mbt.tile_status()
    assert code == 0, info
    assert torch.equal(bits(d.cpu()), bits(want))
    worst, rel, _ = rowsum_errors(out, src[:, :N])
    assert worst <= ROWSUM_RTOL, (worst, rel)


def test_fused_equals_separate_calls_bitwise():
    """Same plan, same order: the fused row sums are the plain row sums."""
    x = synthetic.make_matrix(3000, 20000, "bf16", "normal", seed=8).cuda()
    y = torch.empty_like(x)
    a = mbt.tile_rowsum(x, None, 64, 256, 2)
    b = mbt.tile_copy_rowsum(x, y, None, 64, 256, 2)
    assert mbt.tile_status()[0] == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(y.view(torch.int16), x.view(torch.int16))


@pytest.mark.parametrize("fault", [1, 2])
def test_fused_stall_reports_timeout(fault):
    src, dst, want = copy_case("f16", 512, 1024, seed=3)
    s, d = src.cuda(), dst.cuda()
    mbt.tile_copy_rowsum(s, d, None, 128, 64, 3, max_ctas=4, fault=fault,
                         wait_budget_ns=20_000_000)
    code, info = mbt.tile_status()
    assert code == mbt.MBT_ERR_TIMEOUT, info
    d2 = dst.cuda()
    out = mbt.tile_copy_rowsum(s, d2, None, 128, 64, 3)
    assert mbt.tile_status()[0] == 0
    assert torch.equal(bits(d2.cpu()), bits(want))


FULL = [
    ("f32", 12289, 8191, 128, 32, 1005),
    ("f16", 24577, 16383, 128, 64, 1006),
]


@pytest.mark.parametrize("case", FULL, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}")
def test_full_size_ragged_configs(case):
    dtype, M, N, tm, tn, seed = case
    src, dst, want = copy_case(dtype, M, N, seed=seed)
    s, d = src.cuda(), dst.cuda()
    out = mbt.tile_copy_rowsum(s[:, :N], d[:, :N], None, tm, tn, 3)
    assert mbt.tile_status()[0] == 0
    assert torch.equal(bits(d.cpu()), bits(want))
    assert rowsum_errors(out, src[:, :N])[0] <= ROWSUM_RTOL
