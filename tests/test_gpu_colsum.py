"""GPU parity of tile_colsum against the binary64 CPU oracle, through the C
ABI: fp32 column sums within 1e-5 x max(|sum|, sqrt(sum of squares)) per
column, exact on exactly representable cases, run-to-run bit-identical; pad
columns (NaN patterns) never read; stalls end in MBT_ERR_TIMEOUT."""
import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import ROWSUM_RTOL, colsum_errors, rowsum_errors
from oracle.pipeline_state import sequence

pytestmark = pytest.mark.gpu

BUDGET_NS = 20_000_000   # 20 ms per wait


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


def run_colsum(x_h, N, *args, **kw):
    x = x_h.cuda()
    out = mbt.tile_colsum(x[:, :N], None, *args, **kw)
    code, info = mbt.tile_status()
    assert code == 0, info
    return out


CASES = [
    # dtype, dist, M, N, tile_m, tile_n, stages, consumer_warps, split
    ("bf16", "normal", 200, 1000, 64, 256, 3, 0, True),     # ragged M and N
    ("bf16", "normal", 200, 1000, 64, 256, 3, 0, False),
    ("f16", "uniform", 1, 1, 128, 64, 1, 0, True),
    ("f16", "uniform", 4100, 300, 128, 64, 4, 0, True),
    ("f32", "uniform", 8191, 257, 128, 32, 3, 0, True),
    ("f32", "normal", 33, 1000, 16, 64, 2, 0, True),        # fp32, 2 boxes
    ("f16", "normal", 20000, 65, 8, 512, 2, 2, True),       # 8 boxes, one thread per chunk
    ("bf16", "uniform", 300, 4097, 256, 64, 5, 0, True),
    ("f16", "uniform", 70000, 37, 32, 128, 6, 0, False),    # long strips, one CTA each
    ("bf16", "normal", 5000, 3000, 64, 256, 2, 4, True),
    ("f16", "uniform", 999, 777, 64, 64, 2, 3, True),       # 12 threads per chunk column
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_colsum_matches_oracle(case):
    dtype, dist, M, N, tm, tn, st, W, split = case
    ld = synthetic.pitched_ld(N, dtype) + 16 // synthetic.ESIZE[dtype]
    x = synthetic.make_matrix(M, N, dtype, dist, seed=M + 3 * N, ld=ld)
    out = run_colsum(x, N, tm, tn, st, consumer_warps=W, split=split)
    worst, rel, _ = colsum_errors(out, x[:, :N])
    assert worst <= ROWSUM_RTOL, (worst, rel)


def test_all_ones_exact_and_empty_shapes():
    x = torch.ones(5000, 304, dtype=torch.bfloat16)     # 608-byte rows: 16-byte pitch
    out = run_colsum(x, 300, 64, 256, 2)
    assert out.cpu().tolist() == [5000.0] * 300
    with pytest.raises(mbt.MbtError) as e:              # a dense 600-byte pitch is refused
        mbt.tile_colsum(torch.ones(50, 300, dtype=torch.bfloat16, device="cuda"))
    assert e.value.code == -2
    z = mbt.tile_colsum(torch.empty(0, 7, dtype=torch.float16, device="cuda"), None, 64, 64, 2)
    assert mbt.tile_status()[0] == 0
    assert z.cpu().tolist() == [0.0] * 7
    e = mbt.tile_colsum(torch.empty(7, 0, dtype=torch.float16, device="cuda"), None, 64, 64, 2)
    assert mbt.tile_status()[0] == 0 and e.numel() == 0


def test_repeat_calls_bit_identical_and_workspace_left_zero():
    ws = torch.zeros(1 << 22, dtype=torch.uint8, device="cuda")
    for M, N in ((3000, 20000), (700, 65536), (8192, 1024)):
        x = synthetic.make_matrix(M, N, "bf16", "normal", seed=M).cuda()
        a = mbt.tile_colsum(x, None, 64, 256, 2, workspace=ws)
        b = mbt.tile_colsum(x, None, 64, 256, 2, workspace=ws)
        assert mbt.tile_status()[0] == 0
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
        assert int(ws.count_nonzero()) == 0
        assert colsum_errors(a, x.cpu())[0] <= ROWSUM_RTOL


def test_log_of_one_cta_pipeline_walks_down_the_strips():
    x = synthetic.make_matrix(1024, 128, "f16", "uniform", seed=12)
    log = torch.zeros(2 * 16 * 4, dtype=torch.int32, device="cuda")
    out = run_colsum(x, 128, 128, 64, 3, consumer_warps=4, max_ctas=1, split=False, log=log)
    assert colsum_errors(out, x)[0] <= ROWSUM_RTOL
    rec = log.view(2, 16, 4).cpu()
    assert [(s, p) for _, s, p, _ in rec[0].tolist()] == sequence(3, 1, 16)
    assert [(s, p) for _, s, p, _ in rec[1].tolist()] == sequence(3, 0, 16)
    # tile numbers in strip-major order: strip 0's 8 bands, then strip 1's
    assert [t for *_, t in rec[1].tolist()] == list(range(16))


@pytest.mark.parametrize("fault", [1, 2])
@pytest.mark.parametrize("tile", [(64, 256), (128, 64)], ids=["one-strip", "strip-pairs"])
def test_stalled_pipeline_reports_timeout(fault, tile):
    x = synthetic.make_matrix(512, 4096, "bf16", "normal", seed=5)
    xd = x.cuda()
    mbt.tile_colsum(xd, None, *tile, 3, max_ctas=4, fault=fault, wait_budget_ns=BUDGET_NS)
    code, info = mbt.tile_status()
    assert code == mbt.MBT_ERR_TIMEOUT, info
    assert 0 <= info[1] < 4
    assert mbt.tile_status()[0] == 0
    # The stalled call used the library's own workspace of this stream and may
    # have left strip tickets set; the calls after it start from zeroed ones.
    for _ in range(3):
        out = mbt.tile_colsum(xd, None, *tile, 3, max_ctas=4)
        assert mbt.tile_status()[0] == 0
        assert colsum_errors(out, x)[0] <= ROWSUM_RTOL


def test_log_of_strip_pairs_walks_band_by_band():
    """128-byte tiles with a workspace: strips are taken in pairs, band by
    band (5 strips: the last group is a single strip).  The sums are right
    whichever CTA ends where in a pair, and CTA 0's producer and consumer
    walk the same order positions."""
    M, N, tm, tn = 512, 320, 128, 64            # 4 bands x 5 strips (last pair: one strip)
    x = synthetic.make_matrix(M, N, "f16", "uniform", seed=14)
    info = mbt.tile_device_info()
    plan = mbt.tile_plan(mbt.OP_COLSUM, M, N, tm, tn, 2, torch.float16,
                         num_sms=info["num_sms"], smem_optin=info["smem_optin"], fit_per_sm=1,
                         with_workspace=True, max_ctas=3)
    assert plan["split"] == 1 and plan["col_group"] == 2 and plan["grid"] == 3
    log = torch.zeros(2 * 32 * 4, dtype=torch.int32, device="cuda")
    out = mbt.tile_colsum(x.cuda(), None, tm, tn, 2, max_ctas=3, log=log)
    assert mbt.tile_status()[0] == 0
    assert colsum_errors(out, x)[0] <= ROWSUM_RTOL
    rec = log.view(2, 32, 4).cpu()
    T = 20                                       # CTA 0 owns positions [0, 20 / 3)
    mine = [t for *_, t in rec[0].tolist()][:T // 3]
    assert mine == list(range(T // 3))
    assert [t for *_, t in rec[1].tolist()][:T // 3] == mine
    # every CTA count splits the pairs differently; all give the same sums
    for ctas in (1, 2, 4, 7, 20):
        o2 = mbt.tile_colsum(x.cuda(), None, tm, tn, 2, max_ctas=ctas)
        assert mbt.tile_status()[0] == 0
        assert colsum_errors(o2, x)[0] <= ROWSUM_RTOL, ctas


def test_full_size_sampled_columns_and_totals():
    """bf16 8192 x 65536 (1 GiB), 64 x 256 tiles, 2 stages: the default
    launch.  Sampled column blocks (first, last and scattered strips) against
    the oracle; the sum of all column sums against the sum of all row sums."""
    M, N = 8192, 65536
    x = synthetic.make_matrix(M, N, "bf16", "normal", seed=1004, draw_on="cuda:0")
    out = mbt.tile_colsum(x, None, 64, 256, 2)
    rows = mbt.tile_rowsum(x, None, 64, 256, 2)
    assert mbt.tile_status()[0] == 0
    g = torch.Generator().manual_seed(7)
    starts = [0, N - 256] + (torch.randperm(N // 8, generator=g)[:24] * 8).tolist()
    for c0 in starts:
        w = 256 if c0 in (0, N - 256) else 8
        block = x[:, c0:c0 + w].cpu().contiguous()
        worst, rel, _ = colsum_errors(out[c0:c0 + w], block)
        assert worst <= ROWSUM_RTOL, (c0, worst, rel)
    total_c = out.double().sum().item()
    total_r = rows.double().sum().item()
    scale = x.float().pow(2).sum().sqrt().item()
    assert abs(total_c - total_r) <= 1e-5 * scale


def test_ragged_full_size_configs():
    """fp32 12289 x 8191 and fp16 24577 x 16383, pitched rows: every column.
    Their tiles are 128 bytes wide, so strips are walked in pairs."""
    info = mbt.tile_device_info()
    for dtype, M, N, tm, tn, seed in (("f32", 12289, 8191, 128, 32, 1005),
                                      ("f16", 24577, 16383, 128, 64, 1006)):
        ld = synthetic.pitched_ld(N, dtype)
        plan = mbt.tile_plan(mbt.OP_COLSUM, M, N, tm, tn, 3, synthetic.DTYPES[dtype],
                             num_sms=info["num_sms"], smem_optin=info["smem_optin"],
                             fit_per_sm=2, with_workspace=True, ld_src=ld)
        assert plan["split"] == 1 and plan["col_group"] == 2
        x = synthetic.make_matrix(M, N, dtype, "uniform", seed, ld=ld)
        out = mbt.tile_colsum(x.cuda()[:, :N], None, tm, tn, 3)
        assert mbt.tile_status()[0] == 0
        worst, rel, _ = colsum_errors(out, x[:, :N])
        assert worst <= ROWSUM_RTOL, (dtype, worst, rel)


@pytest.mark.parametrize("case", [("bf16", 2048, 4096, 64, 256), ("bf16", 2048, 4096, 128, 128),
                                  ("f32", 2048, 2048, 64, 64)],
                         ids=["512-byte-strips", "256-byte-strips", "256-byte-f32-strips"])
def test_wide_strip_pairs_where_one_cta_per_sm_runs(case):
    """With one CTA per SM (here asked for: ctas_per_sm=1, 4 stages), strips of
    256 and 512 bytes are walked in pairs.  The grid (one CTA per SM) is large
    against these shapes, so each strip has 10-19 contributors: the last one
    adds more than 8 slots per column, a pair's 512 or 256 columns in chunks of
    128.  Every column against the oracle; repeat calls bit-identical."""
    dtype, M, N, tm, tn = case
    x = synthetic.make_matrix(M, N, dtype, "normal", seed=M + tn)
    plan = mbt.tile_plan_device(mbt.OP_COLSUM, M, N, tm, tn, 4, synthetic.DTYPES[dtype],
                                ctas_per_sm=1)
    assert plan["split"] == 1 and plan["col_group"] == 2 and plan["kmax"] > 8, plan
    xd = x.cuda()
    out = mbt.tile_colsum(xd, None, tm, tn, 4, ctas_per_sm=1)
    assert mbt.tile_status()[0] == 0
    worst, rel, _ = colsum_errors(out, x)
    assert worst <= ROWSUM_RTOL, (worst, rel)
    again = mbt.tile_colsum(xd, None, tm, tn, 4, ctas_per_sm=1)
    assert mbt.tile_status()[0] == 0
    assert torch.equal(out.view(torch.int32), again.view(torch.int32))


def test_default_warp_counts_on_16_kb_tiles():
    """fp16 128 x 64 tiles: at 2 stages the column sum wants four CTAs per SM
    and takes 2 consumer warps (so that four fit the registers), at 3 stages 4
    warps; the row sum at 4 stages with two CTAs per SM takes 4.  Every sum
    against the oracle."""
    M, N = 4096, 4096
    x = synthetic.make_matrix(M, N, "f16", "uniform", seed=4242)
    xd = x.cuda()
    sms = mbt.tile_device_info()["num_sms"]
    p2 = mbt.tile_plan_device(mbt.OP_COLSUM, M, N, 128, 64, 2, torch.float16)
    assert p2["consumer_warps"] == 2 and p2["grid"] == 4 * sms and p2["col_group"] == 2, p2
    p3 = mbt.tile_plan_device(mbt.OP_COLSUM, M, N, 128, 64, 3, torch.float16)
    assert p3["consumer_warps"] == 4, p3
    for st in (2, 3):
        out = mbt.tile_colsum(xd, None, 128, 64, st)
        assert mbt.tile_status()[0] == 0
        assert colsum_errors(out, x)[0] <= ROWSUM_RTOL, st
    pr = mbt.tile_plan_device(mbt.OP_ROWSUM, M, N, 128, 64, 4, torch.float16)
    assert pr["consumer_warps"] == 4 and pr["grid"] == 2 * sms, pr
    rows = mbt.tile_rowsum(xd, None, 128, 64, 4)
    assert mbt.tile_status()[0] == 0
    assert rowsum_errors(rows, x)[0] <= ROWSUM_RTOL


@pytest.mark.parametrize("split", [False, True])
def test_flush_ring_wraps_many_times(split):
    """Three CTAs over 1024 one-tile strips (and 512 strip pairs): each CTA's
    consumers post hundreds of strip groups through the one-slot flush ring."""
    for M, N, tm, tn in ((64, 262144, 64, 256), (100, 65536, 128, 64)):
        x = synthetic.make_matrix(M, N, "bf16", "normal", seed=M + 5)
        out = mbt.tile_colsum(x.cuda(), None, tm, tn, 2, max_ctas=3, split=split)
        assert mbt.tile_status()[0] == 0
        assert colsum_errors(out, x)[0] <= ROWSUM_RTOL, (M, N)
