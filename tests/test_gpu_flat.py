"""GPU parity of the unaligned-pitch path (row pitch not a multiple of 16
bytes, e.g. dense fp16 rows of 16383 elements): 1-D bulk copies of
16-byte-aligned windows through the same mbarrier ring.  Copies bit-exact
(dense src and dst; bytes past the matrix untouched), row sums at any pitch
within 1e-5 of the binary64 oracle, short rows (several per stage) and long
rows (pieces of a row per stage)."""
import math

import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import ROWSUM_RTOL, bits, rowsum_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


def dense_in_poisoned(dtype, M, N, extra=40):
    """A dense (M, N) view at the start of a poisoned flat buffer, so writes
    past the matrix's last byte are caught."""
    es = synthetic.ESIZE[dtype]
    flat = torch.empty(M * N + extra, dtype=synthetic.DTYPES[dtype])
    synthetic.fill_bits(flat, synthetic.POISON_BITS[dtype])
    return flat


@pytest.mark.parametrize("dtype,M,N,tm,tn,st", [
    ("f16", 1, 1, 128, 64, 2),          # 2 bytes: all tail
    ("f16", 3, 5, 128, 64, 1),
    ("f16", 1000, 63, 128, 64, 3),
    ("bf16", 513, 4099, 64, 256, 2),
    ("f32", 777, 8191, 128, 32, 4),
    ("f16", 37, 16383, 128, 64, 3),
])
def test_flat_copy_matches_oracle(dtype, M, N, tm, tn, st):
    src = synthetic.make_matrix(M, N, dtype, "uniform", seed=M + 7 * N)
    assert (N * synthetic.ESIZE[dtype]) % 16 != 0 or M * N < 8
    dflat = dense_in_poisoned(dtype, M, N)
    want = dflat.clone()
    oracle.copy(src, want[:M * N].view(M, N))
    d = dflat.cuda()
    mbt.tile_copy(src.cuda(), d[:M * N].view(M, N), tm, tn, st)
    code, info = mbt.tile_status()
    assert code == 0, info
    assert torch.equal(bits(d.cpu()), bits(want))


@pytest.mark.parametrize("dtype,dist,M,N,ld,tm,tn,st", [
    ("f16", "uniform", 1000, 63, 63, 128, 64, 3),       # short rows, dense
    ("f16", "normal", 300, 63, 70, 128, 64, 2),         # short rows, pitched (140 B)
    ("bf16", "normal", 2000, 33, 33, 64, 256, 2),
    ("f32", "uniform", 5, 3, 3, 128, 32, 1),
    ("bf16", "normal", 3000, 3, 3, 64, 256, 2),         # rows of <= 64 bytes: one thread a row
    ("f16", "uniform", 2500, 7, 9, 128, 64, 3),         # 14-byte rows, odd pitch
    ("f16", "normal", 777, 8, 11, 128, 64, 2),          # 16-byte rows starting mid-word
    ("f32", "normal", 999, 4, 5, 128, 32, 2),
    ("f16", "uniform", 501, 16383, 16383, 128, 64, 3),  # long rows, one piece each
    ("bf16", "normal", 40, 100003, 100003, 64, 256, 2),  # 4 pieces
    ("bf16", "uniform", 301, 30001, 30001, 64, 256, 2),  # 2 pieces
    ("f32", "normal", 77, 15001, 15003, 128, 32, 2),     # 2 pieces, pitched
    ("bf16", "normal", 65, 65535, 65535, 64, 256, 2),    # 5 pieces
    ("bf16", "uniform", 33, 65535, 65535, 64, 256, 3),   # 8 pieces
    ("f32", "normal", 123, 8191, 8191, 128, 32, 4),
])
def test_flat_rowsum_matches_oracle(dtype, dist, M, N, ld, tm, tn, st):
    x = synthetic.make_matrix(M, N, dtype, dist, seed=M + N, ld=ld)
    out = mbt.tile_rowsum(x.cuda()[:, :N], None, tm, tn, st)
    code, info = mbt.tile_status()
    assert code == 0, info
    worst, rel, _ = rowsum_errors(out, x[:, :N])
    assert worst <= ROWSUM_RTOL, (worst, rel)


@pytest.mark.parametrize("dtype,M,N,ld", [
    ("bf16", 100003, 1, 1),          # 2-byte rows
    ("bf16", 50001, 3, 3),           # 6-byte rows, the array's last row past its last
    ("f16", 1001, 3, 3),             #   16-byte boundary (read from global memory)
    ("f16", 40000, 8, 11),           # 16-byte rows, odd pitch
    ("f16", 30000, 9, 9),            # 18 bytes: the rolled loop
    ("bf16", 20000, 17, 17),
    ("bf16", 9999, 31, 33),          # 62-byte rows, pitched
    ("bf16", 8191, 32, 35),          # 64 bytes: the largest of this path
    ("f32", 60001, 1, 1),
    ("f32", 12345, 3, 5),
    ("f32", 7001, 15, 15),
    ("f32", 5003, 16, 17),
])
def test_flat_rowsum_element_rows(dtype, M, N, ld):
    """Rows of at most 64 bytes: each consumer thread sums whole rows element
    by element (unrolled up to 8 elements, a loop beyond).  Every row is
    written (the output starts as NaN) and matches the oracle; the planner
    takes this path exactly up to 64-byte rows."""
    es = synthetic.ESIZE[dtype]
    assert (ld * es) % 16 != 0
    info = mbt.tile_device_info()
    plan = mbt.tile_plan(mbt.OP_ROWSUM, M, N, 64, 256 if es == 2 else 128, 2,
                         synthetic.DTYPES[dtype], num_sms=info["num_sms"],
                         smem_optin=info["smem_optin"], fit_per_sm=3, ld_src=ld)
    assert plan["flat"] == 1 and plan["phase_shift"] == 0
    x = synthetic.make_matrix(M, N, dtype, "normal", seed=M + 13 * N, ld=ld)
    out = torch.full((M,), float("nan"), device="cuda")
    mbt.tile_rowsum(x.cuda()[:, :N], out, 64, 256 if es == 2 else 128, 2)
    code, info = mbt.tile_status()
    assert code == 0, info
    assert not bool(out.isnan().any())
    worst, rel, _ = rowsum_errors(out, x[:, :N])
    assert worst <= ROWSUM_RTOL, (worst, rel)


@pytest.mark.parametrize("dtype,M,N,ld", [
    ("bf16", 200000, 2, 8),      # 16-byte pitch: one pair per row
    ("f16", 150000, 4, 4),       # 8-byte dense pitch
    ("bf16", 100000, 6, 12),     # 24-byte pitch
    ("f16", 80000, 10, 16),      # the loop over pairs: 5 pairs (one left after the pairs of pairs)
    ("bf16", 70000, 16, 16),     # 32-byte dense pitch
    ("f16", 60000, 24, 32),
    ("bf16", 50000, 30, 32),     # 15 pairs
    # pitches of an odd number of 4-byte words: no rotation, pairs from column 0
    ("bf16", 120000, 6, 6),      # 12 bytes
    ("f16", 100000, 10, 10),     # 20 bytes
    ("bf16", 60000, 18, 18),     # 36 bytes: the loop over pairs
    ("f16", 40000, 30, 30),      # 60 bytes
    ("bf16", 70000, 17, 18),     # odd row length: the last element alone
    ("f16", 90000, 1, 2),        # one element in a 4-byte pitch
    ("bf16", 80000, 7, 10),      # 7 elements (unrolled) in a 20-byte pitch
])
def test_flat_rowsum_paired_rows(dtype, M, N, ld):
    """16-bit rows whose pitch is a whole number of 4-byte words, so that every
    row starts on one: two elements per 32-bit load.  Where the pitch in words
    shares a factor with 32 (and the row length is even), lanes start their
    rows at rotated, even columns; else from column 0, an odd row's last
    element alone.  Every row is written and matches the oracle."""
    es = synthetic.ESIZE[dtype]
    pitch = ld * es
    assert N * es <= 64 and pitch % 4 == 0
    assert N % 2 == 0 or math.gcd(pitch // 4, 32) == 1
    dt = synthetic.DTYPES[dtype]
    assert mbt.tile_plan_device(mbt.OP_ROWSUM, M, N, 64, 256, 2, dt, ld_src=ld)["flat"] == 1
    x = synthetic.make_matrix(M, N, dtype, "normal", seed=M + 7 * N, ld=ld)
    out = torch.full((M,), float("nan"), device="cuda")
    mbt.tile_rowsum(x.cuda()[:, :N], out, 64, 256, 2)
    code, info = mbt.tile_status()
    assert code == 0, info
    assert not bool(out.isnan().any())
    worst, rel, _ = rowsum_errors(out, x[:, :N])
    assert worst <= ROWSUM_RTOL, (worst, rel)


@pytest.mark.parametrize("dtype,M,N,ld,tile", [
    ("bf16", 600000, 8, 8, (64, 256)),       # 16-byte rows, dense: a 16-byte pitch
    ("f32", 300001, 16, 16, (128, 32)),      # 64-byte rows, dense
    ("bf16", 70000, 32, 40, (64, 64)),       # 64-byte rows in an 80-byte pitch
    ("f16", 90000, 5, 8, (128, 64)),         # 10-byte rows in a 16-byte pitch
])
def test_narrow_aligned_rows_take_the_element_path(dtype, M, N, ld, tile):
    """Row sums of rows of at most 64 bytes take the 1-D kernels even where the
    pitch is a multiple of 16 bytes (a tiled plan would carry mostly zero
    fill); with more than 8 consumer warps asked for, the tiled kernels."""
    es = synthetic.ESIZE[dtype]
    assert (ld * es) % 16 == 0 and N * es <= 64
    dt = synthetic.DTYPES[dtype]
    assert mbt.tile_plan_device(mbt.OP_ROWSUM, M, N, *tile, 2, dt, ld_src=ld)["flat"] == 1
    assert mbt.tile_plan_device(mbt.OP_ROWSUM, M, N, *tile, 2, dt, ld_src=ld,
                                consumer_warps=12)["flat"] == 0
    x = synthetic.make_matrix(M, N, dtype, "normal", seed=M + N, ld=ld)
    xd = x.cuda()[:, :N]
    out = torch.full((M,), float("nan"), device="cuda")
    mbt.tile_rowsum(xd, out, *tile, 2)
    wide = mbt.tile_rowsum(xd, None, *tile, 2, consumer_warps=12)
    code, info = mbt.tile_status()
    assert code == 0, info
    assert rowsum_errors(out, x[:, :N])[0] <= ROWSUM_RTOL
    assert rowsum_errors(wide, x[:, :N])[0] <= ROWSUM_RTOL


@pytest.mark.parametrize("dtype,M,N,warps,ctas", [
    ("bf16", 5000, 65, 0, 16),      # 224 rows per window padded to blocks of 64
    ("bf16", 4097, 67, 0, 16),
    ("f16", 2049, 255, 0, 16),      # 2 lanes per row, rows 16 apart
    ("f32", 7777, 31, 0, 16),
    ("f16", 3001, 127, 0, 16),
    ("bf16", 3000, 129, 0, 8),
    ("bf16", 100000, 63, 0, 0),     # default grid, ~219 rows per CTA: one short window each
    ("bf16", 5000, 63, 8, 16),      # 8 consumer warps
])
def test_flat_rowsum_permuted_rows_each_written_once(dtype, M, N, warps, ctas):
    """Rows given to lane groups 2^phase_shift apart: every row is summed and
    written (the output starts as NaN), on windows cut short at each CTA's
    last rows as well as whole ones.  The grid is capped where the default
    one would leave each CTA fewer rows than a window holds (its lane groups
    would then take a row each, and no phase would hold several rows)."""
    kw = {"consumer_warps": warps} if warps else {}
    if ctas:
        kw["max_ctas"] = ctas
    info = mbt.tile_device_info()
    plan = mbt.tile_plan(mbt.OP_ROWSUM, M, N, 128, 64, 2, synthetic.DTYPES[dtype],
                         num_sms=info["num_sms"], smem_optin=info["smem_optin"],
                         fit_per_sm=3, **kw)
    assert plan["flat"] == 1 and plan["phase_shift"] > 0
    x = synthetic.make_matrix(M, N, dtype, "normal", seed=31 * M + N)
    out = torch.full((M,), float("nan"), device="cuda")
    mbt.tile_rowsum(x.cuda(), out, 128, 64, 2, **kw)
    code, info = mbt.tile_status()
    assert code == 0, info
    assert not bool(out.isnan().any())
    worst, rel, _ = rowsum_errors(out, x)
    assert worst <= ROWSUM_RTOL, (worst, rel)


def test_flat_full_size_dense_ragged_configs():
    """The ragged fp32 12289 x 8191 and fp16 24577 x 16383 shapes, stored dense (no pitch
    padding)."""
    for dtype, M, N, tm, tn, seed in (("f32", 12289, 8191, 128, 32, 1005),
                                      ("f16", 24577, 16383, 128, 64, 1006)):
        x = synthetic.make_matrix(M, N, dtype, "uniform", seed)
        xd = x.cuda()
        y = torch.empty_like(xd)
        mbt.tile_copy(xd, y, tm, tn, 3)
        out = mbt.tile_rowsum(xd, None, tm, tn, 3)
        assert mbt.tile_status()[0] == 0
        assert torch.equal(bits(y.cpu()), bits(x))
        assert rowsum_errors(out, x)[0] <= ROWSUM_RTOL


@pytest.mark.parametrize("fault", [1, 2])
def test_flat_stall_reports_timeout(fault):
    x = synthetic.make_matrix(512, 1001, "f16", "uniform", seed=2).cuda()
    y = torch.empty_like(x)
    mbt.tile_copy(x, y, 128, 64, 3, max_ctas=4, fault=fault, wait_budget_ns=20_000_000)
    assert mbt.tile_status()[0] == mbt.MBT_ERR_TIMEOUT
    mbt.tile_rowsum(x, None, 128, 64, 3, max_ctas=4, fault=fault, wait_budget_ns=20_000_000)
    assert mbt.tile_status()[0] == mbt.MBT_ERR_TIMEOUT
    mbt.tile_copy(x, y, 128, 64, 3)
    assert mbt.tile_status()[0] == 0
    assert torch.equal(y.view(torch.int16), x.view(torch.int16))
