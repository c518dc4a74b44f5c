"""Brute-force GPU parity over boundary shapes: M and N around 1, one 16-byte
chunk, the tile edges and twice the tile, for every dtype and its tile shape,
stages 1..4, pitched (2-D tensor-map path) and dense (unaligned widths take
the 1-D bulk-copy path).  Copies bit-exact with poisoned pads and a poisoned
region after the destination; row sums within 1e-5 of the binary64 oracle,
with poison after out[M - 1]."""
import itertools

import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import ROWSUM_RTOL, bits, rowsum_errors

pytestmark = pytest.mark.gpu

MS = [1, 2, 7, 8, 9, 63, 64, 65, 127, 128, 129, 255, 256, 257]
NS = [1, 3, 7, 8, 9, 31, 33, 63, 64, 65, 127, 128, 129, 255, 257, 300]
TILES = {"f16": (128, 64), "bf16": (64, 256), "f32": (128, 32)}


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("layout", ["pitched", "dense"])
def test_boundary_shapes(dtype, layout):
    tm, tn = TILES[dtype]
    es = synthetic.ESIZE[dtype]
    failures = []
    for i, (M, N) in enumerate(itertools.product(MS, NS)):
        st = 1 + i % 4
        ld = synthetic.pitched_ld(N, dtype) + (16 // es if layout == "pitched" else 0)
        if layout == "dense":
            ld = N
        src = synthetic.make_matrix(M, N, dtype, "uniform", seed=i, ld=ld)
        # destination: (M + 3) rows of the same pitch, poisoned; the copy may
        # touch only the logical M x N region of the first M rows
        buf = torch.empty(M + 3, ld, dtype=synthetic.DTYPES[dtype])
        synthetic.fill_bits(buf, synthetic.POISON_BITS[dtype])
        want = buf.clone()
        oracle.copy(src[:, :N], want[:M, :N])
        d = buf.cuda()
        s = src.cuda()
        mbt.tile_copy(s[:, :N], d[:M, :N], tm, tn, st)
        out = torch.full((M + 5,), float("nan"), device="cuda")
        mbt.tile_rowsum(s[:, :N], out[:M], tm, tn, st)
        code, info = mbt.tile_status()
        if code != 0:
            failures.append((M, N, st, "status", info))
            continue
        if not torch.equal(bits(d.cpu()), bits(want)):
            failures.append((M, N, st, "copy"))
        o = out.cpu()
        if not bool(torch.isnan(o[M:]).all()):
            failures.append((M, N, st, "rowsum wrote past M"))
        worst, _, _ = rowsum_errors(o[:M], src[:, :N])
        if worst > ROWSUM_RTOL:
            failures.append((M, N, st, "rowsum", worst))
    assert not failures, failures[:10]


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_boundary_shapes_fused(dtype):
    tm, tn = TILES[dtype]
    es = synthetic.ESIZE[dtype]
    failures = []
    for i, (M, N) in enumerate(itertools.product(MS[::2], NS[::2])):
        ld = synthetic.pitched_ld(N, dtype) + 16 // es
        src = synthetic.make_matrix(M, N, dtype, "normal", seed=100 + i, ld=ld)
        buf = torch.empty(M + 2, ld, dtype=synthetic.DTYPES[dtype])
        synthetic.fill_bits(buf, synthetic.POISON_BITS[dtype])
        want = buf.clone()
        oracle.copy(src[:, :N], want[:M, :N])
        d = buf.cuda()
        out = mbt.tile_copy_rowsum(src.cuda()[:, :N], d[:M, :N], None, tm, tn, 1 + i % 3)
        if mbt.tile_status()[0] != 0:
            failures.append((M, N, "status"))
            continue
        if not torch.equal(bits(d.cpu()), bits(want)):
            failures.append((M, N, "copy"))
        if rowsum_errors(out, src[:, :N])[0] > ROWSUM_RTOL:
            failures.append((M, N, "rowsum"))
    assert not failures, failures[:10]
