"""The staged tile's raw shared-memory bytes, as the copy engine wrote them,
equal the oracle's restatement of the 128-byte swizzle ("cute(11) Hopper TMA
copy" §2.2: Sw<3,4,3> on byte addresses), box by box, for every dtype and for
tiles cut by the matrix edge (zero fill)."""
import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from oracle import swizzle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("dtype,M,N,tm,tn,tr,tc", [
    ("f16", 256, 128, 128, 64, 0, 0),      # the lesson's tile
    ("f16", 256, 128, 128, 64, 1, 1),
    ("bf16", 100, 1000, 64, 256, 1, 3),    # 4 boxes, cut at row 100 and column 1000
    ("f32", 77, 70, 16, 32, 4, 2),         # cut at row 77 and column 70
    ("f16", 9, 9, 7, 128, 1, 0),           # 7-row boxes (stage padded to 1 KB)
])
def test_stage_image_equals_oracle_swizzle(dtype, M, N, tm, tn, tr, tc):
    es = synthetic.ESIZE[dtype]
    ld = synthetic.pitched_ld(N, dtype)
    x = synthetic.make_matrix(M, N, dtype, "uniform", seed=M + N, ld=ld)
    img = mbt.tile_stage_image(x.cuda()[:, :N], tm, tn, tr, tc)
    assert mbt.tile_status()[0] == 0
    img = bytes(img.cpu().numpy().tobytes())
    # expected: the unswizzled tile (zero outside the matrix), one 128-byte
    # box column after another, each passed through the oracle's swizzle
    boxes = tn * es // 128
    per_box = 128 // es
    tile = torch.zeros(tm, tn, dtype=x.dtype)
    r0, c0 = tr * tm, tc * tn
    rows, cols = max(0, min(tm, M - r0)), max(0, min(tn, N - c0))
    tile[:rows, :cols] = x[r0:r0 + rows, c0:c0 + cols]
    raw = tile.view(torch.uint8).numpy()
    for b in range(boxes):
        box = raw[:, b * 128:(b + 1) * 128].tobytes()
        want = swizzle.staged_image(box, tm, es)
        got = img[b * tm * 128:(b + 1) * tm * 128]
        assert got == want, (b,)
