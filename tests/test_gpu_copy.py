"""GPU parity of tile_copy against the CPU oracle (bit-exact), through the
C ABI.  Covers the two lesson shapes, multi-box tiles, ragged edges in both
directions, pitched buffers whose pad columns must stay untouched, special
bit patterns, and the full-size streaming and ragged configurations."""
import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from oracle.pipeline_state import sequence
from helpers import bits, copy_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


def run_copy(src_h, dst_h, N, *args, **kw):
    src, dst = src_h.cuda(), dst_h.cuda()
    mbt.tile_copy(src[:, :N], dst[:, :N], *args, **kw)
    code, info = mbt.tile_status()
    assert code == 0, info
    return dst.cpu()


def test_single_tile_lesson_shape():
    """256 x 128 fp16, 128 x 64 tiles, one stage: 4 CTAs, one tile each."""
    src, dst, want = copy_case("f16", 256, 128, seed=1001)
    p = mbt.tile_plan(mbt.OP_COPY, 256, 128, 128, 64, 1, torch.float16,
                      **{k: v for k, v in mbt.tile_device_info().items() if k != "hbm_gbs_theoretical"},
                      fit_per_sm=1)
    assert p["grid"] == 4
    got = run_copy(src, dst, 128, 128, 64, 1)
    assert torch.equal(bits(got), bits(want))


def test_three_stage_pipeline_lesson_shape_and_log():
    """128 x 512 fp16, 8 tiles along the columns, 1 producer + 3 consumer
    warps in one CTA, 3 stages; the logged cursors must equal the oracle's."""
    src, dst, want = copy_case("f16", 128, 512, seed=1002)
    log = torch.zeros(2 * 16 * 4, dtype=torch.int32, device="cuda")
    got = run_copy(src, dst, 512, 128, 64, 3, consumer_warps=3, max_ctas=1, log=log)
    assert torch.equal(bits(got), bits(want))
    rec = log.view(2, 16, 4).cpu()
    prod = [tuple(r) for r in rec[0, :8].tolist()]
    cons = [tuple(r) for r in rec[1, :8].tolist()]
    assert [(k, t) for k, _, _, t in prod] == [(k, k) for k in range(8)]
    assert [(s, p) for _, s, p, _ in prod] == sequence(3, 1, 8)
    assert [(s, p) for _, s, p, _ in cons] == sequence(3, 0, 8)
    assert rec[:, 8:].abs().sum().item() == 0


CASES = [
    # dtype, M, N, tile_m, tile_n, stages, consumer_warps
    ("f16", 1, 1, 128, 64, 1, 4),
    ("f16", 300, 200, 128, 64, 3, 4),
    ("bf16", 129, 1000, 64, 256, 2, 4),
    ("f32", 257, 33, 128, 32, 4, 3),
    ("f32", 70, 500, 16, 64, 6, 2),
    ("f16", 1000, 520, 7, 128, 5, 1),
    ("bf16", 513, 4100, 32, 512, 2, 8),
    ("f16", 2048, 2048, 128, 64, 6, 7),
    ("f16", 65, 8, 1, 64, 8, 1),
    ("f32", 4099, 1025, 256, 32, 3, 5),
    ("bf16", 300, 1001, 64, 256, 3, 4),   # last tile: 4 boxes in whole chunks + a partial one
    ("bf16", 77, 803, 64, 256, 2, 2),     # last tile: boxes 2-4 start past the whole chunks
]


@pytest.mark.parametrize("store_mode", [0, 1, 2])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_copy_matches_oracle(case, store_mode):
    dtype, M, N, tm, tn, st, w = case
    es = synthetic.ESIZE[dtype]
    src, dst, want = copy_case(dtype, M, N, seed=M * 7 + N, src_pad=16 // es, dst_pad=32 // es)
    got = run_copy(src, dst, N, tm, tn, st, consumer_warps=w, store_mode=store_mode)
    assert torch.equal(bits(got), bits(want))


@pytest.mark.parametrize("store_mode", [0, 1, 2])
@pytest.mark.parametrize("dtype,M,N,tm,tn", [("f16", 200, 1000, 128, 64), ("f32", 77, 70, 64, 32),
                                             ("bf16", 5, 3, 128, 64)])
def test_nothing_written_outside_the_logical_region(dtype, M, N, tm, tn, store_mode):
    """Destination views into a larger poisoned buffer: rows past M and
    columns past N (up to the buffer's pitch) must keep their poison."""
    es = synthetic.ESIZE[dtype]
    src = synthetic.make_matrix(M, N, dtype, "uniform", seed=M + N,
                                ld=synthetic.pitched_ld(N, dtype))
    buf = torch.empty(M + 130, synthetic.pitched_ld(N, dtype) + 64 // es,
                      dtype=synthetic.DTYPES[dtype])
    synthetic.fill_bits(buf, synthetic.POISON_BITS[dtype])
    want = buf.clone()
    oracle.copy(src[:, :N], want[:M, :N])
    d = buf.cuda()
    mbt.tile_copy(src.cuda()[:, :N], d[:M, :N], tm, tn, 2, store_mode=store_mode)
    assert mbt.tile_status()[0] == 0
    assert torch.equal(bits(d.cpu()), bits(want))


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_unified_pipeline_matches_oracle(case):
    """The non-specialised pipeline (every warp consumes, one thread issues
    S-1 tiles ahead, a CTA barrier releases each stage)."""
    dtype, M, N, tm, tn, st, w = case
    es = synthetic.ESIZE[dtype]
    src, dst, want = copy_case(dtype, M, N, seed=M * 5 + N, src_pad=16 // es, dst_pad=32 // es)
    got = run_copy(src, dst, N, tm, tn, st, consumer_warps=w, pipeline=1)
    assert torch.equal(bits(got), bits(want))


def test_unified_pipeline_full_size_and_one_cta():
    src, dst, want = copy_case("f16", 16384, 16384, seed=1003)
    s = src.cuda()
    for st, kw in ((3, {}), (1, {}), (4, dict(max_ctas=1))):
        d = dst.cuda() if not kw else dst[:512].cuda()
        sv = s if not kw else s[:512]
        mbt.tile_copy(sv, d, 128, 64, st, pipeline=1, **kw)
        assert mbt.tile_status()[0] == 0
        assert torch.equal(bits(d.cpu()), bits(want if not kw else want[:512])), (st, kw)


@pytest.mark.parametrize("stages", [1, 2, 3])
def test_bulk_store_mode_many_tiles_per_cta(stages):
    """Each CTA streams many tiles through its ring, including a single-stage
    ring (whose stage must be released as soon as its store has read it)."""
    src, dst, want = copy_case("f16", 1000, 700, seed=41, src_pad=8)
    got = run_copy(src, dst, 700, 128, 64, stages, max_ctas=3, store_mode=1)
    assert torch.equal(bits(got), bits(want))


def test_bulk_store_mode_lesson_shapes_and_log():
    src, dst, want = copy_case("f16", 256, 128, seed=1001)
    assert torch.equal(bits(run_copy(src, dst, 128, 128, 64, 1, store_mode=1)), bits(want))
    src, dst, want = copy_case("f16", 128, 512, seed=1002)
    log = torch.zeros(2 * 16 * 4, dtype=torch.int32, device="cuda")
    got = run_copy(src, dst, 512, 128, 64, 3, max_ctas=1, log=log, store_mode=1)
    assert torch.equal(bits(got), bits(want))
    rec = log.view(2, 16, 4).cpu()
    assert [(s, p) for _, s, p, _ in rec[0, :8].tolist()] == sequence(3, 1, 8)
    assert [(s, p) for _, s, p, _ in rec[1, :8].tolist()] == sequence(3, 0, 8)


@pytest.mark.parametrize("max_ctas,ctas_per_sm", [(1, 0), (3, 0), (0, 1), (0, 2)])
def test_grid_sizes(max_ctas, ctas_per_sm):
    src, dst, want = copy_case("f16", 777, 1500, seed=5, src_pad=8)
    got = run_copy(src, dst, 1500, 128, 64, 4, max_ctas=max_ctas, ctas_per_sm=ctas_per_sm)
    assert torch.equal(bits(got), bits(want))


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_special_bit_patterns(dtype):
    pats = synthetic.special_values(dtype)
    es = synthetic.ESIZE[dtype]
    M, N = 130, 300
    flat = torch.tensor([pats[i % len(pats)] for i in range(M * N)], dtype=torch.int64)
    top = 1 << (8 * es)
    flat = torch.where(flat >= top // 2, flat - top, flat)
    src = flat.to(torch.int16 if es == 2 else torch.int32).view(synthetic.DTYPES[dtype]).reshape(M, N)
    src = torch.nn.functional.pad(src.view(torch.int16 if es == 2 else torch.int32),
                                  (0, synthetic.pitched_ld(N, dtype) - N)).view(synthetic.DTYPES[dtype])
    dst = torch.zeros_like(src)
    want = dst.clone()
    oracle.copy(src[:, :N], want[:, :N])
    got = run_copy(src, dst, N, 128, 128 // es, 3)
    assert torch.equal(bits(got), bits(want))


def test_dense_inplace_and_repeat_calls():
    src, dst, want = copy_case("bf16", 640, 1024, seed=9)
    s, d = src.cuda(), dst.cuda()
    for _ in range(3):
        mbt.tile_copy(s, d, 64, 256, 3)
    mbt.tile_copy(d, d, 128, 64, 2)          # in place: identity
    assert mbt.tile_status()[0] == 0
    assert torch.equal(bits(d.cpu()), bits(want))


def test_empty_shapes():
    x = torch.empty(0, 64, dtype=torch.float16, device="cuda")
    mbt.tile_copy(x, torch.empty_like(x), 128, 64, 2)
    y = torch.empty(5, 0, dtype=torch.float16, device="cuda")
    mbt.tile_copy(y, torch.empty_like(y), 128, 64, 2)
    assert mbt.tile_status()[0] == 0


FULL = [
    # large streaming copy: fp16 16384 x 16384, 128 x 64 tiles, stage sweep
    ("f16", 16384, 16384, 128, 64, (1, 2, 3, 4, 6), 1003),
    # ragged fp32 12289 x 8191 (rows pitched to 8192), 128 x 32 tiles
    ("f32", 12289, 8191, 128, 32, (3,), 1005),
    # ragged fp16 24577 x 16383 (rows pitched to 16384), 128 x 64 tiles
    ("f16", 24577, 16383, 128, 64, (3,), 1006),
]


@pytest.mark.parametrize("case", FULL, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}")
def test_full_size_configs(case):
    dtype, M, N, tm, tn, stage_list, seed = case
    src, dst, want = copy_case(dtype, M, N, seed=seed)
    s = src.cuda()
    wb = bits(want)
    runs = [(st, 0) for st in stage_list] + [(stage_list[-1], 1)]
    for st, mode in runs:
        d = dst.cuda()
        mbt.tile_copy(s[:, :N], d[:, :N], tm, tn, st, store_mode=mode)
        assert mbt.tile_status()[0] == 0
        assert torch.equal(bits(d.cpu()), wb), f"stages={st} store_mode={mode}"
        del d
