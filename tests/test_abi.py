"""C ABI checks that need no GPU: the library loads, exports every entry point
declared in include/mbtile.h, rejects bad arguments on the host before any
CUDA call, and plans launches as documented."""
import ctypes
import os
import re

import pytest
import random
import torch

import mbarrier_async_tile_gb300 as mbt
from mbarrier_async_tile_gb300 import C, Opts, _build
from conftest import ROOT, read_golden

HEADER = os.path.join(ROOT, "include", "mbtile.h")


@pytest.fixture(scope="module", autouse=True)
def built_library():
    _build.build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tile_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert {"tile_copy", "tile_rowsum", "tile_copy_ex", "tile_rowsum_ex", "tile_status",
            "tile_plan", "tile_strerror"} <= set(names)
    lib = ctypes.CDLL(_build.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_covers_codes():
    for code in range(0, -9, -1):
        s = mbt.tile_strerror(code)
        assert s and "unknown" not in s
    assert "unknown" in mbt.tile_strerror(-99)


def _copy(src, dst, M, N, tm=128, tn=64, st=3, dt=0, opts=None):
    return C.tile_copy_ex(src, dst, M, N, tm, tn, st, dt, None,
                          ctypes.byref(opts) if opts is not None else None)


A = 0x10000          # fake, 16-byte aligned "device" addresses: never dereferenced
B = 0x20000


@pytest.mark.parametrize("args,code", [
    ((0, B, 8, 64), -1),                         # null src
    ((A, 0, 8, 64), -1),                         # null dst
    ((A, B, -1, 64), -1),                        # negative M
    ((A + 8, B, 8, 64), -2),                     # misaligned src
    ((A, B + 2, 8, 64), -2),                     # misaligned dst
])
def test_copy_argument_errors(args, code):
    assert _copy(*args) == code


def test_unaligned_pitch_routes_and_refusals():
    # dense fp16 rows of 126 bytes: the 1-D bulk-copy path (no 2-D tensor map)
    p = _plan(mbt.OP_COPY, 1000, 63, 128, 64, 3, torch.float16, fit=2)
    assert p["flat"] == 1 and p["num_tiles"] == -(-(1000 * 63 * 2 // 16 * 16) // 16384)
    p = _plan(mbt.OP_ROWSUM, 1000, 63, 128, 64, 3, torch.float16, fit=2, ws=True)
    assert p["flat"] == 1 and p["workspace_bytes"] == 0 and p["grid"] == 304
    # row sum with a pitch of 70 elements (140 bytes): allowed
    assert _plan(mbt.OP_ROWSUM, 10, 63, 128, 64, 3, torch.float16, ld_src=70)["flat"] == 1
    # copies whose src and dst are not both dense, or bulk-store / unified copies: refused
    o = Opts(); o.ld_src = 70                    # 140-byte pitch, dst dense
    assert _copy(A, B, 8, 63, opts=o) == -2
    o = Opts(); o.store_mode = 1
    assert _copy(A, B, 8, 63, opts=o) == -2
    o = Opts(); o.pipeline = 1
    assert _copy(A, B, 8, 63, opts=o) == -2
    assert C.tile_copy_rowsum_ex(A, B, B, 8, 63, 128, 64, 3, 0, None, None) == -2
    # aligned shapes keep the tiled path
    assert _plan(mbt.OP_COPY, 1000, 64, 128, 64, 3, torch.float16)["flat"] == 0


def test_flat_rowsum_windows_follow_the_rows_not_the_tile():
    """Unaligned-pitch row sums load whole rows (32 KB windows while 8 rows
    fit, else up to 64 KB) or equal pieces of longer rows, whatever the tile,
    within what the stages leave of shared memory; the default grid keeps
    about 192 KB of stages per SM."""
    smem = 232448
    plans = [_plan(mbt.OP_ROWSUM, 24577, 16383, tm, tn, 2, torch.float16, fit=8)
             for tm, tn in ((128, 64), (64, 256), (256, 512))]
    for p in plans:
        # one window per 32766-byte row (+ up to 32 bytes of 16-byte rounding)
        assert p["flat"] == 1 and p["num_tiles"] == 24577 and p["stage_bytes"] == 33 * 1024
        assert p["grid"] == 3 * 152 and p["consumer_warps"] == 4
    short = _plan(mbt.OP_ROWSUM, 4194304, 63, 128, 64, 2, torch.float16, fit=8)
    assert short["stage_bytes"] == 32 * 1024                 # 256 rows of 126 bytes
    # 200006-byte rows: four pieces of at most 64 KB at 2 stages; at 8 stages
    # the pieces shrink so that the stages still fit
    p2 = _plan(mbt.OP_ROWSUM, 2000, 100003, 128, 64, 2, torch.bfloat16, fit=8)
    assert p2["num_tiles"] == 2000 * 4 and p2["stage_bytes"] <= 64 * 1024 + 1024
    p8 = _plan(mbt.OP_ROWSUM, 2000, 100003, 128, 64, 8, torch.bfloat16, fit=8)
    assert p8["smem_bytes"] <= smem and p8["num_tiles"] == 2000 * 7
    # tile_m above 32 x consumer_warps does not matter without tile rows
    assert _plan(mbt.OP_ROWSUM, 1000, 63, 256, 64, 2, torch.float16, consumer_warps=1,
                 fit=8)["flat"] == 1


def test_flat_rowsum_pieces_put_most_bytes_in_flight():
    """Long rows in pieces: the piece count with the most bytes of stages in
    flight on an SM (CTAs that fit, at most four, x stages x stage bytes), where
    that beats the fewest pieces by at least 5 %."""
    def pieces(dtype, M, N, S):
        p = _plan(mbt.OP_ROWSUM, M, N, 64, 256, S, dtype, fit=4)
        assert p["flat"] == 1 and p["num_tiles"] % M == 0
        return p["num_tiles"] // M, p["stage_bytes"]
    # 131070-byte rows: 3 pieces (two 2 x 43 KB CTAs per SM) become 5 of 26 KB
    # (four CTAs: 208 KB in flight against 172 KB)
    assert pieces(torch.bfloat16, 4096, 65535, 2) == (5, 26 * 1024)
    # 80002-byte rows: 2 pieces of 40 KB become 3 of 27 KB
    assert pieces(torch.float16, 8192, 40001, 2) == (3, 27 * 1024)
    # 200006-byte rows: 8 pieces would add only 2 %, so 4 of 49 KB stay
    assert pieces(torch.bfloat16, 2000, 100003, 2) == (4, 49 * 1024)
    # at 3 stages one 3 x 43 KB CTA per SM gives way to four of 3 x 17 KB
    assert pieces(torch.bfloat16, 4096, 65535, 3) == (8, 17 * 1024)
    # 60002-byte rows: one 59 KB piece leaves one CTA per SM (118 KB in
    # flight); 2 pieces on 3 CTAs (180 KB) beat 3 on 4 (160 KB)
    assert pieces(torch.bfloat16, 8192, 30001, 2) == (2, 30 * 1024)
    assert pieces(torch.float32, 4096, 15001, 2) == (2, 30 * 1024)
    # ... and at 3 stages 1 piece on one CTA holds as much as any split
    assert pieces(torch.bfloat16, 8192, 30001, 3) == (1, 59 * 1024)
    # whole rows per window are not cut
    assert _plan(mbt.OP_ROWSUM, 16384, 16383, 64, 256, 2, torch.bfloat16,
                 fit=4)["num_tiles"] == 16384


def test_flat_rowsum_piece_plans_cover_rows_and_fit():
    """Seeded random long rows at any pitch and 1-8 stages: each row is cut
    into equal pieces that cover it exactly, a piece (plus 16-byte rounding at
    both ends) fits its stage, the stages fit shared memory, and the pieces
    are never fewer than the window bound allows."""
    rng = random.Random(20261202)
    smem = 232448
    for _ in range(400):
        dtype = rng.choice([torch.bfloat16, torch.float16, torch.float32])
        es = torch.tensor([], dtype=dtype).element_size()
        N = rng.randint(8192, 1 << 20)               # rows of 16 KB and more
        ld = N + rng.choice([0, 1, 3])
        if ld * es % 16 == 0:
            ld += 1                                  # a pitch the 1-D kernels take
        st = rng.randint(1, 8)
        M = rng.randint(1, 50)
        p = _plan(mbt.OP_ROWSUM, M, N, 64, 256 if es == 2 else 128, st, dtype, smem=smem,
                  fit=rng.randint(1, 4), ld_src=ld)
        assert p["flat"] == 1 and p["smem_bytes"] <= smem
        pieces = p["num_tiles"] // M
        assert pieces * M == p["num_tiles"] and pieces >= 1
        piece = -(-N // pieces)
        assert (pieces - 1) * piece < N <= pieces * piece          # equal pieces, no empty one
        assert piece * es + 32 <= p["stage_bytes"]
        window_cap = min(64 * 1024, (smem - 1024) // st // 1024 * 1024) - 32
        assert pieces >= -(-N // (window_cap // es))


def test_flat_rowsum_phase_shift_spreads_bank_groups():
    """Short unaligned rows: the 8 / L lane groups of one 8-lane shared-memory
    phase sum rows 2^phase_shift apart.  A 16-byte read's bank group is its
    window offset / 16 mod 8, so rows s apart start s * pitch / 16 groups
    apart: with 8 rows of one lane each, s * pitch = 16 x odd (mod 128) puts the
    phase's 8 lanes in 8 distinct groups; with 4 rows of 2 lanes each, s * pitch
    = 32 x odd (mod 128) puts their 2-chunk spans side by side.  A shift is
    taken only where it cuts a phase's wavefronts at least 3-fold."""
    def shift(dtype, N, **kw):
        return _plan(mbt.OP_ROWSUM, 2097152, N, 128, 64, 2, dtype, fit=3, **kw)["phase_shift"]
    # one lane per row (4 consumer warps, 224-260 rows per window):
    # 8 x 126 = 1008 = -16, 8 x 130 = 1040 = 16, 8 x 134 = 1072 = 48 (mod 128);
    # a smaller power of two leaves two lanes of a phase in one group
    assert shift(torch.bfloat16, 63) == 3
    assert shift(torch.bfloat16, 65) == 3
    assert shift(torch.bfloat16, 67) == 3
    # 510-byte rows, 64 per window, 2 lanes per row: 16 x 510 = 8160 = 96 = 32 x 3
    # (mod 128); 8 x 510 = 4080 = 112 would overlap two rows' spans
    assert shift(torch.float16, 255) == 4
    # two rows per phase (4 lanes each), or 34-byte rows 2.1 groups apart: at
    # most 2-way conflicts, which a shift could only halve
    assert shift(torch.bfloat16, 300) == 0
    assert shift(torch.bfloat16, 17) == 0
    # 2002-byte rows: 16 per window, a phase reads 8 chunks of one row
    assert shift(torch.float16, 1001) == 0
    # rows of at most 16 bytes are read 4 bytes at a time; long rows in pieces
    assert shift(torch.bfloat16, 3) == 0
    assert _plan(mbt.OP_ROWSUM, 2000, 100003, 128, 64, 2, torch.bfloat16,
                 fit=8)["phase_shift"] == 0
    # the same rows on 8 consumer warps: 4 lanes per row, two rows per phase
    # (at most 2-way); the answer follows the warps, call after call
    assert shift(torch.float16, 255, consumer_warps=8) == 0
    assert shift(torch.float16, 255) == 4
    assert shift(torch.float16, 255, consumer_warps=8) == 0
    # 2-D tensor-map path and the copy: no lane groups over rows
    assert _plan(mbt.OP_ROWSUM, 8192, 65536, 64, 256, 2, torch.bfloat16)["phase_shift"] == 0
    assert _plan(mbt.OP_COPY, 2097152, 63, 128, 64, 2, torch.bfloat16)["phase_shift"] == 0


def test_copy_tile_and_stage_errors():
    assert _copy(A, B, 8, 64, tm=0) == -1
    assert _copy(A, B, 8, 64, tm=257) == -1
    assert _copy(A, B, 8, 64, tn=32) == -3       # 64-byte box rows: unsupported
    assert _copy(A, B, 8, 64, tn=96) == -3       # 192 bytes: not 1/2/4/8 boxes
    assert _copy(A, B, 8, 64, st=0) == -1
    assert _copy(A, B, 8, 64, st=9) == -1
    assert _copy(A, B, 8, 64, dt=7) == -1


def test_option_errors():
    o = Opts()
    o.reserved1 = 1
    assert _copy(A, B, 8, 64, opts=o) == -1
    o = Opts(); o.reserved0 = 1
    assert _copy(A, B, 8, 64, opts=o) == -1
    # no_split: 0 or 1, row and column sums only, never with a workspace
    o = Opts(); o.no_split = 1
    assert _copy(A, B, 8, 64, opts=o) == -1
    o = Opts(); o.no_split = 2
    assert C.tile_rowsum_ex(A, B, 8, 64, 128, 64, 3, 0, None, ctypes.byref(o)) == -1
    o = Opts(); o.no_split = 1; o.workspace = B; o.workspace_bytes = 256
    assert C.tile_rowsum_ex(A, B, 8, 64, 128, 64, 3, 0, None, ctypes.byref(o)) == -1
    assert C.tile_colsum_ex(A, B, 8, 64, 128, 64, 3, 0, None, ctypes.byref(o)) == -1
    o = Opts(); o.status = B + 2                   # a status buffer must be 4-byte aligned
    assert _copy(A, B, 8, 64, opts=o) == -2
    assert C.tile_rowsum_ex(A, B, 8, 64, 128, 64, 3, 0, None, ctypes.byref(o)) == -2
    o = Opts(); o.consumer_warps = 9
    assert _copy(A, B, 8, 64, opts=o) == -1
    o = Opts(); o.fault = 3
    assert _copy(A, B, 8, 64, opts=o) == -1
    o = Opts(); o.pipeline = 4
    assert _copy(A, B, 8, 64, opts=o) == -3
    for pipe in (2, 3):                            # barrier layouts: row sum only
        o = Opts(); o.pipeline = pipe
        assert _copy(A, B, 8, 64, opts=o) == -1
        assert C.tile_copy_rowsum_ex(A, B, B, 8, 64, 128, 64, 3, 0, None,
                                     ctypes.byref(o)) == -1
    o = Opts(); o.pipeline = 1; o.store_mode = 1   # unified pipeline: LSU stores only
    assert _copy(A, B, 8, 64, opts=o) == -3
    o = Opts(); o.pipeline = 1                     # copy only
    assert C.tile_rowsum_ex(A, B, 8, 64, 128, 64, 3, 0, None, ctypes.byref(o)) == -1
    o = Opts(); o.store_mode = 3
    assert _copy(A, B, 8, 64, opts=o) == -3
    o = Opts(); o.store_mode = 2                 # LSU stores: a copy-only option
    assert C.tile_rowsum_ex(A, B, 8, 64, 128, 64, 3, 0, None, ctypes.byref(o)) == -1
    o = Opts(); o.store_mode = 1                 # bulk stores: a copy-only option
    assert C.tile_rowsum_ex(A, B, 8, 64, 128, 64, 3, 0, None, ctypes.byref(o)) == -1
    o = Opts(); o.ld_src = 60                    # pitch below N
    assert _copy(A, B, 8, 64, opts=o) == -1
    o = Opts(); o.ld_dst = 68                    # 136-byte pitch: not a 16-byte multiple
    assert _copy(A, B, 8, 64, opts=o) == -2


def test_fused_argument_errors():
    fn = C.tile_copy_rowsum_ex
    assert fn(A, B, None, 8, 64, 128, 64, 3, 0, None, None) == -1          # out missing
    assert fn(A, B, B + 2, 8, 64, 128, 64, 3, 0, None, None) == -2         # out misaligned
    assert fn(A, B + 8, B, 8, 64, 128, 64, 3, 0, None, None) == -2         # dst misaligned
    o = Opts(); o.store_mode = 1
    assert fn(A, B, B, 8, 64, 128, 64, 3, 0, None, ctypes.byref(o)) == -1
    assert fn(0, 0, None, 0, 64, 128, 64, 3, 0, None, None) == 0


def test_empty_shapes_are_noops_without_device():
    assert _copy(0, 0, 0, 64) == 0
    assert _copy(0, 0, 5, 0) == 0
    # a row sum of rows with no columns must still write M zeros: out required
    assert C.tile_rowsum(A, None, 5, 0, 64, 256, 3, 1, None) == -1
    assert C.tile_rowsum(0, None, 0, 0, 64, 256, 3, 1, None) == 0


def test_host_forms_argument_errors_before_any_cuda_call():
    """The host-buffer forms check their arguments before touching the
    device, so these run without a GPU."""
    src = (ctypes.c_uint16 * 64)()
    out = (ctypes.c_float * 8)(*([7.0] * 8))
    p = ctypes.addressof
    assert C.tile_copy_host(p(src), p(src), 0, 64, 128, 64, 3, 0, None) == 0
    assert C.tile_rowsum_host(p(src), p(out), 8, 0, 64, 64, 2, 0, None) == 0
    assert list(out) == [0.0] * 8                       # empty rows sum to 0
    assert C.tile_rowsum_host(p(src), None, 8, 0, 64, 64, 2, 0, None) == -1
    assert C.tile_rowsum_host(None, p(out), 8, 8, 64, 64, 2, 0, None) == -1
    assert C.tile_copy_host(p(src), None, 8, 8, 64, 64, 2, 0, None) == -1
    assert C.tile_copy_host(p(src), p(src), 8, 8, 64, 64, 2, 7, None) == -1   # dtype
    for field, value in (("log", 16), ("workspace", 16), ("workspace_bytes", 4),
                         ("host_slab_rows", -1), ("ld_src", 4), ("status", 16)):
        o = Opts()
        setattr(o, field, value)
        assert C.tile_copy_host(p(src), p(src), 8, 8, 64, 64, 2, 0, ctypes.byref(o)) == -1, field
    o = Opts(); o.ld_dst = 8                             # a row sum has no dst pitch
    assert C.tile_rowsum_host(p(src), p(out), 8, 8, 64, 64, 2, 0, ctypes.byref(o)) == -1
    cout = (ctypes.c_float * 4)(*([5.0] * 4))
    assert C.tile_colsum_host(p(src), p(cout), 0, 4, 64, 64, 2, 0, None) == 0
    assert list(cout) == [0.0] * 4                      # no rows: zero column sums
    assert C.tile_colsum_host(p(src), None, 8, 0, 64, 64, 2, 0, None) == 0   # no columns
    assert C.tile_colsum_host(p(src), None, 8, 4, 64, 64, 2, 0, None) == -1
    o = Opts(); o.host_slab_rows = 4                     # host-buffer forms only
    assert _copy(A, B, 8, 64, opts=o) == -1
    assert C.tile_rowsum_ex(A, B, 8, 64, 128, 64, 3, 0, None, ctypes.byref(o)) == -1


def _plan(op, M, N, tm, tn, st, dtype, sms=152, smem=232448, fit=1, ws=False, **opt):
    return mbt.tile_plan(op, M, N, tm, tn, st, dtype, num_sms=sms, smem_optin=smem,
                         fit_per_sm=fit, with_workspace=ws, **opt)


def test_plan_single_tile_lesson_shape():
    sizes = {r[0]: int(r[-1]) for r in read_golden("lesson_sizes.txt")}
    p = _plan(mbt.OP_COPY, 256, 128, 128, 64, 1, torch.float16, fit=4)
    assert p["tx_bytes"] == sizes["tx_bytes"]
    assert p["box_inner"] == sizes["tma_box_inner"] and p["box_rows"] == sizes["tma_box_outer"]
    assert p["grid"] == 4 and p["num_tiles"] == 4 and p["boxes"] == 1
    # one 16 KiB stage plus 1 KiB of alignment slack for the swizzle atom
    assert p["smem_bytes"] == 16384 + 1024


def test_plan_pipeline_lesson_shape():
    p = _plan(mbt.OP_COPY, 128, 512, 128, 64, 3, torch.float16, max_ctas=1, consumer_warps=3)
    assert p["grid"] == 1 and p["threads"] == 128 and p["num_tiles"] == 8
    assert p["smem_bytes"] == 3 * 16384 + 1024


def test_plan_default_grid_follows_bytes_in_flight():
    # row sum, 64 x 256 bf16 (32 KB stages): 2 stages x 2 CTAs = 128 KB per SM, 8 warps
    p = _plan(mbt.OP_ROWSUM, 8192, 65536, 64, 256, 2, torch.bfloat16, fit=4, ws=True)
    assert p["grid"] == 304 and p["consumer_warps"] == 8
    # the same tiles at 3 stages (96 KB per CTA): still 2 CTAs, with 4 warps; at 4
    # stages only one 128 KB CTA fits an SM: 8 consumer warps (each thread one
    # round of 8 chunks; + producer and flush warps); the column sum keeps 8 too
    p = _plan(mbt.OP_ROWSUM, 8192, 65536, 64, 256, 3, torch.bfloat16, fit=2, ws=True)
    assert p["grid"] == 304 and p["consumer_warps"] == 4
    p = _plan(mbt.OP_ROWSUM, 8192, 65536, 64, 256, 4, torch.bfloat16, fit=1, ws=True)
    assert p["grid"] == 152 and p["consumer_warps"] == 8 and p["threads"] == 32 * 10
    assert p["box_barriers"] == 0
    # tiles whose rows would give each of 256 threads two rounds of 8 chunks
    # (boxes x tile_m > 256): the wide CTA of 16 consumer warps
    p = _plan(mbt.OP_ROWSUM, 8192, 32768, 128, 128, 3, torch.float32, fit=1, ws=True)
    assert p["grid"] == 152 and p["consumer_warps"] == 16 and p["threads"] == 32 * 18
    # (one CTA per SM: its 512-byte strips walked in pairs)
    p = _plan(mbt.OP_COLSUM, 8192, 65536, 64, 256, 4, torch.bfloat16, fit=1, ws=True)
    assert p["grid"] == 152 and p["consumer_warps"] == 8 and p["col_group"] == 2
    p = _plan(mbt.OP_COLSUM, 8192, 65536, 64, 256, 4, torch.bfloat16, fit=1, ws=True,
              consumer_warps=16)
    assert p["threads"] == 32 * 18 and p["col_group"] == 1
    # a caller's one CTA per SM is planned the same way; 128-byte column-sum
    # tiles walked in strip pairs, the fused operation and copies never get the
    # wide CTA
    p = _plan(mbt.OP_ROWSUM, 8192, 65536, 64, 256, 2, torch.bfloat16, fit=4, ws=True,
              ctas_per_sm=1)
    assert p["consumer_warps"] == 8
    p = _plan(mbt.OP_ROWSUM, 8192, 65536, 128, 256, 2, torch.bfloat16, fit=4, ws=True,
              ctas_per_sm=1)
    assert p["consumer_warps"] == 16
    p = _plan(mbt.OP_COLSUM, 12289, 8191, 128, 32, 8, torch.float32, fit=1, ws=True,
              ld_src=8192)
    assert p["col_group"] == 2 and p["consumer_warps"] == 8
    p = _plan(mbt.OP_COLSUM, 12289, 8191, 128, 32, 3, torch.float32, fit=1, ws=True,
              ld_src=8192, consumer_warps=12)   # more than 8 warps: one strip at a time
    assert p["col_group"] == 1 and p["consumer_warps"] == 12
    # strip pairs only with an even warp count (4 W threads per chunk column, a
    # multiple of 8, so each thread's rows share one swizzle term)
    for W, cg in ((2, 2), (3, 1), (4, 2), (5, 1), (6, 2), (7, 1), (8, 2)):
        p = _plan(mbt.OP_COLSUM, 12289, 8191, 128, 32, 3, torch.float32, fit=2, ws=True,
                  ld_src=8192, consumer_warps=W)
        assert p["col_group"] == cg, W
    # wider strips in pairs only where one CTA per SM runs, and only with tpc =
    # 32 W / (8 boxes) a multiple of 8 (512-byte rows: W = 8)
    for fit, W, cg in ((2, 8, 1), (1, 8, 2), (1, 4, 1), (1, 6, 1)):
        p = _plan(mbt.OP_COLSUM, 8192, 65536, 64, 256, 4 if fit == 1 else 2, torch.bfloat16,
                  fit=fit, ws=True, consumer_warps=W)
        assert p["col_group"] == cg, (fit, W)
    p = _plan(mbt.OP_COLSUM, 8192, 65536, 128, 128, 4, torch.bfloat16, fit=1, ws=True)
    assert p["col_group"] == 2 and p["consumer_warps"] == 8        # 256-byte rows: tpc 16


def test_plan_colsum_shared_memory_holds_the_flush_ring():
    """The column sum's dynamic shared memory: 1024 bytes of alignment slack,
    the stages, then one flush-ring slot of one float per consumer thread,
    element of a 16-byte chunk and strip of the group (32 W x 16 / es x g)."""
    for dt, es, M, N, tm, tn, st, fit, ld, W, g in (
            (torch.float32, 4, 12289, 8191, 128, 32, 3, 3, 8192, 4, 2),
            (torch.float16, 2, 24577, 16383, 128, 64, 3, 3, 16384, 4, 2),
            (torch.bfloat16, 2, 8192, 65536, 64, 256, 3, 2, 65536, 8, 1),
            (torch.bfloat16, 2, 8192, 65536, 64, 256, 4, 1, 65536, 8, 2)):
        p = _plan(mbt.OP_COLSUM, M, N, tm, tn, st, dt, fit=fit, ws=True, ld_src=ld)
        assert (p["consumer_warps"], p["col_group"]) == (W, g), p
        ring = 32 * W * (16 // es) * g * 4
        assert p["smem_bytes"] == 1024 + st * p["stage_bytes"] + ring, (p, ring)


def test_plan_warp_counts_on_16_kb_tiles():
    """Defaults on the ragged shapes' one-box tiles of 128 rows: the row sum
    takes 4 warps at 3 and 4 stages with two CTAs per SM; the column sum takes
    2 where four CTAs per SM are wanted (2 stages), so that four fit."""
    for st, fit, W, grid in ((3, 3, 4, 456), (4, 2, 4, 304), (2, 3, 4, 456)):
        p = _plan(mbt.OP_ROWSUM, 24577, 16383, 128, 64, st, torch.float16, fit=fit, ws=True,
                  ld_src=16384)
        assert (p["consumer_warps"], p["grid"]) == (W, grid), (st, p)
    p = _plan(mbt.OP_COLSUM, 24577, 16383, 128, 64, 2, torch.float16, fit=5, ws=True,
              ld_src=16384)
    assert (p["consumer_warps"], p["grid"], p["col_group"]) == (2, 608, 2)
    p = _plan(mbt.OP_COLSUM, 24577, 16383, 128, 64, 3, torch.float16, fit=3, ws=True,
              ld_src=16384)
    assert (p["consumer_warps"], p["grid"]) == (4, 456)
    p = _plan(mbt.OP_COLSUM, 24577, 16383, 128, 64, 4, torch.float16, fit=2, ws=True,
              ld_src=16384)
    assert (p["consumer_warps"], p["grid"]) == (8, 304)
    p = _plan(mbt.OP_COPY_ROWSUM, 8192, 65536, 64, 256, 4, torch.bfloat16, fit=1, ws=True)
    assert p["consumer_warps"] <= 8
    assert _plan(mbt.OP_COPY, 16384, 16384, 128, 64, 8, torch.float16)["consumer_warps"] == 4
    # an explicit count above 8: row and column sums only, never the 1-D kernels
    assert _plan(mbt.OP_ROWSUM, 8192, 65536, 64, 256, 2, torch.bfloat16, fit=1,
                 consumer_warps=12)["threads"] == 32 * 14
    with pytest.raises(mbt.MbtError):
        _plan(mbt.OP_COPY, 16384, 16384, 128, 64, 3, torch.float16, consumer_warps=9)
    with pytest.raises(mbt.MbtError):
        _plan(mbt.OP_ROWSUM, 1000, 63, 128, 64, 2, torch.float16, consumer_warps=9)
    with pytest.raises(mbt.MbtError):
        _plan(mbt.OP_ROWSUM, 100, 256, 64, 256, 2, torch.bfloat16, consumer_warps=17)
    # 3 stages of 256-row tiles: 4 warps cannot give each row a thread
    p = _plan(mbt.OP_ROWSUM, 16384, 32768, 256, 64, 3, torch.float16, fit=2, ws=True)
    assert p["consumer_warps"] == 8
    # row sum, 128 x 64 fp16 (16 KB stages), 3 stages: 3 CTAs per SM with 4 warps
    p = _plan(mbt.OP_ROWSUM, 24577, 16383, 128, 64, 3, torch.float16, fit=4, ws=True,
              ld_src=16384)
    assert p["grid"] == 456 and p["consumer_warps"] == 4
    # copy, 16 KB stages: 3 stages -> 2 CTAs, 1 stage -> 4 CTAs
    assert _plan(mbt.OP_COPY, 16384, 16384, 128, 64, 3, torch.float16, fit=4)["grid"] == 304
    assert _plan(mbt.OP_COPY, 16384, 16384, 128, 64, 1, torch.float16, fit=6)["grid"] == 608
    # bulk stores hold one stage: 2 stages count as 1 -> 4 CTAs
    assert _plan(mbt.OP_COPY, 16384, 16384, 128, 64, 2, torch.float16, fit=8,
                 store_mode=1)["grid"] == 608
    # an explicit value wins, capped by what fits
    assert _plan(mbt.OP_COPY, 16384, 16384, 128, 64, 3, torch.float16, fit=3,
                 ctas_per_sm=5)["grid"] == 456


def test_plan_fused_adds_a_store_warp_and_a_flush_warp():
    p = _plan(mbt.OP_COPY_ROWSUM, 24577, 16383, 128, 64, 3, torch.float16, fit=2, ws=True,
              ld_src=16384, ld_dst=16384)
    # 16 KB stages, one held by the store in flight: 2 live x 2 CTAs = 64 KB per SM;
    # producer, store warp, flush warp and (one-box tiles of 128 rows) 4 row-sum warps
    assert p["grid"] == 304 and p["consumer_warps"] == 4 and p["threads"] == 32 * 7
    p = _plan(mbt.OP_COPY_ROWSUM, 8192, 65536, 64, 256, 2, torch.bfloat16, fit=2, ws=True)
    assert p["consumer_warps"] == 8 and p["threads"] == 32 * 11   # four-box tiles: 8


def test_plan_tiled_rowsum_adds_a_flush_warp():
    """The tiled row sum runs a producer warp, a flush warp and the consumer
    warps; the flat row sum has no flush warp."""
    p = _plan(mbt.OP_ROWSUM, 8192, 65536, 64, 256, 2, torch.bfloat16, fit=2, ws=True)
    assert p["consumer_warps"] == 8 and p["threads"] == 32 * 10
    p = _plan(mbt.OP_ROWSUM, 24577, 16383, 128, 64, 3, torch.float16, fit=4, ws=True,
              ld_src=16384)
    assert p["threads"] == 32 * (2 + p["consumer_warps"])
    f = _plan(mbt.OP_ROWSUM, 1000, 63, 128, 64, 2, torch.float16, fit=4)
    assert f["flat"] == 1 and f["threads"] == 32 * (1 + f["consumer_warps"])


def test_plan_store_mode_default_follows_the_row_end():
    """0 picks bulk stores where rows end inside a 16-byte chunk, LSU stores
    otherwise (and always LSU with the unified pipeline)."""
    ragged = _plan(mbt.OP_COPY, 24577, 16383, 128, 64, 3, torch.float16, ld_src=16384,
                   ld_dst=16384)
    assert ragged["bulk_stores"] == 1 and ragged["consumer_warps"] == 1
    aligned = _plan(mbt.OP_COPY, 16384, 16384, 128, 64, 3, torch.float16)
    assert aligned["bulk_stores"] == 0 and aligned["consumer_warps"] == 4
    assert _plan(mbt.OP_COPY, 24577, 16383, 128, 64, 3, torch.float16, ld_src=16384,
                 ld_dst=16384, store_mode=2)["bulk_stores"] == 0
    assert _plan(mbt.OP_COPY, 16384, 16384, 128, 64, 3, torch.float16,
                 store_mode=1)["bulk_stores"] == 1
    assert _plan(mbt.OP_COPY, 24577, 16383, 128, 64, 3, torch.float16, ld_src=16384,
                 ld_dst=16384, pipeline=1)["bulk_stores"] == 0
    assert _plan(mbt.OP_COPY_ROWSUM, 1024, 4096, 64, 256, 2, torch.bfloat16)["bulk_stores"] == 1
    assert _plan(mbt.OP_ROWSUM, 1024, 4095, 64, 256, 2, torch.bfloat16,
                 ld_src=4096)["bulk_stores"] == 0


def test_plan_bulk_store_mode_uses_one_consumer_warp():
    p = _plan(mbt.OP_COPY, 16384, 16384, 128, 64, 4, torch.float16, store_mode=1,
              consumer_warps=7)
    assert p["consumer_warps"] == 1 and p["threads"] == 64


def test_plan_errors_and_limits():
    with pytest.raises(mbt.MbtError) as e:
        _plan(mbt.OP_COPY, 1024, 1024, 256, 64, 8, torch.float16, smem=200000)
    assert e.value.code == -4
    with pytest.raises(mbt.MbtError) as e:
        _plan(mbt.OP_ROWSUM, 1024, 1024, 256, 64, 2, torch.float16, consumer_warps=4)
    assert e.value.code == -3
    p = _plan(mbt.OP_ROWSUM, 1024, 1024, 256, 64, 2, torch.float16, fit=2)
    assert p["consumer_warps"] == 8
    p = _plan(mbt.OP_ROWSUM, 1024, 1024, 256, 64, 2, torch.float16, fit=1)
    assert p["consumer_warps"] == 8                  # one CTA per SM, one round a thread
    p = _plan(mbt.OP_ROWSUM, 1024, 1024, 256, 128, 2, torch.float16, fit=1)
    assert p["consumer_warps"] == 16                 # two rounds with 8 warps: the wide CTA


def test_plan_rowsum_multibox_tile():
    p = _plan(mbt.OP_ROWSUM, 8192, 65536, 64, 256, 3, torch.bfloat16, fit=1)
    assert p["boxes"] == 4 and p["tx_bytes"] == 32768 and p["stage_bytes"] == 32768
    assert p["grid"] == 128 and p["split"] == 0      # whole bands, one CTA each


def _warp_boxes(tile_m, boxes, W):
    """Boxes each consumer warp reads when thread t of 32 W sums chunks
    [sub cpr / tpr, (sub + 1) cpr / tpr) of row t % tile_m (sub = t // tile_m)."""
    tpr, cpr = 32 * W // tile_m, 8 * boxes
    out = []
    for w in range(W):
        seen = set()
        for t in range(32 * w, 32 * w + 32):
            if t >= tile_m * tpr:
                continue
            sub = t // tile_m
            seen |= {q // 8 for q in range(sub * cpr // tpr, (sub + 1) * cpr // tpr)}
        out.append(seen)
    return out


@pytest.mark.parametrize("tm,tn,dt,W", [
    (64, 256, torch.bfloat16, 8), (64, 256, torch.bfloat16, 4), (128, 128, torch.float16, 8),
    (128, 256, torch.bfloat16, 8), (64, 512, torch.float16, 8), (32, 256, torch.float32, 8),
    (96, 256, torch.bfloat16, 8), (128, 64, torch.float16, 4), (16, 512, torch.bfloat16, 1),
    (64, 128, torch.float32, 2), (256, 128, torch.float16, 8), (48, 128, torch.float16, 3),
])
def test_plan_box_barriers_only_where_each_warp_reads_one_box(tm, tn, dt, W):
    p = _plan(mbt.OP_ROWSUM, 4096, 8192, tm, tn, 2, dt, consumer_warps=W)
    # forced per-box pairs at 3 stages follow the same geometric rule;
    # the default keeps stage-wide pairs there
    p3 = _plan(mbt.OP_ROWSUM, 4096, 8192, tm, tn, 3, dt, consumer_warps=W, pipeline=3)
    assert p3["box_barriers"] == p["box_barriers"]
    assert _plan(mbt.OP_ROWSUM, 4096, 8192, tm, tn, 3, dt, consumer_warps=W)[
        "box_barriers"] == 0
    per_warp = _warp_boxes(tm, p["boxes"], W)
    every_thread_busy = (32 * W) % tm == 0
    one_box = all(len(b) == 1 for b in per_warp)
    assert p["box_barriers"] == int(p["boxes"] > 1 and every_thread_busy and one_box)
    if p["box_barriers"]:
        # the barrier counts: every box is read by the same number of warps
        counts = [sum(1 for b in per_warp if b == {k}) for k in range(p["boxes"])]
        assert counts == [W // p["boxes"]] * p["boxes"]
    # never for the fused operation, the flat kernels, or with pipeline=2
    assert _plan(mbt.OP_COPY_ROWSUM, 4096, 8192, tm, tn, 2, dt, consumer_warps=W)[
        "box_barriers"] == 0
    assert _plan(mbt.OP_ROWSUM, 4096, 8192, tm, tn, 2, dt, consumer_warps=W,
                 pipeline=2)["box_barriers"] == 0
    flat = _plan(mbt.OP_ROWSUM, 4096, 8191, tm, tn, 2, dt, consumer_warps=W)  # odd pitch
    assert flat["flat"] == 1 and flat["box_barriers"] == 0


def test_plan_box_barriers_in_the_bench_row_sum():
    p = _plan(mbt.OP_ROWSUM, 8192, 65536, 64, 256, 2, torch.bfloat16, fit=4, ws=True)
    assert p["boxes"] == 4 and p["consumer_warps"] == 8 and p["box_barriers"] == 1


def _ranges(G, units, gran):
    return [((b * units // G) * gran, ((b + 1) * units // G) * gran) for b in range(G)]


@pytest.mark.parametrize("M,N,tm,tn,dt,sms,fit", [
    (8192, 65536, 64, 256, torch.bfloat16, 152, 1),
    (8192, 65536, 64, 256, torch.bfloat16, 152, 2),
    (12289, 8191, 128, 32, torch.float32, 152, 2),
    (24577, 16383, 128, 64, torch.float16, 152, 3),
    (1000, 300, 16, 64, torch.float16, 7, 1),
    (64, 64, 64, 64, torch.float16, 152, 4),
])
def test_plan_rowsum_split_covers_every_tile_once(M, N, tm, tn, dt, sms, fit):
    es = torch.empty(0, dtype=dt).element_size()
    ld = -(-N * es // 16) * 16 // es                    # pitched rows
    p = _plan(mbt.OP_ROWSUM, M, N, tm, tn, 3, dt, sms=sms, fit=fit, ws=True, ld_src=ld)
    tiles_n, T = p["tiles_n"], p["num_tiles"]
    if not p["split"]:
        assert p["workspace_bytes"] == 0
        return
    G = p["grid"]
    assert G <= min(T, sms * fit) and G >= min(T, sms * min(fit, 2))
    rng = _ranges(G, T, 1)
    assert rng[0][0] == 0 and rng[-1][1] == T
    assert all(a[1] == b[0] for a, b in zip(rng, rng[1:]))
    # brute-force contributors per band
    contrib = {}
    for b, (lo, hi) in enumerate(rng):
        for band in range(lo // tiles_n, (hi - 1) // tiles_n + 1) if hi > lo else []:
            contrib.setdefault(band, []).append(b)
    kmax = max(len(v) for v in contrib.values())
    assert p["kmax"] == kmax
    bands = p["tiles_m"]
    assert p["workspace_bytes"] == ((bands * 4 + 255) // 256) * 256 + bands * kmax * tm * 4


@pytest.mark.parametrize("M,N,tm,tn,dt,sms,fit", [
    (8192, 65536, 64, 256, torch.bfloat16, 152, 2),
    (65536, 8192, 64, 256, torch.bfloat16, 152, 2),
    (12289, 8191, 128, 32, torch.float32, 152, 3),
    (24577, 16383, 128, 64, torch.float16, 152, 3),
    (300, 1000, 16, 64, torch.float16, 7, 1),
    (64, 64, 64, 64, torch.float16, 152, 4),
])
def test_plan_colsum_split_covers_every_tile_once(M, N, tm, tn, dt, sms, fit):
    """Column sums take tiles in strip-group order: groups of col_group
    adjacent strips, band by band inside a group.  CTA b owns an even,
    contiguous range of that order; every tile is owned once, and a strip's
    contributors are the CTAs from the owner of its first tile to the owner
    of its last."""
    es = torch.empty(0, dtype=dt).element_size()
    ld = -(-N * es // 16) * 16 // es
    p = _plan(mbt.OP_COLSUM, M, N, tm, tn, 3, dt, sms=sms, fit=fit, ws=True, ld_src=ld)
    tiles_m, strips, T = p["tiles_m"], p["tiles_n"], p["num_tiles"]
    if not p["split"]:
        assert p["workspace_bytes"] == 0 and p["grid"] == min(strips, sms * fit)
        assert p["col_group"] == 1
        return
    g = p["col_group"]
    assert g == (2 if tn * es == 128 else 1)
    # order position of every tile, built band by band inside each group
    pos = {}
    t = 0
    for g0 in range(0, strips, g):
        wg = min(g, strips - g0)
        for band in range(tiles_m):
            for k in range(wg):
                pos[(band, g0 + k)] = t
                t += 1
    assert t == T and len(set(pos.values())) == T
    G = p["grid"]
    owner = [None] * T
    for b, (lo, hi) in enumerate(_ranges(G, T, 1)):
        for x in range(lo, hi):
            owner[x] = b
    assert None not in owner
    kmax = 1
    for s_ in range(strips):
        own = [owner[pos[(band, s_)]] for band in range(tiles_m)]
        assert own == sorted(own)
        kmax = max(kmax, own[-1] - own[0] + 1)
    assert p["kmax"] == kmax
    assert p["workspace_bytes"] == ((strips * 4 + 255) // 256) * 256 + strips * kmax * tn * 4


def test_plan_colsum_limits_and_errors():
    # one thread per 16-byte chunk column: 1024-byte rows (64 chunks) need 2 warps
    with pytest.raises(mbt.MbtError) as e:
        _plan(mbt.OP_COLSUM, 1024, 4096, 64, 512, 2, torch.float16, consumer_warps=1)
    assert e.value.code == -3
    assert _plan(mbt.OP_COLSUM, 1024, 4096, 64, 512, 2, torch.float16,
                 consumer_warps=2)["consumer_warps"] == 2
    # a 16-byte row pitch is required (no flat column sum)
    with pytest.raises(mbt.MbtError) as e:
        _plan(mbt.OP_COLSUM, 100, 4095, 64, 256, 2, torch.bfloat16)
    assert e.value.code == -2
    # barrier layouts and bulk stores belong to other operations
    for kw in ({"pipeline": 1}, {"pipeline": 2}, {"pipeline": 3}, {"store_mode": 1}):
        with pytest.raises(mbt.MbtError) as e:
            _plan(mbt.OP_COLSUM, 1024, 4096, 64, 256, 2, torch.bfloat16, **kw)
        assert e.value.code in (-1, -3), kw
    p = _plan(mbt.OP_COLSUM, 8192, 65536, 64, 256, 2, torch.bfloat16, fit=4, ws=True)
    assert p["consumer_warps"] == 8 and p["threads"] == 320 and p["box_barriers"] == 0   # + flush warp
    assert p["grid"] == 304 and p["split"] == 1


def test_colsum_argument_errors():
    assert C.tile_colsum(A, B + 2, 8, 64, 64, 64, 2, 0, None) == -2      # out not 4-aligned
    assert C.tile_colsum(A, None, 8, 64, 64, 64, 2, 0, None) == -1
    assert C.tile_colsum(A + 8, B, 8, 64, 64, 64, 2, 0, None) == -2      # src not 16-aligned
    assert C.tile_colsum(A, B, 8, 64, 0, 64, 2, 0, None) == -1
    assert C.tile_colsum(A, B, 8, 64, 64, 32, 2, 0, None) == -3          # 64-byte rows
    assert C.tile_colsum(None, None, 0, 0, 64, 64, 2, 0, None) == 0
    o = Opts(); o.ld_dst = 64                                             # sums have no dst pitch
    assert C.tile_colsum_ex(A, B, 8, 64, 64, 64, 2, 0, None, ctypes.byref(o)) == -1


def test_ctypes_mirrors_match_the_c_structs(tmp_path):
    """Sizes and field offsets of mbt_opts / mbt_plan as the C compiler lays
    them out, against the binding's ctypes mirrors."""
    import subprocess
    fields = {"mbt_opts": [n for n, _ in Opts._fields_],
              "mbt_plan": [n for n, _ in mbt.Plan._fields_]}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "mbtile.h"', "int main(void) {"]
    for struct, names in fields.items():
        lines.append(f'printf("{struct} %zu\\n", sizeof({struct}));')
        for n in names:
            lines.append(f'printf("{struct}.{n} %zu\\n", offsetof({struct}, {n}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe)], check=True)
    out = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                 check=True).stdout.splitlines())
    for struct, cls in (("mbt_opts", Opts), ("mbt_plan", mbt.Plan)):
        assert int(out[struct]) == ctypes.sizeof(cls), struct
        for n, _ in cls._fields_:
            assert int(out[f"{struct}.{n}"]) == getattr(cls, n).offset, (struct, n)


def test_binding_exports_what_it_lists():
    assert all(hasattr(mbt, name) for name in mbt.__all__)
    for name in ("tile_colsum", "tile_copy_host", "tile_rowsum_host", "tile_colsum_host"):
        assert name in mbt.__all__
