"""tile_rowsum_noalloc: the row sum for callers that cannot allocate device
memory (their memory is owned by another allocator, or they must not call
cudaMalloc / cudaFree on a latency-critical path).  Its scratch is a static
device array inside the library.  Through the C ABI, this file checks that:

* its sums are bit-identical to tile_rowsum_ex's with a workspace of the
  caller's on the same plan, call after call, and within the row-sum
  tolerance of the binary64 oracle;
* shapes that need no scratch (the 1-D bulk-copy path, empty shapes, bands
  that are never split) still give the oracle's sums;
* a call after one that stopped on a timed-out wait (tickets and partials
  left in the shared array) is right again;
* shapes too large for the array, and options that name a workspace, are
  refused before anything runs.

Collected last on purpose (file name), so that a run stopping at the first
failure has already run every other test."""
import ctypes

import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import ROWSUM_RTOL, rowsum_errors
from mbarrier_async_tile_gb300 import C, Opts

pytestmark = pytest.mark.gpu

MBT_ERR_ARG = -1
MBT_ERR_WORKSPACE = -8
SCRATCH_BYTES = 1 << 20


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)
    fn = C.tile_rowsum_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                   ctypes.POINTER(Opts)]
    fn.restype = ctypes.c_int


def _stream():
    return torch.cuda.current_stream().cuda_stream


def call_noalloc(x, out, tm, tn, st, ld, **opt):
    o = Opts()
    o.ld_src = ld
    for k, v in opt.items():
        setattr(o, k, v)
    return C.tile_rowsum_noalloc(x.data_ptr() if x.numel() else 16,
                                 out.data_ptr() if out.numel() else 16,
                                 x.shape[0], x.shape[1], tm, tn, st, mbt.DTYPE_CODE[x.dtype],
                                 _stream(), ctypes.byref(o))


def call_ex_with_workspace(x, out, tm, tn, st, ld, ws):
    """tile_rowsum_ex with a zero-filled workspace of the caller's: the plan
    the no-alloc entry point runs with its own array."""
    o = Opts()
    o.ld_src = ld
    o.workspace = ws.data_ptr()
    o.workspace_bytes = ws.numel()
    return C.tile_rowsum_ex(x.data_ptr(), out.data_ptr(), x.shape[0], x.shape[1], tm, tn, st,
                            mbt.DTYPE_CODE[x.dtype], _stream(), ctypes.byref(o))


@pytest.mark.parametrize("dtype,dist,M,N,tm,tn,st", [
    ("bf16", "normal", 8192, 65536, 64, 256, 3),     # 128 bands split over the grid
    ("f32", "uniform", 12289, 8191, 128, 32, 3),     # ragged, pitched
    ("f16", "uniform", 300, 4100, 128, 64, 4),
])
def test_bit_identical_to_workspace_entry_point_and_oracle(dtype, dist, M, N, tm, tn, st):
    ld = synthetic.pitched_ld(N, dtype)
    x_h = synthetic.make_matrix(M, N, dtype, dist, seed=2024, ld=ld)
    x = x_h.cuda()[:, :N]
    need = mbt.tile_rowsum_workspace_bytes(M, N, tm, tn, st, x.dtype, ld_src=ld)
    assert 0 < need <= SCRATCH_BYTES          # the bands are split: the array is used
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    want = torch.full((M,), float("nan"), device="cuda")
    assert call_ex_with_workspace(x, want, tm, tn, st, ld, ws) == 0
    assert mbt.tile_status()[0] == 0
    worst, rel, _ = rowsum_errors(want, x_h[:, :N])
    assert worst <= ROWSUM_RTOL, (worst, rel)
    for _ in range(2):
        out = torch.full((M,), float("nan"), device="cuda")
        assert call_noalloc(x, out, tm, tn, st, ld) == 0
        code, info = mbt.tile_status()
        assert code == 0, info
        assert torch.equal(out.view(torch.int32), want.view(torch.int32))
        worst, rel, _ = rowsum_errors(out, x_h[:, :N])
        assert worst <= ROWSUM_RTOL, (worst, rel)


@pytest.mark.parametrize("case", ["flat-63-columns", "whole-bands", "no-columns", "no-rows"])
def test_shapes_that_need_no_scratch(case):
    if case == "flat-63-columns":      # dense rows of 126 bytes: the 1-D bulk-copy kernels
        M, N, ld, tm, tn, st = 5000, 63, 63, 64, 256, 2
    elif case == "whole-bands":        # more bands than the grid holds CTAs: no split
        M, N, ld, tm, tn, st = 100000, 256, 256, 64, 256, 2
    elif case == "no-columns":
        M, N, ld, tm, tn, st = 77, 0, 0, 64, 256, 2
    else:
        M, N, ld, tm, tn, st = 0, 512, 512, 64, 256, 2
    x_h = synthetic.make_matrix(M, N, "bf16", "normal", seed=99) if M * N else \
        torch.empty(M, N, dtype=torch.bfloat16)
    if N and M:
        assert mbt.tile_rowsum_workspace_bytes(M, N, tm, tn, st, torch.bfloat16, ld_src=ld) == 0
    x = x_h.cuda()
    for _ in range(2):
        out = torch.full((M,), float("nan"), device="cuda")
        assert call_noalloc(x, out, tm, tn, st, max(ld, 1)) == 0
        assert mbt.tile_status()[0] == 0
        if M:
            assert rowsum_errors(out, x_h)[0] <= ROWSUM_RTOL


def test_call_after_a_timed_out_call_is_right():
    """A call whose consumers never release a stage (test hook 2, 20 ms wait
    budget) stops with a timeout after some CTAs have taken band tickets and
    written partial sums into the shared array; the next call clears what it
    uses and returns the oracle's sums."""
    M, N, tm, tn, st = 2048, 16384, 64, 256, 2
    x_h = synthetic.make_matrix(M, N, "bf16", "normal", seed=4242)
    x = x_h.cuda()
    assert 0 < mbt.tile_rowsum_workspace_bytes(M, N, tm, tn, st, torch.bfloat16) <= SCRATCH_BYTES
    out = torch.zeros(M, device="cuda")
    assert call_noalloc(x, out, tm, tn, st, N, fault=2, wait_budget_ns=20_000_000) == 0
    code, info = mbt.tile_status()
    assert code == mbt.MBT_ERR_TIMEOUT, info
    for _ in range(2):
        out = torch.full((M,), float("nan"), device="cuda")
        assert call_noalloc(x, out, tm, tn, st, N) == 0
        assert mbt.tile_status()[0] == 0
        assert rowsum_errors(out, x_h)[0] <= ROWSUM_RTOL


def test_options_naming_a_workspace_are_refused():
    M, N = 1024, 4096
    x = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(M, dtype=torch.float32, device="cuda")
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    assert call_noalloc(x, out, 64, 256, 2, N, workspace=ws.data_ptr(),
                        workspace_bytes=ws.numel()) == MBT_ERR_ARG
    assert call_noalloc(x, out, 64, 256, 2, N, workspace_bytes=256) == MBT_ERR_ARG
    assert mbt.tile_status()[0] == 0


def test_shape_needing_more_scratch_is_refused():
    # 2^20 rows in 16384 bands split over the persistent grid need several MiB
    # of partial sums: refused on the host, nothing launched.
    M, N = 1 << 20, 1024
    need = mbt.tile_rowsum_workspace_bytes(M, N, 64, 256, 3, torch.bfloat16)
    assert need > SCRATCH_BYTES
    x = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(M, dtype=torch.float32, device="cuda")
    assert call_noalloc(x, out, 64, 256, 3, N) == MBT_ERR_WORKSPACE
    assert mbt.tile_status()[0] == 0
    assert int(out.count_nonzero()) == 0
