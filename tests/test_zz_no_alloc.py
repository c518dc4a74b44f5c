"""tile_rowsum_noalloc: the row sum for callers that cannot allocate device
memory (their memory is owned by another allocator, or they must not call
cudaMalloc / cudaFree on a latency-critical path).  Its scratch is a static
device array inside the library; this file checks, through the C ABI, that it
returns what the workspace-taking entry point returns, call after call, and
that shapes too large for the array are refused before anything runs.

Collected last on purpose (file name), so that a run stopping at the first
failure has already run every other test."""
import ctypes

import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import ROWSUM_RTOL
from mbarrier_async_tile_gb300 import C, Opts

pytestmark = pytest.mark.gpu

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


def call_noalloc(x, out, tm, tn, st, ld):
    o = Opts()
    o.ld_src = ld
    stream = torch.cuda.current_stream().cuda_stream
    return C.tile_rowsum_noalloc(x.data_ptr(), out.data_ptr(), x.shape[0], x.shape[1], tm, tn,
                                 st, mbt.DTYPE_CODE[x.dtype], stream, ctypes.byref(o))


@pytest.mark.parametrize("dtype,dist,M,N,tm,tn,st", [
    ("bf16", "normal", 8192, 65536, 64, 256, 3),     # bands split over the grid
    ("f32", "uniform", 12289, 8191, 128, 32, 3),
    ("f16", "uniform", 300, 4100, 128, 64, 4),
])
def test_matches_workspace_entry_point_on_two_calls(dtype, dist, M, N, tm, tn, st):
    ld = synthetic.pitched_ld(N, dtype)
    x_h = synthetic.make_matrix(M, N, dtype, dist, seed=2024, ld=ld)
    x = x_h.cuda()[:, :N]
    need = mbt.tile_rowsum_workspace_bytes(M, N, tm, tn, st, x.dtype, ld_src=ld)
    assert need <= SCRATCH_BYTES
    want = mbt.tile_rowsum(x, None, tm, tn, st)          # caller-provided workspace
    assert mbt.tile_status()[0] == 0
    _, sq = oracle.rowsum(x_h[:, :N], with_sumsq=True)
    scale = torch.maximum(want.cpu().double().abs(), sq.sqrt())
    for _ in range(2):
        out = torch.full((M,), float("nan"), device="cuda")
        assert call_noalloc(x, out, tm, tn, st, ld) == 0
        code, info = mbt.tile_status()
        assert code == 0, info
        diff = (out.cpu().double() - want.cpu().double()).abs()
        assert bool((diff <= ROWSUM_RTOL * scale).all())


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
