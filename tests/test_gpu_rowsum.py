"""GPU parity of tile_rowsum against the binary64 CPU oracle, through the C
ABI: fp32 sums within 1e-5 x max(|sum|, sqrt(sum of squares)) per row, exact
on exactly representable cases, run-to-run bit-identical."""
import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import ROWSUM_RTOL, rowsum_errors
from oracle.pipeline_state import sequence

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


def run_rowsum(x_h, N, *args, **kw):
    x = x_h.cuda()
    out = mbt.tile_rowsum(x[:, :N], None, *args, **kw)
    code, info = mbt.tile_status()
    assert code == 0, info
    return out


CASES = [
    # dtype, dist, M, N, tile_m, tile_n, stages, split
    ("bf16", "normal", 200, 1000, 64, 256, 3, True),
    ("bf16", "normal", 200, 1000, 64, 256, 3, False),
    ("f16", "uniform", 1, 1, 128, 64, 1, True),
    ("f16", "uniform", 300, 4100, 128, 64, 4, True),
    ("f32", "uniform", 257, 8191, 128, 32, 3, True),
    ("f32", "normal", 1000, 33, 16, 64, 2, True),
    ("f16", "normal", 65, 20000, 8, 512, 2, True),
    ("bf16", "uniform", 4097, 300, 256, 64, 5, True),
    ("f16", "uniform", 37, 70000, 32, 128, 6, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_rowsum_matches_oracle(case):
    dtype, dist, M, N, tm, tn, st, split = case
    ld = synthetic.pitched_ld(N, dtype) + 16 // synthetic.ESIZE[dtype]
    x = synthetic.make_matrix(M, N, dtype, dist, seed=M + N, ld=ld)
    out = run_rowsum(x, N, tm, tn, st, split=split)
    worst, rel, _ = rowsum_errors(out, x[:, :N])
    assert worst <= ROWSUM_RTOL, (worst, rel)


def test_all_ones_exact_and_empty_rows():
    x = torch.ones(300, 5000, dtype=torch.bfloat16)
    out = run_rowsum(x, 5000, 64, 256, 3)
    assert out.cpu().tolist() == [5000.0] * 300
    z = mbt.tile_rowsum(torch.empty(7, 0, dtype=torch.float16, device="cuda"), None, 64, 64, 2)
    assert mbt.tile_status()[0] == 0
    assert z.cpu().tolist() == [0.0] * 7


def test_repeat_calls_bit_identical_and_workspace_reuse():
    x = synthetic.make_matrix(1000, 30000, "bf16", "normal", seed=4)
    xd = x.cuda()
    a = mbt.tile_rowsum(xd, None, 64, 256, 3)
    b = mbt.tile_rowsum(xd, None, 64, 256, 3)
    c = mbt.tile_rowsum(xd, None, 64, 256, 4)
    assert mbt.tile_status()[0] == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert rowsum_errors(c, x)[0] <= ROWSUM_RTOL


def test_one_workspace_shared_by_different_shapes():
    """A workspace is reused across calls whose ticket and partial regions
    differ in size; every call must leave all of it zero-filled."""
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    shapes = [(300, 40000, 64, 256), (8192, 4096, 64, 256), (1000, 30000, 64, 256),
              (5000, 9000, 128, 64)]
    for M, N, tm, tn in shapes:
        x = synthetic.make_matrix(M, N, "bf16", "normal", seed=M)
        out = mbt.tile_rowsum(x.cuda(), None, tm, tn, 3, workspace=ws)
        assert mbt.tile_status()[0] == 0
        assert rowsum_errors(out, x)[0] <= ROWSUM_RTOL, (M, N)
        assert int(ws.count_nonzero()) == 0
        # the library's own workspace on a fresh stream, grown as the plans
        # need more tickets or partial sums, gives the same bits
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        own = mbt.tile_rowsum(x.cuda(), None, tm, tn, 3, stream=s)
        torch.cuda.synchronize()
        assert mbt.tile_status()[0] == 0
        assert torch.equal(own.view(torch.int32), out.view(torch.int32))


def test_library_workspace_grows_across_shapes_on_one_stream():
    """Shapes whose plans need more band tickets or partial sums than the
    stream's workspace holds: it is replaced in stream order, and every call
    (before and after the growth) gives the caller's-workspace bits."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    for M, N, tm, tn in [(300, 40000, 64, 256), (60000, 2048, 32, 256), (1000, 30000, 64, 256),
                         (200000, 1024, 16, 512), (8192, 4096, 64, 256)]:
        x = synthetic.make_matrix(M, N, "bf16", "normal", seed=M + 1)
        xd = x.cuda()
        need = mbt.tile_rowsum_workspace_bytes(M, N, tm, tn, 2, torch.bfloat16)
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
        want = mbt.tile_rowsum(xd, None, tm, tn, 2, workspace=ws)
        torch.cuda.synchronize()
        got = mbt.tile_rowsum(xd, None, tm, tn, 2, stream=s)
        torch.cuda.synchronize()
        assert mbt.tile_status()[0] == 0
        assert torch.equal(got.view(torch.int32), want.view(torch.int32)), (M, N)
        assert rowsum_errors(got, x)[0] <= ROWSUM_RTOL, (M, N)


def test_log_of_one_cta_pipeline():
    x = synthetic.make_matrix(128, 512, "f16", "uniform", seed=12)
    log = torch.zeros(2 * 16 * 4, dtype=torch.int32, device="cuda")
    out = run_rowsum(x, 512, 128, 64, 3, consumer_warps=4, max_ctas=1, split=False, log=log)
    assert rowsum_errors(out, x)[0] <= ROWSUM_RTOL
    rec = log.view(2, 16, 4).cpu()
    assert [(s, p) for _, s, p, _ in rec[0, :8].tolist()] == sequence(3, 1, 8)
    assert [(s, p) for _, s, p, _ in rec[1, :8].tolist()] == sequence(3, 0, 8)


FULL = [
    # pipelined row reduction: bf16 8192 x 65536, normal(0,1), 64 x 256 tiles
    ("bf16", "normal", 8192, 65536, 64, 256, (2, 3, 4), 1004),
    # ragged fp32 12289 x 8191 and fp16 24577 x 16383, pitched rows
    ("f32", "uniform", 12289, 8191, 128, 32, (3,), 1005),
    ("f16", "uniform", 24577, 16383, 128, 64, (3,), 1006),
]


@pytest.mark.parametrize("case", FULL, ids=lambda c: f"{c[0]}-{c[2]}x{c[3]}")
def test_full_size_configs(case):
    dtype, dist, M, N, tm, tn, stage_list, seed = case
    x = synthetic.make_matrix(M, N, dtype, dist, seed, ld=synthetic.pitched_ld(N, dtype))
    xd = x.cuda()
    for st in stage_list:
        out = mbt.tile_rowsum(xd[:, :N], None, tm, tn, st)
        assert mbt.tile_status()[0] == 0
        worst, rel, _ = rowsum_errors(out, x[:, :N])
        assert worst <= ROWSUM_RTOL, (st, worst, rel)


def test_library_workspace_per_stream():
    """Without a workspace of the caller's, each stream gets the library's
    own (allocated and zero-filled in stream order on its first call): row
    sums on 20 streams at once are right and bit-identical to the sums with a
    caller's workspace; releasing a stream's workspace and calling again
    allocates a fresh one."""
    x = synthetic.make_matrix(3000, 20000, "bf16", "normal", seed=17)
    xd = x.cuda()
    need = mbt.tile_rowsum_workspace_bytes(3000, 20000, 64, 256, 2, torch.bfloat16)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    want = mbt.tile_rowsum(xd, None, 64, 256, 2, workspace=ws)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(20)]
    outs = []
    for rep in range(2):
        for s in streams:
            s.wait_stream(torch.cuda.current_stream())
            outs.append(mbt.tile_rowsum(xd, None, 64, 256, 2, stream=s))
        torch.cuda.synchronize()
        if rep == 0:
            for s in streams[:5]:
                mbt.tile_workspace_release(s)
    assert mbt.tile_status()[0] == 0
    for o in outs:
        assert torch.equal(o.view(torch.int32), want.view(torch.int32))
    assert rowsum_errors(want, x)[0] <= ROWSUM_RTOL
    assert int(ws.count_nonzero()) == 0              # the caller's is left zero-filled


def test_library_workspace_recovers_after_timeout():
    """A stalled call on the library's workspace may leave band tickets set;
    the workspace alternates two ticket sets and each call zeroes the one it
    does not use, so every later call on the stream is right."""
    M, N = 2048, 16384
    x = synthetic.make_matrix(M, N, "bf16", "normal", seed=18)
    xd = x.cuda()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    want = mbt.tile_rowsum(xd, None, 64, 256, 2, stream=s)
    for fault in (2, 1, 2):
        mbt.tile_rowsum(xd, None, 64, 256, 2, fault=fault, wait_budget_ns=20_000_000, stream=s)
        code, info = mbt.tile_status(s)
        assert code == mbt.MBT_ERR_TIMEOUT, info
        for _ in range(3):
            out = mbt.tile_rowsum(xd, None, 64, 256, 2, stream=s)
            assert mbt.tile_status(s)[0] == 0
            assert torch.equal(out.view(torch.int32), want.view(torch.int32))
    assert rowsum_errors(want, x)[0] <= ROWSUM_RTOL


def test_library_workspace_is_not_allocated_during_capture():
    """The first call on a fresh stream inside a stream capture would have to
    allocate: refused with MBT_ERR_WORKSPACE before anything is enqueued; after
    a call outside the capture the same call captures and replays right."""
    M, N = 1000, 20480
    x = synthetic.make_matrix(M, N, "bf16", "normal", seed=19)
    xd = x.cuda()
    out = torch.empty(M, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.capture_begin()
        try:
            rc = mbt.C.tile_rowsum(xd.data_ptr(), out.data_ptr(), M, N, 64, 256, 2,
                                   mbt.DTYPE_CODE[xd.dtype], s.cuda_stream)
        finally:
            g.capture_end()
    assert rc == -8
    torch.cuda.synchronize()
    mbt.tile_rowsum(xd, out, 64, 256, 2, stream=s)   # outside: allocates
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):                              # an odd count of calls
            mbt.tile_rowsum(xd, out, 64, 256, 2, stream=s)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert mbt.tile_status()[0] == 0
        assert rowsum_errors(out, x)[0] <= ROWSUM_RTOL


@pytest.mark.parametrize("split", [False, True])
def test_flush_ring_wraps_many_times(split):
    """Three CTAs over 1563 single-tile bands: each CTA's consumers post ~520
    segments through the two-slot flush ring (with a workspace, bands shared
    by two CTAs add their partials through tickets)."""
    M, N = 100003, 256
    x = synthetic.make_matrix(M, N, "bf16", "normal", seed=77)
    out = mbt.tile_rowsum(x.cuda(), None, 64, 256, 2, max_ctas=3, split=split)
    assert mbt.tile_status()[0] == 0
    assert rowsum_errors(out, x)[0] <= ROWSUM_RTOL


def test_library_workspace_from_concurrent_host_threads():
    """Host threads calling the plain row sum at once, each on a stream of its own
    and each through the per-thread default stream (cudaStreamPerThread, one
    handle for all threads, a different stream in each): every thread's
    workspace is its own, and every result is the caller's-workspace bits."""
    import ctypes
    import threading

    M, N = 3000, 20000
    x = synthetic.make_matrix(M, N, "bf16", "normal", seed=23)
    xd = x.cuda()
    need = mbt.tile_rowsum_workspace_bytes(M, N, 64, 256, 2, torch.bfloat16)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    want = mbt.tile_rowsum(xd, None, 64, 256, 2, workspace=ws)
    torch.cuda.synchronize()
    per_thread_stream = 0x2   # cudaStreamPerThread
    results, errors = {}, []

    def worker(k):
        try:
            torch.cuda.set_device(0)
            outs = []
            if k % 2 == 0:
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                for _ in range(6):
                    outs.append(mbt.tile_rowsum(xd, None, 64, 256, 2, stream=s))
                s.synchronize()
            else:
                for _ in range(6):
                    o = torch.empty(M, dtype=torch.float32, device="cuda")
                    torch.cuda.synchronize()
                    rc = mbt.C.tile_rowsum(xd.data_ptr(), o.data_ptr(), M, N, 64, 256, 2,
                                           mbt.DTYPE_CODE[xd.dtype], per_thread_stream)
                    assert rc == 0, rc
                    outs.append(o)
                torch.cuda.synchronize()
            results[k] = outs
        except Exception as e:   # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(6)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert mbt.tile_status()[0] == 0
    for k, outs in results.items():
        for o in outs:
            assert torch.equal(o.view(torch.int32), want.view(torch.int32)), k
    assert rowsum_errors(want, x)[0] <= ROWSUM_RTOL
