"""Sizes past 2^32 bytes and concurrent host threads.

Large: every byte offset computation must be 64-bit.  Inputs are drawn on the
device (seeded); the results are checked against the CPU oracle on sampled
rows (first, last, and rows near the 4 GiB and 2^32-element boundaries).
Concurrency: several host threads, each with its own stream (and workspace),
call the library at the same time."""
import threading

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


def sample_rows(M, N, es):
    rows = {0, 1, M - 2, M - 1, M // 2}
    for boundary in (1 << 32, 1 << 33):            # bytes
        r = boundary // (N * es)
        rows |= {r - 1, r, r + 1}
    r = (1 << 32) // N                               # elements
    rows |= {r - 1, r, r + 1}
    return sorted(x for x in rows if 0 <= x < M)


@pytest.mark.parametrize("dtype,M,N,tm,tn", [
    ("f16", 131072, 32832, 128, 64),      # 8.6 GB, pitch 65,664 B: tiled path
    ("bf16", 70001, 65535, 64, 256),      # 9.2 GB, 131,070-byte rows: 1-D bulk-copy path
])
def test_copy_and_rowsum_past_4gib(dtype, M, N, tm, tn):
    es = synthetic.ESIZE[dtype]
    x = synthetic.make_matrix(M, N, dtype, "uniform", seed=4242, draw_on="cuda:0")
    y = torch.empty_like(x)
    mbt.tile_copy(x, y, tm, tn, 3)
    out = mbt.tile_rowsum(x, None, tm, tn, 2)
    assert mbt.tile_status()[0] == 0
    rows = sample_rows(M, N, es)
    xs = x[rows].cpu()
    ys = y[rows].cpu()
    want = torch.empty_like(xs)
    oracle.copy(xs, want)
    assert torch.equal(bits(ys), bits(want))
    worst, _, _ = rowsum_errors(out[rows], xs)
    assert worst <= ROWSUM_RTOL
    del x, y
    torch.cuda.empty_cache()


def test_concurrent_host_threads_with_own_streams():
    jobs = []
    for t in range(6):
        dtype = ("f16", "bf16", "f32")[t % 3]
        M, N = 1000 + 37 * t, 3000 + 101 * t
        x = synthetic.make_matrix(M, N, dtype, "normal", seed=t,
                                  ld=synthetic.pitched_ld(N, dtype))
        jobs.append((dtype, M, N, x))
    results = [None] * len(jobs)
    errors = []

    def work(i):
        try:
            dtype, M, N, x = jobs[i]
            s = torch.cuda.Stream()
            tm, tn = {"f16": (128, 64), "bf16": (64, 256), "f32": (128, 32)}[dtype]
            with torch.cuda.stream(s):
                xd = x.cuda(non_blocking=False)[:, :N]
                yd = torch.empty(x.shape, dtype=x.dtype, device="cuda")[:, :N]   # same pitch
                ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
                for _ in range(20):
                    mbt.tile_copy(xd, yd, tm, tn, 3, stream=s)
                    out = mbt.tile_rowsum(xd, None, tm, tn, 2, workspace=ws, stream=s)
                s.synchronize()
                results[i] = (yd.cpu(), out.cpu())
        except Exception as exc:       # reported below
            errors.append(repr(exc))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert mbt.tile_status()[0] == 0
    for (dtype, M, N, x), (y, out) in zip(jobs, results):
        want = torch.empty(M, N, dtype=x.dtype)
        oracle.copy(x[:, :N], want)
        assert torch.equal(bits(y), bits(want))
        assert rowsum_errors(out, x[:, :N])[0] <= ROWSUM_RTOL
