"""Host-buffer forms (tile_copy_host, tile_rowsum_host, tile_colsum_host):
HOST matrices moved through the device in row slabs with the copies in, the
tile pipeline and the copies out overlapped on three streams.  Copies are
bit-exact against the oracle (pads of dst untouched), row and column sums
within the fp32 bound; any host pitch, ragged slab counts, pinned and
pageable memory, stalls, threads."""
import threading

import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import DTYPES, ROWSUM_RTOL, bits, colsum_errors, rowsum_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


def host_case(dtype, M, N, ld_s, ld_d, seed, pinned):
    src = synthetic.make_matrix(M, N, dtype, "uniform", seed, ld=ld_s)
    dst = torch.empty(M, ld_d, dtype=DTYPES[dtype])
    synthetic.fill_bits(dst, synthetic.POISON_BITS[dtype])
    if pinned:
        src, dst = src.pin_memory(), dst.pin_memory()
    want = dst.clone()
    oracle.copy(src[:, :N], want[:, :N])
    return src, dst, want


COPY_CASES = [
    # dtype, M, N, host ld_src, host ld_dst, slab rows (0 = default), pinned
    ("f16", 1000, 1000, 1003, 1010, 97, True),     # odd host pitches, 11 ragged slabs
    ("bf16", 777, 4096, 4096, 4100, 64, True),     # dense src, padded dst
    ("f32", 513, 8191, 8191, 8192, 100, True),     # rows not a multiple of 16 bytes
    ("f16", 300, 2048, 2050, 2048, 0, False),      # pageable, one slab
    ("f16", 1, 70001, 70001, 70001, 0, True),      # a single long row
]


@pytest.mark.parametrize("case", COPY_CASES, ids=lambda c: "-".join(map(str, c)))
def test_copy_host_matches_oracle(case):
    dtype, M, N, ld_s, ld_d, slab, pinned = case
    src, dst, want = host_case(dtype, M, N, ld_s, ld_d, seed=M + N, pinned=pinned)
    mbt.tile_copy_host(src[:, :N], dst[:, :N], 128, 64 if dtype != "f32" else 32, 3,
                       slab_rows=slab)
    assert torch.equal(bits(dst), bits(want))


ROWSUM_CASES = [
    # dtype, M, N, host ld_src, slab rows, pinned
    ("bf16", 3000, 20000, 20000, 256, True),       # 12 slabs, 3 slots reused
    ("f32", 1234, 8191, 8193, 300, True),          # odd pitch, ragged last slab
    ("f16", 4097, 777, 781, 0, False),             # pageable, one slab
    ("bf16", 70, 65536, 65536, 1, True),           # one row per slab
]


@pytest.mark.parametrize("case", ROWSUM_CASES, ids=lambda c: "-".join(map(str, c)))
def test_rowsum_host_matches_oracle(case):
    dtype, M, N, ld_s, slab, pinned = case
    x = synthetic.make_matrix(M, N, dtype, "normal", seed=M ^ N, ld=ld_s)
    if pinned:
        x = x.pin_memory()
    tn = 128 if dtype == "f32" else 256
    out = mbt.tile_rowsum_host(x[:, :N], None, 64, tn, 2, slab_rows=slab)
    assert out.device.type == "cpu"
    worst, rel, _ = rowsum_errors(out, x[:, :N])
    assert worst <= ROWSUM_RTOL, (worst, rel)


COLSUM_CASES = [
    # dtype, M, N, host ld_src, slab rows (0 = default), pinned
    ("bf16", 3000, 20000, 20000, 256, True),       # 12 slabs added in order
    ("f32", 1234, 8191, 8193, 300, True),          # odd pitch (repacked), ragged last slab
    ("f16", 4097, 777, 781, 0, False),             # pageable, one slab
    ("f16", 70, 4000, 4000, 1, True),              # one row per slab
]


@pytest.mark.parametrize("case", COLSUM_CASES, ids=lambda c: "-".join(map(str, c)))
def test_colsum_host_matches_oracle(case):
    dtype, M, N, ld_s, slab, pinned = case
    x = synthetic.make_matrix(M, N, dtype, "normal", seed=M + N, ld=ld_s)
    if pinned:
        x = x.pin_memory()
    tn = 128 if dtype == "f32" else 256
    out = mbt.tile_colsum_host(x[:, :N], None, 64, tn, 2, slab_rows=slab)
    assert out.device.type == "cpu" and out.numel() == N
    worst, rel, _ = colsum_errors(out, x[:, :N])
    assert worst <= ROWSUM_RTOL, (worst, rel)


def test_default_slabs_of_a_quarter_gigabyte_matrix():
    """bf16 8192 x 16384 (256 MiB): four default slabs of 64 MiB each way."""
    M, N = 8192, 16384
    x = synthetic.make_matrix(M, N, "bf16", "normal", seed=77).pin_memory()
    y = torch.empty_like(x).pin_memory()
    mbt.tile_copy_host(x, y, 128, 64, 3)
    assert torch.equal(bits(y), bits(x))
    out = mbt.tile_rowsum_host(x, None, 64, 256, 2)
    assert rowsum_errors(out, x)[0] <= ROWSUM_RTOL
    cols = mbt.tile_colsum_host(x, None, 64, 256, 2)
    assert colsum_errors(cols, x)[0] <= ROWSUM_RTOL


def test_empty_shapes():
    out = mbt.tile_rowsum_host(torch.empty(5, 0, dtype=torch.float16), None)
    assert out.tolist() == [0.0] * 5
    mbt.tile_copy_host(torch.empty(0, 9, dtype=torch.float16),
                       torch.empty(0, 9, dtype=torch.float16))
    assert mbt.tile_colsum_host(torch.empty(0, 6, dtype=torch.bfloat16)).tolist() == [0.0] * 6


def test_stall_reports_timeout_and_pool_recovers():
    x = synthetic.make_matrix(512, 4096, "bf16", "normal", seed=5).pin_memory()
    with pytest.raises(mbt.MbtError) as e:
        mbt.tile_rowsum_host(x, None, 64, 256, 2, slab_rows=128, fault=2,
                             wait_budget_ns=20_000_000, max_ctas=4)
    assert e.value.code == mbt.MBT_ERR_TIMEOUT
    assert mbt.tile_status()[0] == 0      # recorded in the call's own buffer only
    out = mbt.tile_rowsum_host(x, None, 64, 256, 2, slab_rows=128)
    assert rowsum_errors(out, x)[0] <= ROWSUM_RTOL
    mbt.tile_host_release()
    out = mbt.tile_rowsum_host(x, None, 64, 256, 2)
    assert rowsum_errors(out, x)[0] <= ROWSUM_RTOL


def test_concurrent_host_threads_use_separate_staging():
    xs = [synthetic.make_matrix(2000, 6000, "f16", "uniform", seed=s).pin_memory()
          for s in range(4)]
    ys = [torch.empty_like(x).pin_memory() for x in xs]
    sums = [None] * 4
    errors = []

    def work(i):
        try:
            torch.cuda.set_device(0)
            for _ in range(3):
                if i % 2:
                    mbt.tile_copy_host(xs[i], ys[i], 128, 64, 3, slab_rows=300)
                else:
                    sums[i] = mbt.tile_rowsum_host(xs[i], None, 128, 64, 3, slab_rows=300)
        except Exception as exc:  # noqa: BLE001 -- reported below
            errors.append(exc)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(4):
        if i % 2:
            assert torch.equal(bits(ys[i]), bits(xs[i]))
        else:
            assert rowsum_errors(sums[i], xs[i])[0] <= ROWSUM_RTOL
