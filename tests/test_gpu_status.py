"""Per-call status buffers (mbt_opts.status): a pipeline that stalls by
construction on one stream records its timed-out wait in its own buffer,
while a clean call of the same kind on a second stream, running at the same
time, finishes with its buffer and the per-device status word untouched.
Covers every kernel family: LSU and bulk-store copies, the stage-wide and
per-box row sums, the column sum, the wide (one CTA per SM) row and column
sums, the fused copy + row sum, and the 1-D
bulk-copy (unaligned pitch) copy and row sums.  The host-buffer forms use a
buffer per staging set, so a stalled host call and clean host calls in other
threads do not see one another's timeouts."""
import threading

import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import ROWSUM_RTOL, bits, colsum_errors, rowsum_errors

pytestmark = pytest.mark.gpu

BUDGET_NS = 20_000_000   # 20 ms per wait


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


def _copy(**kw):
    return lambda x, y, **o: mbt.tile_copy(x, y, 128, 64, 3, **kw, **o)


# name: (dtype, M, N, call, result kind)
CASES = {
    "copy_lsu": ("bf16", 512, 4096, _copy(store_mode=2), "copy"),
    "copy_bulk": ("bf16", 512, 4096, _copy(store_mode=1), "copy"),
    "rowsum_stage_pairs": ("bf16", 512, 4096, lambda x, y, **o: mbt.tile_rowsum(
        x, None, 64, 256, 3, split=False, pipeline=2, **o), "rows"),
    "rowsum_box_pairs": ("bf16", 512, 4096, lambda x, y, **o: mbt.tile_rowsum(
        x, None, 64, 256, 3, consumer_warps=8, split=False, pipeline=3, **o), "rows"),
    "colsum": ("bf16", 512, 4096, lambda x, y, **o: mbt.tile_colsum(
        x, None, 64, 256, 3, split=False, **o), "cols"),
    "rowsum_wide": ("bf16", 512, 4096, lambda x, y, **o: mbt.tile_rowsum(
        x, None, 64, 256, 4, consumer_warps=16, split=False, **o), "rows"),
    "colsum_wide": ("bf16", 512, 4096, lambda x, y, **o: mbt.tile_colsum(
        x, None, 64, 256, 4, consumer_warps=16, split=False, **o), "cols"),
    "fused": ("bf16", 512, 4096, lambda x, y, **o: mbt.tile_copy_rowsum(
        x, y, None, 128, 64, 3, split=False, **o), "rows+copy"),
    "flat_copy": ("f16", 512, 1001, _copy(), "copy"),
    "flat_rowsum_rows": ("f16", 512, 1001, lambda x, y, **o: mbt.tile_rowsum(
        x, None, 128, 64, 3, split=False, **o), "rows"),
    "flat_rowsum_pieces": ("f16", 64, 20001, lambda x, y, **o: mbt.tile_rowsum(
        x, None, 128, 64, 3, split=False, **o), "rows"),
}


@pytest.mark.parametrize("case", list(CASES))
def test_stall_is_recorded_in_its_own_buffer(case):
    dtype, M, N, call, kind = CASES[case]
    x = synthetic.make_matrix(M, N, dtype, "normal", seed=41)
    assert mbt.tile_status()[0] == 0
    xa, xb = x.cuda(), x.cuda()
    ya, yb = torch.empty_like(xa), torch.empty_like(xb)
    st_a = torch.zeros(4, dtype=torch.int32, device="cuda")
    st_b = torch.zeros(4, dtype=torch.int32, device="cuda")
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(sa):
        call(xa, ya, fault=2, max_ctas=4, wait_budget_ns=BUDGET_NS, status=st_a, stream=sa)
    with torch.cuda.stream(sb):
        got = call(xb, yb, status=st_b, stream=sb)
    torch.cuda.synchronize()
    a, b = st_a.tolist(), st_b.tolist()
    assert a[0] == mbt.MBT_ERR_TIMEOUT and 0 <= a[1] < 4, a
    assert b == [0, 0, 0, 0], b
    assert mbt.tile_status()[0] == 0      # the per-device word saw neither call
    if "copy" in kind:
        assert torch.equal(bits(yb.cpu()), bits(x))
    if "rows" in kind:
        assert rowsum_errors(got, x)[0] <= ROWSUM_RTOL
    if kind == "cols":
        assert colsum_errors(got, x)[0] <= ROWSUM_RTOL


def test_without_a_buffer_the_device_word_takes_it():
    x = synthetic.make_matrix(512, 4096, "bf16", "normal", seed=42).cuda()
    mbt.tile_copy(x, torch.empty_like(x), 128, 64, 3, max_ctas=4, fault=2,
                  wait_budget_ns=BUDGET_NS)
    code, info = mbt.tile_status()
    assert code == mbt.MBT_ERR_TIMEOUT and 0 <= info[1] < 4, info


def test_status_buffer_argument_checks():
    x = synthetic.make_matrix(64, 256, "bf16", "normal", seed=43).cuda()
    y = torch.empty_like(x)
    for bad in (torch.zeros(4, dtype=torch.int64, device="cuda"),
                torch.zeros(3, dtype=torch.int32, device="cuda"),
                torch.zeros(4, dtype=torch.int32)):
        with pytest.raises(ValueError):
            mbt.tile_copy(x, y, 64, 128, 2, status=bad)
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    mbt.tile_copy(x, y, 64, 128, 2, status=st)
    torch.cuda.synchronize()
    assert st.tolist() == [0, 0, 0, 0] and torch.equal(bits(y.cpu()), bits(x.cpu()))


def test_host_calls_in_other_threads_do_not_see_a_stall():
    x = synthetic.make_matrix(512, 4096, "bf16", "normal", seed=44).pin_memory()
    clean = [synthetic.make_matrix(3000, 5000, "f16", "uniform", seed=s).pin_memory()
             for s in range(2)]
    results, errors = {}, []

    def stalled():
        try:
            torch.cuda.set_device(0)
            mbt.tile_rowsum_host(x, None, 64, 256, 2, slab_rows=128, fault=2,
                                 wait_budget_ns=BUDGET_NS, max_ctas=4)
            errors.append("stalled call returned")
        except mbt.MbtError as e:
            results["stalled"] = e.code
        except Exception as e:                 # noqa: BLE001 - reported below
            errors.append(repr(e))

    def worker(i):
        try:
            torch.cuda.set_device(0)
            for _ in range(4):
                results[i] = mbt.tile_rowsum_host(clean[i], None, 128, 64, 3, slab_rows=400)
        except Exception as e:                 # noqa: BLE001 - reported below
            errors.append(repr(e))

    ts = [threading.Thread(target=stalled)] + [threading.Thread(target=worker, args=(i,))
                                               for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in ts)
    assert errors == []
    assert results["stalled"] == mbt.MBT_ERR_TIMEOUT
    for i in range(2):
        assert rowsum_errors(results[i], clean[i])[0] <= ROWSUM_RTOL
    assert mbt.tile_status()[0] == 0
