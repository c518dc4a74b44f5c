"""The device calls capture into a CUDA graph: planning is host-only and the
launches take no synchronising call, so a graph of tile_copy, tile_rowsum
and tile_colsum replays correctly on new data written into the captured
input buffers (the workspaces the kernels leave zero-filled are reused by
every replay).  Checked against the oracle on every replay."""
import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import ROWSUM_RTOL, bits, colsum_errors, rowsum_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    mbt._build.build()
    oracle.build()
    torch.cuda.set_device(0)


def test_graph_of_copy_rowsum_colsum_replays_on_new_data():
    M, N = 1500, 5000                                   # ragged against 64 x 256 tiles
    ld = synthetic.pitched_ld(N, "bf16")
    x = torch.empty(M, ld, dtype=torch.bfloat16, device="cuda")[:, :N]
    y = torch.empty_like(x)
    rows = torch.empty(M, dtype=torch.float32, device="cuda")
    cols = torch.empty(N, dtype=torch.float32, device="cuda")
    ws_r = torch.zeros(mbt.tile_rowsum_workspace_bytes(M, N, 64, 256, 2, torch.bfloat16,
                                                       ld_src=ld) or 256,
                       dtype=torch.uint8, device="cuda")
    ws_c = torch.zeros(mbt.tile_colsum_workspace_bytes(M, N, 64, 256, 2, torch.bfloat16,
                                                       ld_src=ld) or 256,
                       dtype=torch.uint8, device="cuda")
    x.copy_(synthetic.make_matrix(M, N, "bf16", "normal", seed=1).cuda())
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())

    def calls():
        mbt.tile_copy(x, y, 64, 256, 3, stream=stream)
        mbt.tile_rowsum(x, rows, 64, 256, 2, workspace=ws_r, stream=stream)
        mbt.tile_colsum(x, cols, 64, 256, 2, workspace=ws_c, stream=stream)

    with torch.cuda.stream(stream):
        calls()                                         # warm the plan caches
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        calls()
    for seed in (2, 3, 4):
        xh = synthetic.make_matrix(M, N, "bf16", "uniform" if seed % 2 else "normal", seed)
        x.copy_(xh.cuda())
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert mbt.tile_status()[0] == 0
        assert torch.equal(bits(y.cpu()), bits(xh))
        assert rowsum_errors(rows, xh)[0] <= ROWSUM_RTOL
        assert colsum_errors(cols, xh)[0] <= ROWSUM_RTOL
        assert int(ws_r.count_nonzero()) == 0 and int(ws_c.count_nonzero()) == 0
