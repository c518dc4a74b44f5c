"""The library through its C ABI alone: a plain C program (no Python, no
PyTorch) includes mbtile.h, links libmbtile.so and the CUDA runtime, and runs
tile_copy, tile_rowsum_ex and tile_colsum_ex on a pitched bf16 matrix read
from a file, then the plain tile_rowsum and tile_colsum (no options: the
library's own workspace) twice each on a dense matrix, and the _ex forms with
a workspace of the program's on the same matrix; its outputs are checked here
against the oracle, and the plain calls' sums against the _ex forms' bits."""
import os
import subprocess

import pytest
import torch

import mbarrier_async_tile_gb300 as mbt
import oracle
import synthetic
from helpers import ROWSUM_RTOL, bits, colsum_errors, rowsum_errors

pytestmark = pytest.mark.gpu

C_SOURCE = r"""
#include <stdio.h>
#include <stdlib.h>
#include <stdint.h>
#include <cuda_runtime.h>
#include "mbtile.h"

#define CHECK(x) do { int rc_ = (x); if (rc_ != 0) { \
    fprintf(stderr, "%s: %d (%s)\n", #x, rc_, rc_ < 0 ? tile_strerror(rc_) : "cuda"); \
    return 1; } } while (0)

int main(int argc, char **argv) {
    const int64_t M = atoll(argv[1]), N = atoll(argv[2]), ld = atoll(argv[3]);
    const size_t bytes = (size_t)M * ld * 2;
    uint16_t *h = (uint16_t *)malloc(bytes);
    FILE *f = fopen(argv[4], "rb");
    if (!f || fread(h, 1, bytes, f) != bytes) return 2;
    fclose(f);
    void *src, *dst, *ws;
    float *rows, *cols;
    CHECK(cudaMalloc(&src, bytes));
    CHECK(cudaMalloc(&dst, bytes));
    CHECK(cudaMalloc((void **)&rows, M * 4));
    CHECK(cudaMalloc((void **)&cols, N * 4));
    CHECK(cudaMemcpy(src, h, bytes, cudaMemcpyHostToDevice));
    CHECK(cudaMemset(dst, 0, bytes));

    mbt_opts o = {0};
    o.ld_src = ld;
    o.ld_dst = ld;
    CHECK(tile_copy_ex(src, dst, M, N, 64, 256, 3, MBT_BF16, NULL, &o));

    mbt_opts r = {0};
    r.ld_src = ld;
    size_t need_r = 0, need_c = 0;
    CHECK(tile_rowsum_workspace_bytes(M, N, 64, 256, 2, MBT_BF16, &r, &need_r));
    CHECK(tile_colsum_workspace_bytes(M, N, 64, 256, 2, MBT_BF16, &r, &need_c));
    size_t need = need_r > need_c ? need_r : need_c;
    CHECK(cudaMalloc(&ws, need ? need : 256));
    CHECK(cudaMemset(ws, 0, need ? need : 256));
    r.workspace = need ? ws : NULL;
    r.workspace_bytes = need;
    CHECK(tile_rowsum_ex(src, rows, M, N, 64, 256, 2, MBT_BF16, NULL, &r));
    CHECK(tile_colsum_ex(src, cols, M, N, 64, 256, 2, MBT_BF16, NULL, &r));
    int32_t info[4];
    CHECK(tile_status(NULL, info));

    /* dense matrix: the plain signatures, then the _ex forms with a
       workspace of our own on the same plan */
    const int64_t M2 = atoll(argv[6]), N2 = atoll(argv[7]);
    const size_t bytes2 = (size_t)M2 * N2 * 2;
    uint16_t *h2 = (uint16_t *)malloc(bytes2);
    f = fopen(argv[8], "rb");
    if (!f || fread(h2, 1, bytes2, f) != bytes2) return 2;
    fclose(f);
    void *src2, *ws2;
    float *sums2;   /* rows x 3, then cols x 3 */
    const size_t nsum = (size_t)(3 * M2 + 3 * N2);
    CHECK(cudaMalloc(&src2, bytes2));
    CHECK(cudaMalloc((void **)&sums2, nsum * 4));
    CHECK(cudaMemcpy(src2, h2, bytes2, cudaMemcpyHostToDevice));
    CHECK(tile_rowsum(src2, sums2, M2, N2, 64, 256, 2, MBT_BF16, NULL));
    CHECK(tile_rowsum(src2, sums2 + M2, M2, N2, 64, 256, 2, MBT_BF16, NULL));
    CHECK(tile_colsum(src2, sums2 + 3 * M2, M2, N2, 64, 256, 2, MBT_BF16, NULL));
    CHECK(tile_colsum(src2, sums2 + 3 * M2 + N2, M2, N2, 64, 256, 2, MBT_BF16, NULL));
    mbt_opts d = {0};
    CHECK(tile_rowsum_workspace_bytes(M2, N2, 64, 256, 2, MBT_BF16, &d, &need_r));
    CHECK(tile_colsum_workspace_bytes(M2, N2, 64, 256, 2, MBT_BF16, &d, &need_c));
    if (need_r == 0 || need_c == 0) return 3;   /* the shape must split */
    need = need_r > need_c ? need_r : need_c;
    CHECK(cudaMalloc(&ws2, need));
    CHECK(cudaMemset(ws2, 0, need));
    d.workspace = ws2;
    d.workspace_bytes = need;
    CHECK(tile_rowsum_ex(src2, sums2 + 2 * M2, M2, N2, 64, 256, 2, MBT_BF16, NULL, &d));
    CHECK(tile_colsum_ex(src2, sums2 + 3 * M2 + 2 * N2, M2, N2, 64, 256, 2, MBT_BF16, NULL,
                         &d));
    CHECK(tile_status(NULL, info));
    CHECK(tile_workspace_release(NULL));
    float *hs2 = (float *)malloc(nsum * 4);
    CHECK(cudaMemcpy(hs2, sums2, nsum * 4, cudaMemcpyDeviceToHost));

    uint16_t *hd = (uint16_t *)malloc(bytes);
    float *hr = (float *)malloc(M * 4), *hc = (float *)malloc(N * 4);
    CHECK(cudaMemcpy(hd, dst, bytes, cudaMemcpyDeviceToHost));
    CHECK(cudaMemcpy(hr, rows, M * 4, cudaMemcpyDeviceToHost));
    CHECK(cudaMemcpy(hc, cols, N * 4, cudaMemcpyDeviceToHost));
    f = fopen(argv[5], "wb");
    fwrite(hd, 1, bytes, f);
    fwrite(hr, 4, M, f);
    fwrite(hc, 4, N, f);
    fwrite(hs2, 4, nsum, f);
    fclose(f);
    printf("ok\n");
    return 0;
}
"""


def test_c_program_copy_rowsum_colsum(tmp_path):
    lib = mbt._build.build()
    oracle.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    src_c = tmp_path / "prog.c"
    src_c.write_text(C_SOURCE)
    exe = tmp_path / "prog"
    libdir = os.path.dirname(lib)
    subprocess.run(["gcc", "-O1", "-std=c11", str(src_c), "-o", str(exe),
                    "-I", os.path.join(mbt._build.ROOT, "include"), "-I", f"{cuda}/include",
                    "-L", libdir, "-lmbtile", "-L", f"{cuda}/lib64", "-lcudart",
                    f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cuda}/lib64"], check=True)
    M, N = 777, 3001
    ld = synthetic.pitched_ld(N, "bf16")
    x = synthetic.make_matrix(M, N, "bf16", "normal", seed=31, ld=ld)
    M2, N2 = 1000, 20480                       # 16 bands x 80 strips: both split
    x2 = synthetic.make_matrix(M2, N2, "bf16", "normal", seed=32)
    inp, outp, inp2 = tmp_path / "in.bin", tmp_path / "out.bin", tmp_path / "in2.bin"
    inp.write_bytes(x.contiguous().view(torch.int16).numpy().tobytes())
    inp2.write_bytes(x2.contiguous().view(torch.int16).numpy().tobytes())
    res = subprocess.run([str(exe), str(M), str(N), str(ld), str(inp), str(outp), str(M2),
                          str(N2), str(inp2)], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stderr
    raw = outp.read_bytes()
    nb = M * ld * 2
    y = torch.frombuffer(bytearray(raw[:nb]), dtype=torch.int16).view(M, ld)
    rows = torch.frombuffer(bytearray(raw[nb:nb + 4 * M]), dtype=torch.float32)
    cols = torch.frombuffer(bytearray(raw[nb + 4 * M:nb + 4 * M + 4 * N]), dtype=torch.float32)
    sums2 = torch.frombuffer(bytearray(raw[nb + 4 * M + 4 * N:]), dtype=torch.float32)
    rows2 = sums2[:3 * M2].view(3, M2)
    cols2 = sums2[3 * M2:].view(3, N2)
    for k in range(3):
        assert rowsum_errors(rows2[k], x2)[0] <= ROWSUM_RTOL, k
        assert colsum_errors(cols2[k], x2)[0] <= ROWSUM_RTOL, k
    # the plain calls run the _ex forms' plan: identical bits, call after call
    for k in range(2):
        assert torch.equal(rows2[k].view(torch.int32), rows2[2].view(torch.int32)), k
        assert torch.equal(cols2[k].view(torch.int32), cols2[2].view(torch.int32)), k
    assert torch.equal(y[:, :N], bits(x[:, :N]))
    assert int(y[:, N:].abs().sum()) == 0            # pad columns of dst untouched
    assert rowsum_errors(rows, x[:, :N])[0] <= ROWSUM_RTOL
    assert colsum_errors(cols, x[:, :N])[0] <= ROWSUM_RTOL
