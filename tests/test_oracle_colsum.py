"""Pins for the oracle's column sums, out[j] = sum over rows i of x[i][j].

Like the row sum, the column sum is the plain definition of a reduction of
the pipeline's tiles (the pages' consumer only "uses" each tile).  Pinned by
exact special cases (all ones give exactly M, +x / -x row pairs cancel,
powers of two), by the exactly rounded ``math.fsum`` of the values as PyTorch
converts them (a library path independent of the oracle's decoder) within
the binary64 bound M * 2^-53 * sum|x|, by pad columns that must not be read,
and by orientation checks that a swapped row / column loop would fail.
"""
import math

import pytest
import torch

import oracle
from synthetic import DTYPES, make_matrix, pitched_ld


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_colsum_all_ones_is_exact(dtype):
    for M in (1, 7, 64, 1000, 4097):
        x = torch.ones(M, 3, dtype=DTYPES[dtype])
        assert oracle.colsum(x).tolist() == [float(M)] * 3


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_colsum_cancelling_rows_is_zero(dtype):
    x = make_matrix(64, 5, dtype, "uniform", seed=11)
    pairs = torch.cat([x, -x], dim=0)
    assert oracle.colsum(pairs).tolist() == [0.0] * 5


def test_colsum_powers_of_two_exact():
    # column 0 holds 2^-k for k = 0..M-1: sum = 2 - 2^-(M-1), exactly representable
    M = 20
    col = torch.tensor([[2.0 ** -k, 1.0] for k in range(M)], dtype=torch.float32)
    s = oracle.colsum(col).tolist()
    assert s == [2.0 - 2.0 ** -(M - 1), float(M)]
    assert oracle.colsum(col.to(torch.bfloat16)).tolist() == s


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("dist", ["uniform", "normal"])
def test_colsum_matches_fsum_within_binary64_bound(dtype, dist):
    M, N = 257, 9
    ld = pitched_ld(N, dtype) + 8
    x = make_matrix(M, N, dtype, dist, seed=6, ld=ld)
    sums, sumsq = oracle.colsum(x[:, :N], with_sumsq=True)
    cols = x[:, :N].to(torch.float64).t().tolist()
    for j in range(N):
        exact = math.fsum(cols[j])
        bound = M * 2.0 ** -53 * math.fsum(abs(v) for v in cols[j])
        assert abs(sums[j].item() - exact) <= bound
        sq = math.fsum(v * v for v in cols[j])
        assert abs(sumsq[j].item() - sq) <= 2 * M * 2.0 ** -53 * sq


def test_colsum_orientation():
    """Column j sums column j: a distinct constant per column and per row
    gives sums a swapped loop (or a transposed operand) cannot produce."""
    M, N = 5, 3
    x = torch.tensor([[float(10 ** j) * (i + 1) for j in range(N)] for i in range(M)],
                     dtype=torch.float32)
    assert oracle.colsum(x).tolist() == [15.0 * 10 ** j for j in range(N)]
    # and the row sums of the same matrix differ from its column sums
    assert oracle.rowsum(x).tolist() == [111.0 * (i + 1) for i in range(M)]


def test_colsum_reads_only_logical_columns_and_rows():
    """Pad columns hold NaN patterns: a sum that strayed into them is NaN."""
    x = make_matrix(13, 4, "f32", "uniform", seed=2, ld=24)
    s = oracle.colsum(x[:, :4])
    assert all(math.isfinite(v) for v in s.tolist())
    s_short = oracle.colsum(x[:12, :4])      # dropping the last row changes every sum
    assert all(a != b for a, b in zip(s.tolist(), s_short.tolist()))


def test_colsum_special_values_and_empty():
    x = torch.tensor([[1.0, 1.0, math.inf, -0.0], [math.inf, math.nan, -math.inf, -0.0],
                      [2.0, 0.0, 0.0, -0.0]], dtype=torch.float32)
    s = oracle.colsum(x).tolist()
    assert s[0] == math.inf
    assert math.isnan(s[1]) and math.isnan(s[2])
    assert s[3] == 0.0
    assert oracle.colsum(torch.empty(0, 4, dtype=torch.float16)).tolist() == [0.0] * 4
    assert oracle.colsum(torch.empty(4, 0, dtype=torch.float16)).tolist() == []


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_colsum_equals_rowsum_of_the_transpose_bitwise(dtype):
    """Column j of x is row j of x^T, and both functions add in index order,
    so the two binary64 results must agree bit for bit."""
    M, N = 301, 77
    x = make_matrix(M, N, dtype, "normal", seed=9, ld=pitched_ld(N, dtype) + 8)[:, :N]
    s, q = oracle.colsum(x, with_sumsq=True)
    r, rq = oracle.rowsum(x.t().contiguous(), with_sumsq=True)
    assert torch.equal(s, r) and torch.equal(q, rq)
