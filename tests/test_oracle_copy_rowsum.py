"""Pins for the oracle's copy and row-sum results.

Copy: the result is defined as the identity on the logical region
("cute(11) Hopper TMA copy", §4: the written-back tile must equal the input);
checked by brute force against ``torch.equal`` on the raw bits, with pitched
buffers whose pad columns must not change.

Row sums: exact special cases (all ones, +x/-x pairs, powers of two), the
exactly rounded ``math.fsum`` of values converted by PyTorch (a library path
independent of the oracle's decoder) within the binary64 bound
N * 2^-53 * sum|x|, and IEEE special values.
"""
import math

import pytest
import torch

import oracle
import synthetic
from synthetic import DTYPES, fill_bits, make_matrix, pitched_ld

INT_VIEW = {2: torch.int16, 4: torch.int32}


def _bits(t):
    return t.contiguous().view(INT_VIEW[t.element_size()])


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("M,N", [(1, 1), (3, 5), (17, 33), (64, 129), (130, 7)])
def test_copy_is_identity_on_logical_region(dtype, M, N):
    ld_s = pitched_ld(N, dtype) + 8
    ld_d = pitched_ld(N, dtype) + 16
    src = make_matrix(M, N, dtype, "uniform", seed=M * 1000 + N, ld=ld_s)
    dst_buf = torch.empty(M, ld_d, dtype=DTYPES[dtype])
    fill_bits(dst_buf, synthetic.POISON_BITS[dtype])
    before = dst_buf.clone()
    oracle.copy(src[:, :N], dst_buf[:, :N])
    assert torch.equal(_bits(dst_buf[:, :N]), _bits(src[:, :N]))
    assert torch.equal(_bits(dst_buf[:, N:]), _bits(before[:, N:]))


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_copy_preserves_special_bit_patterns(dtype):
    pats = synthetic.special_values(dtype)
    es = synthetic.ESIZE[dtype]
    src = torch.tensor([p - (1 << 8 * es) if p >= 1 << (8 * es - 1) else p for p in pats],
                       dtype=INT_VIEW[es]).view(DTYPES[dtype]).reshape(1, -1)
    dst = torch.zeros_like(src)
    oracle.copy(src, dst)
    assert torch.equal(_bits(dst), _bits(src))


def test_copy_transposed_operands_detected():
    """A copy that swapped (row, column) would fail the identity check."""
    src = make_matrix(4, 6, "f16", "uniform", seed=3)
    dst = torch.empty_like(src)
    oracle.copy(src, dst)
    assert not torch.equal(dst[:4, :4], src[:4, :4].t().contiguous())
    assert torch.equal(dst, src)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_rowsum_all_ones_is_exact(dtype):
    for N in (1, 7, 64, 1000, 4097):
        x = torch.ones(3, N, dtype=DTYPES[dtype])
        s = oracle.rowsum(x)
        assert s.tolist() == [float(N)] * 3


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_rowsum_cancelling_pairs_is_zero(dtype):
    x = make_matrix(5, 64, dtype, "uniform", seed=11)
    pairs = torch.cat([x, -x], dim=1)
    s = oracle.rowsum(pairs)
    assert s.tolist() == [0.0] * 5


def test_rowsum_powers_of_two_exact():
    # row i holds 2^-k for k = 0..N-1: sum = 2 - 2^-(N-1), exactly representable
    N = 20
    row = torch.tensor([2.0 ** -k for k in range(N)], dtype=torch.float32).reshape(1, -1)
    assert oracle.rowsum(row).item() == 2.0 - 2.0 ** -(N - 1)
    assert oracle.rowsum(row.to(torch.bfloat16)).item() == 2.0 - 2.0 ** -(N - 1)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("dist", ["uniform", "normal"])
def test_rowsum_matches_fsum_within_binary64_bound(dtype, dist):
    M, N = 9, 257
    ld = pitched_ld(N, dtype) + 8
    x = make_matrix(M, N, dtype, dist, seed=5, ld=ld)
    sums, sumsq = oracle.rowsum(x[:, :N], with_sumsq=True)
    vals = x[:, :N].to(torch.float64).tolist()
    for i in range(M):
        exact = math.fsum(vals[i])
        bound = N * 2.0 ** -53 * math.fsum(abs(v) for v in vals[i])
        assert abs(sums[i].item() - exact) <= bound
        assert abs(sumsq[i].item() - math.fsum(v * v for v in vals[i])) <= \
            2 * N * 2.0 ** -53 * math.fsum(v * v for v in vals[i])


def test_rowsum_reads_only_logical_columns():
    """Pad columns hold NaN patterns: a sum that strayed into them is NaN."""
    x = make_matrix(4, 13, "f32", "uniform", seed=2, ld=24)
    s = oracle.rowsum(x[:, :13])
    assert all(math.isfinite(v) for v in s.tolist())
    # dropping the last column would change every row sum
    s_short = oracle.rowsum(x[:, :12])
    assert all(a != b for a, b in zip(s.tolist(), s_short.tolist()))


def test_rowsum_special_values():
    x = torch.tensor([[1.0, math.inf, 2.0], [1.0, math.nan, 0.0],
                      [math.inf, -math.inf, 0.0], [-0.0, -0.0, -0.0]],
                     dtype=torch.float32)
    s = oracle.rowsum(x).tolist()
    assert s[0] == math.inf
    assert math.isnan(s[1])
    assert math.isnan(s[2])
    assert s[3] == 0.0


def test_rowsum_empty_rows_are_zero():
    x = torch.empty(3, 0, dtype=torch.float16)
    assert oracle.rowsum(x).tolist() == [0.0, 0.0, 0.0]
