"""Shared helpers of the GPU parity tests."""
import torch

import oracle
import synthetic
from synthetic import DTYPES, ESIZE

INT_VIEW = {2: torch.int16, 4: torch.int32}

# Row-sum tolerance: the fp32 result may differ from the binary64 oracle by at
# most 1e-5 times max(|sum|, sqrt(sum of squares)) -- a relative bound that
# stays meaningful for rows whose sum is close to zero.
ROWSUM_RTOL = 1e-5


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(INT_VIEW[t.element_size()])


def copy_case(dtype, M, N, seed, src_pad=0, dst_pad=0, dist="uniform"):
    """Pitched host source, poisoned host destination, and the oracle's
    expected destination (pads left as poison)."""
    ld_s = synthetic.pitched_ld(N, dtype) + src_pad
    ld_d = synthetic.pitched_ld(N, dtype) + dst_pad
    src = synthetic.make_matrix(M, N, dtype, dist, seed, ld=ld_s)
    dst = torch.empty(M, ld_d, dtype=DTYPES[dtype])
    synthetic.fill_bits(dst, synthetic.POISON_BITS[dtype])
    want = dst.clone()
    oracle.copy(src[:, :N], want[:, :N])
    return src, dst, want


def rowsum_errors(got: torch.Tensor, x_cpu: torch.Tensor):
    """(worst |got - ref| / scale, worst relative error on rows with
    |ref| >= sqrt(sum of squares), ref) for a logical CPU matrix x_cpu."""
    ref, sq = oracle.rowsum(x_cpu, with_sumsq=True)
    g = got.detach().cpu().double()
    scale = torch.maximum(ref.abs(), sq.sqrt()).clamp_min(1e-300)
    err = (g - ref).abs()
    worst = (err / scale).max().item() if len(ref) else 0.0
    big = ref.abs() >= sq.sqrt()
    rel = (err[big] / ref.abs()[big]).max().item() if bool(big.any()) else 0.0
    return worst, rel, ref


def colsum_errors(got: torch.Tensor, x_cpu: torch.Tensor):
    """(worst |got - ref| / scale, worst relative error on columns with
    |ref| >= sqrt(sum of squares), ref) for a logical CPU matrix x_cpu; the
    column-sum counterpart of rowsum_errors, same tolerance."""
    ref, sq = oracle.colsum(x_cpu, with_sumsq=True)
    g = got.detach().cpu().double()
    scale = torch.maximum(ref.abs(), sq.sqrt()).clamp_min(1e-300)
    err = (g - ref).abs()
    worst = (err / scale).max().item() if len(ref) else 0.0
    big = ref.abs() >= sq.sqrt()
    rel = (err[big] / ref.abs()[big]).max().item() if bool(big.any()) else 0.0
    return worst, rel, ref
