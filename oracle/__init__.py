"""CPU oracle of the mbarrier/TMA tile pipeline -- TEST INFRASTRUCTURE.

Only ``tests/``, the smoke check in ``__graft_entry__`` and the CPU-baseline leg
of ``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and this package never
imports the product: the two share nothing but the seeded input generator.

Contents, each pinned by ``tests/test_oracle_*.py`` against what the pages fix:

* ``copy``            -- the tile copy's result (plain C, ``oracle_ref.c``).
* ``rowsum``          -- binary64 row sums (plain C, ``oracle_ref.c``).
* ``colsum``          -- binary64 column sums (plain C, ``oracle_ref.c``).
* ``xor_fold``        -- XOR of a buffer's 32-bit words (plain C): the result
                         of the read-bandwidth reference.
* ``f16_to_f64`` ...  -- exact element widening (plain C).
* ``pipeline_state``  -- the (index, phase, count) ring cursor.
* ``mbarrier``        -- the mbarrier phase / arrival / tx-count model.
* ``simulator``       -- one CTA's producer / copy engine / consumers under
                         random interleavings, plus the lessons' lock-step
                         barrier timeline and 2-stage parity walk.
* ``swizzle``         -- the 128-byte shared-memory swizzle on byte offsets.
* ``smem``            -- the lessons' shared-memory and tx-byte formulas.

Parity status: every function above has at least one pin that does not come
from the oracle itself (page tables, closed forms, exact special cases, a
library routine, brute force).  None is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

from . import mbarrier, pipeline_state, simulator, smem, swizzle  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_ref.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_ref.so")

_DTYPE_CODE = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle_ref.c`` with the host C compiler (plain -O2, no
    threads, no vector flags) and return the library path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_f32_to_f64.argtypes = [ctypes.c_uint32]
            lib.oracle_f32_to_f64.restype = ctypes.c_double
            lib.oracle_copy.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
            lib.oracle_copy.restype = None
            lib.oracle_rowsum.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
            lib.oracle_rowsum.restype = None
            lib.oracle_colsum.argtypes = lib.oracle_rowsum.argtypes
            lib.oracle_colsum.restype = None
            lib.oracle_xor_fold.argtypes = [ctypes.c_void_p, ctypes.c_int64]
            lib.oracle_xor_fold.restype = ctypes.c_uint32
            _lib = lib
    return _lib


def f16_to_f64(bits: int) -> float:
    return _load().oracle_f16_to_f64(bits & 0xFFFF)


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(bits & 0xFFFF)


def f32_to_f64(bits: int) -> float:
    return _load().oracle_f32_to_f64(bits & 0xFFFFFFFF)


def _check_2d(t: torch.Tensor, name: str) -> None:
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a CPU tensor")
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D row-major (pitched) view")


def copy(src: torch.Tensor, dst: torch.Tensor) -> torch.Tensor:
    """dst[i, j] = src[i, j] bitwise for the logical shape of ``src``;
    ``dst`` must have the same logical shape; its pad columns (if it is a view
    into a wider buffer) are not touched."""
    _check_2d(src, "src")
    _check_2d(dst, "dst")
    if src.shape != dst.shape or src.dtype != dst.dtype:
        raise ValueError("src and dst must have the same shape and dtype")
    M, N = src.shape
    _load().oracle_copy(src.data_ptr(), dst.data_ptr(), M, N, src.stride(0),
                        dst.stride(0), src.element_size())
    return dst


def rowsum(src: torch.Tensor, with_sumsq: bool = False):
    """Binary64 row sums of the logical matrix ``src`` (a CPU view)."""
    _check_2d(src, "src")
    if src.dtype not in _DTYPE_CODE:
        raise ValueError("unsupported dtype")
    M, N = src.shape
    sums = torch.empty(M, dtype=torch.float64)
    sumsq = torch.empty(M, dtype=torch.float64) if with_sumsq else None
    _load().oracle_rowsum(src.data_ptr(), sums.data_ptr(),
                          sumsq.data_ptr() if with_sumsq else None,
                          M, N, src.stride(0), _DTYPE_CODE[src.dtype])
    return (sums, sumsq) if with_sumsq else sums


def colsum(src: torch.Tensor, with_sumsq: bool = False):
    """Binary64 column sums of the logical matrix ``src`` (a CPU view)."""
    _check_2d(src, "src")
    if src.dtype not in _DTYPE_CODE:
        raise ValueError("unsupported dtype")
    M, N = src.shape
    sums = torch.empty(N, dtype=torch.float64)
    sumsq = torch.empty(N, dtype=torch.float64) if with_sumsq else None
    _load().oracle_colsum(src.data_ptr(), sums.data_ptr(),
                          sumsq.data_ptr() if with_sumsq else None,
                          M, N, src.stride(0), _DTYPE_CODE[src.dtype])
    return (sums, sumsq) if with_sumsq else sums


def xor_fold(buf: torch.Tensor) -> int:
    """XOR of all 32-bit little-endian words of a contiguous CPU tensor's
    bytes (its byte count a multiple of 4)."""
    if buf.device.type != "cpu" or not buf.is_contiguous():
        raise ValueError("buf must be a contiguous CPU tensor")
    nbytes = buf.numel() * buf.element_size()
    if nbytes % 4:
        raise ValueError("byte count must be a multiple of 4")
    return int(_load().oracle_xor_fold(buf.data_ptr() if nbytes else None, nbytes // 4))
