"""Python binding of libmbtile, the sm_103a mbarrier/TMA tile pipeline.

Argument marshalling only: every step of ``tile_copy``, ``tile_rowsum``,
``tile_colsum`` and ``tile_copy_rowsum`` runs in the library's CUDA kernels,
and the host-buffer forms (``tile_*_host``) are the library's own slab
pipeline.  PyTorch supplies device memory and streams.  If the compiled
library is missing, every call raises; there is no fallback path.

The C entry points are reachable with the header's names through ``C`` (a
ctypes handle); the functions below take ``torch.Tensor`` arguments.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

__all__ = [
    "MbtError", "C", "library_path", "Opts", "Plan", "DTYPE_CODE",
    "OP_COPY", "OP_ROWSUM", "OP_COPY_ROWSUM", "OP_COLSUM", "MBT_OK", "MBT_ERR_TIMEOUT",
    "tile_copy", "tile_rowsum", "tile_colsum", "tile_copy_rowsum", "tile_rowsum_noalloc",
    "tile_rowsum_workspace_bytes", "tile_colsum_workspace_bytes",
    "tile_copy_host", "tile_rowsum_host", "tile_colsum_host", "tile_host_release",
    "tile_workspace_release", "tile_read_checksum",
    "tile_status", "tile_plan", "tile_plan_device", "tile_device_info", "tile_strerror",
    "tile_stage_image",
]

MBT_OK = 0
MBT_ERR_TIMEOUT = -6
OP_COPY, OP_ROWSUM, OP_COPY_ROWSUM, OP_COLSUM = 0, 1, 2, 3
DTYPE_CODE = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}


class Opts(ctypes.Structure):
    """Mirror of ``mbt_opts`` in include/mbtile.h."""
    _fields_ = [
        ("ld_src", ctypes.c_int64),
        ("ld_dst", ctypes.c_int64),
        ("max_ctas", ctypes.c_int32),
        ("ctas_per_sm", ctypes.c_int32),
        ("consumer_warps", ctypes.c_int32),
        ("store_mode", ctypes.c_int32),
        ("wait_budget_ns", ctypes.c_uint64),
        ("log", ctypes.c_void_p),
        ("log_capacity", ctypes.c_int64),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("fault", ctypes.c_int32),
        ("pipeline", ctypes.c_int32),
        ("host_slab_rows", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("status", ctypes.c_void_p),
        ("no_split", ctypes.c_int32),
        ("reserved1", ctypes.c_int32),
    ]


class Plan(ctypes.Structure):
    """Mirror of ``mbt_plan`` in include/mbtile.h."""
    _fields_ = [
        ("grid", ctypes.c_int32),
        ("threads", ctypes.c_int32),
        ("consumer_warps", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("boxes", ctypes.c_int32),
        ("box_inner", ctypes.c_int32),
        ("box_rows", ctypes.c_int32),
        ("tx_bytes", ctypes.c_int32),
        ("stage_bytes", ctypes.c_int32),
        ("split", ctypes.c_int32),
        ("kmax", ctypes.c_int32),
        ("flat", ctypes.c_int32),
        ("box_barriers", ctypes.c_int32),
        ("col_group", ctypes.c_int32),
        ("bulk_stores", ctypes.c_int32),
        ("phase_shift", ctypes.c_int32),
        ("tiles_m", ctypes.c_int64),
        ("tiles_n", ctypes.c_int64),
        ("num_tiles", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_size_t),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class MbtError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {tile_strerror(code)} (status {code})" if what
                         else f"{tile_strerror(code)} (status {code})")


_lock = threading.Lock()
_C = None


def library_path() -> str:
    return _build.LIB_PATH


def _load():
    global _C
    with _lock:
        if _C is not None:
            return _C
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"libmbtile.so is not built ({path}); run __graft_entry__.build() "
                "or mbarrier_async_tile_gb300._build.build()")
        lib = ctypes.CDLL(path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        sig = [vp, vp, i64, i64, i32, i32, i32, i32, vp]
        lib.tile_copy.argtypes = sig
        lib.tile_copy_ex.argtypes = sig + [ctypes.POINTER(Opts)]
        lib.tile_rowsum.argtypes = sig
        lib.tile_rowsum_ex.argtypes = sig + [ctypes.POINTER(Opts)]
        lib.tile_copy_rowsum.argtypes = [vp, vp, vp, i64, i64, i32, i32, i32, i32, vp]
        lib.tile_copy_rowsum_ex.argtypes = [vp, vp, vp, i64, i64, i32, i32, i32, i32, vp,
                                            ctypes.POINTER(Opts)]
        lib.tile_rowsum_workspace_bytes.argtypes = [i64, i64, i32, i32, i32, i32,
                                                    ctypes.POINTER(Opts),
                                                    ctypes.POINTER(ctypes.c_size_t)]
        lib.tile_copy_rowsum_workspace_bytes.argtypes = [i64, i64, i32, i32, i32, i32,
                                                         ctypes.POINTER(Opts),
                                                         ctypes.POINTER(ctypes.c_size_t)]
        lib.tile_plan.argtypes = [i32, i64, i64, i32, i32, i32, i32, ctypes.POINTER(Opts),
                                  i32, i32, i32, i32, ctypes.POINTER(Plan)]
        lib.tile_plan_device.argtypes = [i32, i64, i64, i32, i32, i32, i32,
                                         ctypes.POINTER(Opts), ctypes.POINTER(Plan)]
        lib.tile_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        lib.tile_strerror.argtypes = [i32]
        lib.tile_strerror.restype = ctypes.c_char_p
        lib.tile_device_info.argtypes = [i32, ctypes.POINTER(ctypes.c_int),
                                         ctypes.POINTER(ctypes.c_int),
                                         ctypes.POINTER(ctypes.c_double)]
        lib.tile_colsum.argtypes = sig
        lib.tile_colsum_ex.argtypes = sig + [ctypes.POINTER(Opts)]
        lib.tile_colsum_workspace_bytes.argtypes = [i64, i64, i32, i32, i32, i32,
                                                    ctypes.POINTER(Opts),
                                                    ctypes.POINTER(ctypes.c_size_t)]
        host_sig = [vp, vp, i64, i64, i32, i32, i32, i32, ctypes.POINTER(Opts)]
        lib.tile_copy_host.argtypes = host_sig
        lib.tile_rowsum_host.argtypes = host_sig
        lib.tile_colsum_host.argtypes = host_sig
        lib.tile_host_release.argtypes = []
        lib.tile_workspace_release.argtypes = [vp]
        lib.tile_read_checksum.argtypes = [vp, ctypes.c_size_t, vp, vp]
        for name in ("tile_copy", "tile_copy_ex", "tile_rowsum", "tile_rowsum_ex",
                     "tile_copy_rowsum", "tile_copy_rowsum_ex",
                     "tile_rowsum_workspace_bytes", "tile_copy_rowsum_workspace_bytes",
                     "tile_plan", "tile_plan_device", "tile_status", "tile_device_info",
                     "tile_copy_host", "tile_rowsum_host", "tile_colsum_host",
                     "tile_host_release", "tile_workspace_release", "tile_read_checksum",
                     "tile_colsum", "tile_colsum_ex", "tile_colsum_workspace_bytes"):
            getattr(lib, name).restype = ctypes.c_int
        _C = lib
        return lib


class _LazyC:
    """``C.tile_copy(...)`` etc.: the raw C entry points, loaded on first use."""

    def __getattr__(self, name):
        return getattr(_load(), name)


C = _LazyC()


def tile_strerror(code: int) -> str:
    return _load().tile_strerror(code).decode()


def _check(code: int, what: str) -> None:
    if code != MBT_OK:
        raise MbtError(code, what)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _matrix(t: torch.Tensor, name: str) -> tuple[int, int, int]:
    if not isinstance(t, torch.Tensor) or t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in DTYPE_CODE:
        raise ValueError(f"{name} has unsupported dtype {t.dtype}")
    M, N = t.shape
    if M > 0 and N > 0 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major (unit column stride)")
    ld = t.stride(0) if M > 1 else max(N, t.stride(0))
    return M, N, ld


def _host_matrix(t: torch.Tensor, name: str) -> tuple[int, int, int]:
    if not isinstance(t, torch.Tensor) or t.dim() != 2:
        raise ValueError(f"{name} must be a 2-D tensor")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype not in DTYPE_CODE:
        raise ValueError(f"{name} has unsupported dtype {t.dtype}")
    M, N = t.shape
    if M > 0 and N > 0 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major (unit column stride)")
    ld = t.stride(0) if M > 1 else max(N, t.stride(0))
    return M, N, ld


def _opts(**kw) -> Opts:
    o = Opts()
    for k, v in kw.items():
        if v is not None:
            setattr(o, k, v)
    return o


def _set_log_status(o: Opts, log: torch.Tensor | None, status: torch.Tensor | None,
                    device: torch.device) -> None:
    """Point ``o`` at the caller's log records and per-call status buffer."""
    if log is not None:
        o.log = log.data_ptr()
        o.log_capacity = log.numel() // 8
    if status is not None:
        if (status.dtype != torch.int32 or status.device != device or status.numel() < 4
                or not status.is_contiguous()):
            raise ValueError("status must be a contiguous int32 tensor of at least 4 "
                             "elements on the matrix's device")
        o.status = status.data_ptr()


def tile_copy(src: torch.Tensor, dst: torch.Tensor, tile_m: int = 128, tile_n: int = 64,
              stages: int = 4, *, consumer_warps: int = 0, max_ctas: int = 0,
              ctas_per_sm: int = 0, wait_budget_ns: int = 0, log: torch.Tensor | None = None,
              fault: int = 0, store_mode: int = 0, pipeline: int = 0,
              status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dst[i, j] = src[i, j] (bit-exact) through the tile pipeline.

    ``src`` and ``dst`` are 2-D CUDA views of the same shape and dtype with
    unit column stride; their row strides may differ (pitched storage).
    ``store_mode``: 1 bulk tensor stores, 2 16-byte LSU stores, 0 (default)
    bulk where rows end inside a 16-byte chunk, else LSU.  ``status``: an
    optional zero-filled CUDA int32[4] that records this call's timed-out
    wait (as :func:`tile_status` reports it) instead of the per-device word;
    the sums and the fused call take it too."""
    M, N, ld_s = _matrix(src, "src")
    Md, Nd, ld_d = _matrix(dst, "dst")
    if (M, N) != (Md, Nd) or src.dtype != dst.dtype:
        raise ValueError("src and dst must have the same shape and dtype")
    o = _opts(ld_src=ld_s, ld_dst=ld_d, consumer_warps=consumer_warps, max_ctas=max_ctas,
              ctas_per_sm=ctas_per_sm, wait_budget_ns=wait_budget_ns, fault=fault,
              store_mode=store_mode, pipeline=pipeline)
    _set_log_status(o, log, status, src.device)
    rc = _load().tile_copy_ex(src.data_ptr(), dst.data_ptr(), M, N, tile_m, tile_n, stages,
                              DTYPE_CODE[src.dtype], _stream_handle(stream), ctypes.byref(o))
    _check(rc, "tile_copy")
    return dst


def _device_empty(n: int, device: torch.device, stream=None) -> torch.Tensor:
    """fp32[n] for a result, allocated on the stream that will write it (so the
    caching allocator orders any later reuse of the block after that work)."""
    with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream()):
        return torch.empty(n, dtype=torch.float32, device=device)


def _set_split(o: Opts, split: bool, workspace: torch.Tensor | None) -> None:
    """Bands (strips) split over CTAs with the caller's workspace if given, else
    with the library's own for (device, stream); ``split=False``: one CTA each."""
    if not split:
        if workspace is not None:
            raise ValueError("workspace given with split=False")
        o.no_split = 1
    elif workspace is not None:
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()


def tile_rowsum_workspace_bytes(M: int, N: int, tile_m: int, tile_n: int, stages: int,
                                dtype: torch.dtype, fused: bool = False, **opt) -> int:
    """Workspace bytes of tile_rowsum (or, with ``fused``, tile_copy_rowsum)."""
    o = _opts(**opt)
    out = ctypes.c_size_t(0)
    fn = (_load().tile_copy_rowsum_workspace_bytes if fused
          else _load().tile_rowsum_workspace_bytes)
    rc = fn(M, N, tile_m, tile_n, stages, DTYPE_CODE[dtype], ctypes.byref(o), ctypes.byref(out))
    _check(rc, "tile_rowsum_workspace_bytes")
    return out.value


def tile_colsum_workspace_bytes(M: int, N: int, tile_m: int, tile_n: int, stages: int,
                                dtype: torch.dtype, **opt) -> int:
    """Workspace bytes of tile_colsum."""
    o = _opts(**opt)
    out = ctypes.c_size_t(0)
    rc = _load().tile_colsum_workspace_bytes(M, N, tile_m, tile_n, stages, DTYPE_CODE[dtype],
                                             ctypes.byref(o), ctypes.byref(out))
    _check(rc, "tile_colsum_workspace_bytes")
    return out.value


def tile_colsum(src: torch.Tensor, out: torch.Tensor | None = None, tile_m: int = 64,
                tile_n: int = 256, stages: int = 2, *, split: bool = True,
                consumer_warps: int = 0, max_ctas: int = 0, ctas_per_sm: int = 0,
                wait_budget_ns: int = 0, log: torch.Tensor | None = None, fault: int = 0,
                workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """out[j] = sum_i src[i, j] in fp32 through the tile pipeline (tiles taken
    down each column strip).  With ``split`` (default) strips may be shared by
    several CTAs, using ``workspace`` (zero-filled, see
    :func:`tile_colsum_workspace_bytes`) or, if none is given, the library's
    own for (device, stream)."""
    M, N, ld_s = _matrix(src, "src")
    if out is None:
        out = _device_empty(N, src.device, stream)
    if out.dtype != torch.float32 or out.numel() != N or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 tensor of N elements")
    o = _opts(ld_src=ld_s, consumer_warps=consumer_warps, max_ctas=max_ctas,
              ctas_per_sm=ctas_per_sm, wait_budget_ns=wait_budget_ns, fault=fault)
    _set_log_status(o, log, status, src.device)
    _set_split(o, split, workspace)
    rc = _load().tile_colsum_ex(src.data_ptr(), out.data_ptr(), M, N, tile_m, tile_n, stages,
                                DTYPE_CODE[src.dtype], _stream_handle(stream), ctypes.byref(o))
    _check(rc, "tile_colsum")
    return out


def tile_rowsum(src: torch.Tensor, out: torch.Tensor | None = None, tile_m: int = 64,
                tile_n: int = 256, stages: int = 4, *, split: bool = True,
                consumer_warps: int = 0, max_ctas: int = 0, ctas_per_sm: int = 0,
                wait_budget_ns: int = 0, log: torch.Tensor | None = None, fault: int = 0,
                workspace: torch.Tensor | None = None, pipeline: int = 0,
                status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[i] = sum_j src[i, j] in fp32 through the tile pipeline.

    With ``split`` (default) row bands may be shared by several CTAs, using
    ``workspace`` (zero-filled, see :func:`tile_rowsum_workspace_bytes`) or,
    if none is given, the library's own for (device, stream).
    ``pipeline=2`` keeps one barrier pair per stage, ``pipeline=3`` gives
    every box of a stage its own pair where the tile allows it
    (``Plan.box_barriers``), 0 picks 3 for at most 2 stages; the sums are the
    same in all three."""
    M, N, ld_s = _matrix(src, "src")
    if out is None:
        out = _device_empty(M, src.device, stream)
    if out.dtype != torch.float32 or out.numel() != M or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 tensor of M elements")
    o = _opts(ld_src=ld_s, consumer_warps=consumer_warps, max_ctas=max_ctas,
              ctas_per_sm=ctas_per_sm, wait_budget_ns=wait_budget_ns, fault=fault,
              pipeline=pipeline)
    _set_log_status(o, log, status, src.device)
    _set_split(o, split, workspace)
    rc = _load().tile_rowsum_ex(src.data_ptr(), out.data_ptr(), M, N, tile_m, tile_n, stages,
                                DTYPE_CODE[src.dtype], _stream_handle(stream), ctypes.byref(o))
    _check(rc, "tile_rowsum")
    return out


def tile_copy_rowsum(src: torch.Tensor, dst: torch.Tensor, out: torch.Tensor | None = None,
                     tile_m: int = 128, tile_n: int = 64, stages: int = 3, *,
                     split: bool = True, consumer_warps: int = 0, max_ctas: int = 0,
                     ctas_per_sm: int = 0, wait_budget_ns: int = 0,
                     log: torch.Tensor | None = None, fault: int = 0,
                     workspace: torch.Tensor | None = None,
                     status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dst[i, j] = src[i, j] and out[i] = sum_j src[i, j] in one pass; returns out."""
    M, N, ld_s = _matrix(src, "src")
    Md, Nd, ld_d = _matrix(dst, "dst")
    if (M, N) != (Md, Nd) or src.dtype != dst.dtype:
        raise ValueError("src and dst must have the same shape and dtype")
    if out is None:
        out = _device_empty(M, src.device, stream)
    if out.dtype != torch.float32 or out.numel() != M or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 tensor of M elements")
    o = _opts(ld_src=ld_s, ld_dst=ld_d, consumer_warps=consumer_warps, max_ctas=max_ctas,
              ctas_per_sm=ctas_per_sm, wait_budget_ns=wait_budget_ns, fault=fault)
    _set_log_status(o, log, status, src.device)
    _set_split(o, split, workspace)
    rc = _load().tile_copy_rowsum_ex(src.data_ptr(), dst.data_ptr(), out.data_ptr(), M, N,
                                     tile_m, tile_n, stages, DTYPE_CODE[src.dtype],
                                     _stream_handle(stream), ctypes.byref(o))
    _check(rc, "tile_copy_rowsum")
    return out


def tile_stage_image(src: torch.Tensor, tile_m: int, tile_n: int, tile_row: int = 0,
                     tile_col: int = 0, stream=None) -> torch.Tensor:
    """Raw shared-memory bytes of one staged tile (debug; see include/mbtile.h)."""
    lib = _load()
    fn = lib.tile_stage_image
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                   ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    M, N, ld = _matrix(src, "src")
    boxes = tile_n * src.element_size() // 128
    image = torch.zeros(boxes * tile_m * 128, dtype=torch.uint8, device=src.device)
    rc = fn(src.data_ptr(), M, N, ld, tile_m, tile_n, DTYPE_CODE[src.dtype], tile_row, tile_col,
            image.data_ptr(), _stream_handle(stream))
    _check(rc, "tile_stage_image")
    return image


def tile_status(stream=None) -> tuple[int, list[int]]:
    """Synchronise ``stream`` and read-and-clear the device status word.
    Returns (code, [code, block, stage, role * 2 + parity])."""
    info = (ctypes.c_int32 * 4)()
    rc = _load().tile_status(_stream_handle(stream), info)
    return rc, list(info)


def tile_plan(op: int, M: int, N: int, tile_m: int, tile_n: int, stages: int,
              dtype: torch.dtype, *, num_sms: int, smem_optin: int, fit_per_sm: int,
              with_workspace: bool = False, **opt) -> dict:
    o = _opts(**opt)
    p = Plan()
    rc = _load().tile_plan(op, M, N, tile_m, tile_n, stages, DTYPE_CODE[dtype],
                           ctypes.byref(o), num_sms, smem_optin, fit_per_sm,
                           int(with_workspace), ctypes.byref(p))
    _check(rc, "tile_plan")
    return p.as_dict()


def tile_plan_device(op: int, M: int, N: int, tile_m: int, tile_n: int, stages: int,
                     dtype: torch.dtype, **opt) -> dict:
    """The plan the call would run on the current device (see include/mbtile.h)."""
    o = _opts(**opt)
    p = Plan()
    rc = _load().tile_plan_device(op, M, N, tile_m, tile_n, stages, DTYPE_CODE[dtype],
                                  ctypes.byref(o), ctypes.byref(p))
    _check(rc, "tile_plan_device")
    return p.as_dict()


def tile_device_info(device: int | None = None) -> dict:
    dev = torch.cuda.current_device() if device is None else device
    sms, smem = ctypes.c_int(0), ctypes.c_int(0)
    gbs = ctypes.c_double(0.0)
    rc = _load().tile_device_info(dev, ctypes.byref(sms), ctypes.byref(smem), ctypes.byref(gbs))
    _check(rc, "tile_device_info")
    return {"num_sms": sms.value, "smem_optin": smem.value, "hbm_gbs_theoretical": gbs.value}


def tile_rowsum_noalloc(src: torch.Tensor, out: torch.Tensor, tile_m: int = 64,
                        tile_n: int = 256, stages: int = 4, *, stream=None,
                        **opt) -> torch.Tensor:
    """Row sums through ``tile_rowsum_noalloc``: for callers that cannot
    allocate device memory, the library uses its own static scratch array
    instead of a workspace (see include/mbtile.h).  ``out`` must be given."""
    lib = _load()
    fn = lib.tile_rowsum_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                   ctypes.POINTER(Opts)]
    fn.restype = ctypes.c_int
    M, N, ld_s = _matrix(src, "src")
    if out.dtype != torch.float32 or out.numel() != M or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 tensor of M elements")
    o = _opts(ld_src=ld_s, **opt)
    rc = fn(src.data_ptr(), out.data_ptr(), M, N, tile_m, tile_n, stages,
            DTYPE_CODE[src.dtype], _stream_handle(stream), ctypes.byref(o))
    _check(rc, "tile_rowsum_noalloc")
    return out


def tile_copy_host(src: torch.Tensor, dst: torch.Tensor, tile_m: int = 128, tile_n: int = 64,
                   stages: int = 3, *, slab_rows: int = 0, **opt) -> torch.Tensor:
    """dst[i, j] = src[i, j] for HOST tensors: the library streams row slabs
    through the current device (copy in, tile pipeline, copy out, overlapped).
    Pinned tensors (``pin_memory=True``) let the copies overlap.  Synchronous."""
    M, N, ld_s = _host_matrix(src, "src")
    Md, Nd, ld_d = _host_matrix(dst, "dst")
    if (M, N) != (Md, Nd) or src.dtype != dst.dtype:
        raise ValueError("src and dst must have the same shape and dtype")
    o = _opts(ld_src=ld_s, ld_dst=ld_d, host_slab_rows=slab_rows, **opt)
    rc = _load().tile_copy_host(src.data_ptr(), dst.data_ptr(), M, N, tile_m, tile_n, stages,
                                DTYPE_CODE[src.dtype], ctypes.byref(o))
    _check(rc, "tile_copy_host")
    return dst


def tile_rowsum_host(src: torch.Tensor, out: torch.Tensor | None = None, tile_m: int = 64,
                     tile_n: int = 256, stages: int = 2, *, slab_rows: int = 0,
                     **opt) -> torch.Tensor:
    """out[i] = sum_j src[i, j] in fp32 for a HOST tensor (out on the host
    too), streamed through the current device in row slabs.  Synchronous."""
    M, N, ld_s = _host_matrix(src, "src")
    if out is None:
        out = torch.empty(M, dtype=torch.float32, pin_memory=src.is_pinned())
    if (out.device.type != "cpu" or out.dtype != torch.float32 or out.numel() != M
            or not out.is_contiguous()):
        raise ValueError("out must be a contiguous float32 host tensor of M elements")
    o = _opts(ld_src=ld_s, host_slab_rows=slab_rows, **opt)
    rc = _load().tile_rowsum_host(src.data_ptr(), out.data_ptr(), M, N, tile_m, tile_n, stages,
                                  DTYPE_CODE[src.dtype], ctypes.byref(o))
    _check(rc, "tile_rowsum_host")
    return out


def tile_colsum_host(src: torch.Tensor, out: torch.Tensor | None = None, tile_m: int = 64,
                     tile_n: int = 256, stages: int = 2, *, slab_rows: int = 0,
                     **opt) -> torch.Tensor:
    """out[j] = sum_i src[i, j] in fp32 for a HOST tensor (out on the host too),
    streamed through the current device in row slabs whose column sums are
    added on the device in slab order.  Any row pitch.  Synchronous."""
    M, N, ld_s = _host_matrix(src, "src")
    if out is None:
        out = torch.empty(N, dtype=torch.float32, pin_memory=src.is_pinned())
    if (out.device.type != "cpu" or out.dtype != torch.float32 or out.numel() != N
            or not out.is_contiguous()):
        raise ValueError("out must be a contiguous float32 host tensor of N elements")
    o = _opts(ld_src=ld_s, host_slab_rows=slab_rows, **opt)
    rc = _load().tile_colsum_host(src.data_ptr(), out.data_ptr(), M, N, tile_m, tile_n, stages,
                                  DTYPE_CODE[src.dtype], ctypes.byref(o))
    _check(rc, "tile_colsum_host")
    return out


def tile_host_release() -> None:
    """Free the current device's idle staging memory of the host-buffer forms."""
    _check(_load().tile_host_release(), "tile_host_release")


def tile_workspace_release(stream=None) -> None:
    """Free (in stream order) the sum workspace the library keeps for the
    current device and ``stream``."""
    _check(_load().tile_workspace_release(_stream_handle(stream)), "tile_workspace_release")


def tile_read_checksum(buf: torch.Tensor, out: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """XOR of all 32-bit words of a contiguous CUDA tensor's bytes (the
    read-bandwidth reference, see include/mbtile.h); returns an int32[1]
    device tensor holding the checksum's bits."""
    if buf.device.type != "cuda" or not buf.is_contiguous():
        raise ValueError("buf must be a contiguous CUDA tensor")
    if out is None:
        with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream()):
            out = torch.empty(1, dtype=torch.int32, device=buf.device)
    rc = _load().tile_read_checksum(buf.data_ptr(), buf.numel() * buf.element_size(),
                                    out.data_ptr(), _stream_handle(stream))
    _check(rc, "tile_read_checksum")
    return out
