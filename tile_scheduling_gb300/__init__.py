"""Python binding of libtsgemm (persistent bf16 GEMM with static / Cluster Launch
Control tile scheduling, and the grid-stride int16 copy) for one GB300.

This module only marshals arguments: torch tensors become device pointers and
sizes, the current torch stream becomes a cudaStream_t, and every computation
runs in the library's CUDA kernels.  There is no fallback: if the shared
library is missing or fails to load, importing this package raises.

The C entry points are declared in include/tsgemm.h; the functions here have
the same names.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libtsgemm.so")

TS_OK, TS_ERR_INVALID_ARG, TS_ERR_UNSUPPORTED, TS_ERR_CUDA, TS_ERR_TIMEOUT = range(5)
TS_SCHED_STATIC, TS_SCHED_CLC, TS_SCHED_NONPERSISTENT = 0, 1, 2
TS_OUT_BF16, TS_OUT_F32 = 0, 1
TS_TILE_AUTO, TS_TILE_128x128, TS_TILE_128x256, TS_TILE_256x256_2CTA = range(4)
PROTOCOL_LOG_ROLES = 20  # roles per CTA in a protocol log (ts_gemm_opts.protocol_log)

_SCHED = {"static": TS_SCHED_STATIC, "clc": TS_SCHED_CLC, "nonpersistent": TS_SCHED_NONPERSISTENT}
_TILE = {"auto": TS_TILE_AUTO, "128x128": TS_TILE_128x128, "128x256": TS_TILE_128x256,
         "256x256": TS_TILE_256x256_2CTA}
_OUT = {torch.bfloat16: TS_OUT_BF16, torch.float32: TS_OUT_F32}

EXPORTED = ("ts_gemm_bf16", "ts_gemm_bf16_ex", "ts_gemm_launch_info", "ts_gemm_bf16_checked_noalloc",
            "ts_copy_i16", "ts_spin",
            "ts_spin_wait_started", "ts_sync_and_check", "ts_num_sms", "ts_status_string",
            "ts_last_error_detail")


class TsError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{_status_name(status)}: {detail}")
        self.status = status
        self.detail = detail


class GemmOpts(ctypes.Structure):
    _fields_ = [("tile", ctypes.c_int32), ("max_workers", ctypes.c_int32), ("lda", ctypes.c_int64),
                ("ldb", ctypes.c_int64), ("ldd", ctypes.c_int64), ("timeout_s", ctypes.c_double),
                ("trace", ctypes.c_void_p), ("raster_group", ctypes.c_int32), ("split_tail", ctypes.c_int32),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_int64), ("skip_tiles", ctypes.c_void_p),
                ("row_sums", ctypes.c_void_p), ("epi_warps", ctypes.c_int32), ("merge", ctypes.c_int32),
                ("inputs_ready", ctypes.c_int32), ("protocol_log", ctypes.c_void_p),
                ("protocol_log_cap", ctypes.c_int32)]


class LaunchInfo(ctypes.Structure):
    _fields_ = [("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("tiles_m", ctypes.c_int64), ("tiles_n", ctypes.c_int64),
                ("num_tiles", ctypes.c_int64), ("grid_ctas", ctypes.c_int64), ("workers", ctypes.c_int64),
                ("smem_bytes", ctypes.c_int32), ("tma_store", ctypes.c_int32), ("num_units", ctypes.c_int64),
                ("split_tiles", ctypes.c_int64), ("split_parts", ctypes.c_int32), ("resident", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("epi_warps", ctypes.c_int32), ("merge", ctypes.c_int32),
                ("clc_lazy", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class RowsOpts(ctypes.Structure):
    _fields_ = [("tiles", ctypes.c_int64), ("rows_device", ctypes.c_void_p), ("skip_rows", ctypes.c_void_p),
                ("threads", ctypes.c_int32), ("max_workers", ctypes.c_int32), ("timeout_s", ctypes.c_double),
                ("trace", ctypes.c_void_p), ("chunk", ctypes.c_int64), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_int64), ("pack", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class GemmProtocol(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "cluster", "stages", "tx_bytes", "full_arrivals", "empty_arrivals", "accumulators", "tmem_full_arrivals",
        "tmem_empty_arrivals", "clc_slots", "clc_full_arrivals", "clc_empty_arrivals", "clc_response_bytes",
        "epilogue_warps", "stage_bytes", "aux_empty_arrivals", "merge", "a_stage_bytes")]


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libtsgemm.so not built ({path}); run python tile_scheduling_gb300/build.py")
    lib = ctypes.CDLL(path)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.ts_gemm_bf16.argtypes = [P, P, P, I64, I64, I64, I32, I32, P]
    lib.ts_gemm_bf16_ex.argtypes = [P, P, P, I64, I64, I64, I32, I32, ctypes.POINTER(GemmOpts), P]
    lib.ts_gemm_bf16_host.argtypes = [P, P, P, P, P, P, I64, I64, I64, I32, I32, ctypes.POINTER(GemmOpts), P]
    lib.ts_gemm_launch_info.argtypes = [I64, I64, I64, I32, I32, ctypes.POINTER(GemmOpts),
                                        ctypes.POINTER(LaunchInfo)]
    lib.ts_gemm_bf16_checked_noalloc.argtypes = [P, P, P, I64, I64, I64, I32, I32, P, P]
    lib.ts_gemm_tile_coords.argtypes = [I64, I64, I64, I32, I32, ctypes.POINTER(GemmOpts), I64, I64, P, P]
    lib.ts_gemm_protocol_info.argtypes = [I32, I32, I32, I32, ctypes.POINTER(GemmProtocol)]
    lib.ts_protocol_check.argtypes = [I32, P, I32, I32, P, P, P, ctypes.c_char_p, I64, ctypes.POINTER(I64),
                                      ctypes.c_char_p, I32]
    lib.ts_protocol_check.restype = I32
    lib.ts_protocol_check_ex.argtypes = [I32, P, I32, I32, P, P, P, I32, P, ctypes.c_char_p, I64, ctypes.POINTER(I64),
                                         ctypes.c_char_p, I32]
    lib.ts_protocol_check_ex.restype = I32
    lib.ts_gemm_bf16_grouped.argtypes = [P, P, P, I64, I64, I64, P, I32, I32, ctypes.POINTER(GemmOpts), P]
    lib.ts_gemm_grouped_launch_info.argtypes = [I64, I64, I64, P, I32, I32, ctypes.POINTER(GemmOpts),
                                                ctypes.POINTER(LaunchInfo)]
    lib.ts_gemm_grouped_order.argtypes = [I64, P, P]
    lib.ts_copy_i16.argtypes = [P, P, I64, P]
    lib.ts_copy_i16_rows.argtypes = [P, P, I64, P, I64, I32, ctypes.POINTER(RowsOpts), P]
    lib.ts_copy_rows_launch_info.argtypes = [I64, I64, I32, ctypes.POINTER(RowsOpts), ctypes.POINTER(LaunchInfo)]
    lib.ts_spin.argtypes = [I32, I64, P, P]
    lib.ts_spin_wait_started.argtypes = [P, I32, ctypes.c_double]
    lib.ts_sync_and_check.argtypes = [P]
    lib.ts_num_sms.argtypes = []
    lib.ts_num_sms.restype = I32
    lib.ts_status_string.argtypes = [ctypes.c_int]
    lib.ts_status_string.restype = ctypes.c_char_p
    lib.ts_last_error_detail.argtypes = []
    lib.ts_last_error_detail.restype = ctypes.c_char_p
    for name in ("ts_gemm_bf16", "ts_gemm_bf16_ex", "ts_gemm_launch_info", "ts_gemm_bf16_checked_noalloc",
                 "ts_gemm_tile_coords", "ts_gemm_protocol_info", "ts_gemm_bf16_grouped", "ts_gemm_grouped_launch_info",
                 "ts_gemm_grouped_order", "ts_copy_i16", "ts_copy_i16_rows", "ts_copy_rows_launch_info", "ts_spin",
                 "ts_spin_wait_started", "ts_sync_and_check"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


_lib = load_library()


def _status_name(s: int) -> str:
    return _lib.ts_status_string(s).decode()


def _check(status: int) -> None:
    if status != TS_OK:
        raise TsError(status, _lib.ts_last_error_detail().decode())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _sched(s) -> int:
    return _SCHED[s] if isinstance(s, str) else int(s)


def _opts(tile="auto", max_workers=0, lda=0, ldb=0, ldd=0, timeout_s=0.0, trace=None, raster_group=0,
          split_tail=0, workspace=None, skip_tiles=None, row_sums=None, epi_warps=0, merge=0, inputs_ready=0,
          protocol_log=None):
    o = GemmOpts()
    o.epi_warps = int(epi_warps)
    o.merge = int(merge)
    o.inputs_ready = int(inputs_ready)
    if protocol_log is not None:
        if protocol_log.dtype != torch.int32 or not protocol_log.is_cuda or protocol_log.dim() != 3 or \
                not protocol_log.is_contiguous() or protocol_log.shape[1] != PROTOCOL_LOG_ROLES:
            raise TypeError(f"protocol_log must be a contiguous int32 CUDA tensor [CTAs][{PROTOCOL_LOG_ROLES}][cap + 1]")
        o.protocol_log = protocol_log.data_ptr()
        o.protocol_log_cap = protocol_log.shape[2] - 1
    if row_sums is not None:
        if row_sums.dtype != torch.float32 or not row_sums.is_cuda or not row_sums.is_contiguous():
            raise TypeError("row_sums must be a contiguous float32 CUDA tensor")
        o.row_sums = row_sums.data_ptr()
    if skip_tiles is not None:
        if skip_tiles.dtype not in (torch.uint8, torch.bool) or not skip_tiles.is_cuda or not skip_tiles.is_contiguous():
            raise TypeError("skip_tiles must be a contiguous uint8/bool CUDA tensor (one entry per tile)")
        o.skip_tiles = skip_tiles.data_ptr()
    o.split_tail = int(split_tail)
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise TypeError("workspace must be a contiguous CUDA tensor")
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    o.tile = _TILE[tile] if isinstance(tile, str) else int(tile)
    o.max_workers = int(max_workers)
    o.lda, o.ldb, o.ldd = int(lda), int(ldb), int(ldd)
    o.timeout_s = float(timeout_s)
    if trace is not None:
        if trace.dtype != torch.int64 or not trace.is_cuda or not trace.is_contiguous():
            raise TypeError("trace must be a contiguous int64 CUDA tensor")
        o.trace = trace.data_ptr()
    o.raster_group = int(raster_group)
    return o


def _matrix(t: torch.Tensor, name: str, dtype) -> int:
    if not isinstance(t, torch.Tensor) or t.dtype != dtype:
        raise TypeError(f"{name} must be a {dtype} tensor")
    if not t.is_cuda:
        raise TypeError(f"{name} must be on a CUDA device")
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with unit column stride")
    return t.stride(0)


def _gemm_args(A, B, D):
    lda = _matrix(A, "A", torch.bfloat16)
    ldb = _matrix(B, "B", torch.bfloat16)
    if D.dtype not in _OUT:
        raise TypeError("D must be bfloat16 or float32")
    ldd = _matrix(D, "D", D.dtype)
    M, K = A.shape
    N, K2 = B.shape
    if K2 != K or tuple(D.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}, D {tuple(D.shape)}")
    return M, N, K, lda, ldb, ldd


_WORKSPACES: dict = {}


def workspace_for(nbytes: int, device=None, stream=None) -> torch.Tensor:
    """A zero-filled device workspace of at least ``nbytes``, cached per device and stream.

    The kernel leaves the workspace zeroed after every normal launch, so one
    buffer serves every call on a stream; calls on different streams, which may
    overlap on the GPU, get buffers of their own.  A buffer is allocated and
    zeroed on the stream it serves, so the zeroing is ordered before the
    launches that use it (``stream``: a torch stream or a raw handle; default
    the current stream)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    elif not isinstance(stream, torch.cuda.Stream):
        stream = torch.cuda.ExternalStream(int(stream), device=dev)
    key = (dev, stream.cuda_stream)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < nbytes:
        with torch.cuda.stream(stream):
            ws = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=dev)
        _WORKSPACES[key] = ws
    return ws


def ts_gemm_bf16_ex(A: torch.Tensor, B: torch.Tensor, D: torch.Tensor, sched="static", tile="auto",
                    max_workers=0, timeout_s=0.0, trace=None, raster_group=0, workspace="auto", split_tail=0,
                    skip_tiles=None, row_sums=None, epi_warps=0, merge=0, inputs_ready=0, protocol_log=None,
                    stream=None) -> None:
    """D = A @ B.T for bf16 A [M, K] and B [N, K]; D [M, N] is bf16 or fp32.

    Rows may be strided (the row stride becomes lda / ldb / ldd).  ``workspace``
    ("auto": a cached zero-filled buffer; None: no split tiles; or a CUDA tensor)
    lets the tiles that would leave the last wave partly empty be split along K.  ``epi_warps``: 4, 8,
    16 (256-column tiles) or 0 (automatic); ``merge``: 1 for the Merge barrier layout (A and B from
    separate producer warps); ``inputs_ready``: 1 when A, B and skip_tiles were final before the
    previous kernel in the stream began (their loads then overlap that kernel's tail);
    ``protocol_log``: a zeroed int32 CUDA tensor [CTAs][PROTOCOL_LOG_ROLES][cap + 1] that the
    protocol-logging build fills with every role's barrier operations (a test instrument).
    Asynchronous on ``stream`` (default: torch's current stream)."""
    M, N, K, lda, ldb, ldd = _gemm_args(A, B, D)
    lda, ldb, ldd = (lda if M > 1 else 0), (ldb if N > 1 else 0), (ldd if M > 1 else 0)
    workspace = _resolve_workspace(M, N, K, _OUT[D.dtype], sched, workspace,
                                   -1 if (skip_tiles is not None or row_sums is not None) else split_tail, tile=tile,
                                   max_workers=max_workers, lda=lda, ldb=ldb, ldd=ldd, stream=stream)
    o = _opts(tile, max_workers, lda, ldb, ldd, timeout_s, trace, raster_group, split_tail, workspace, skip_tiles,
              row_sums, epi_warps, merge, inputs_ready, protocol_log)
    _check(_lib.ts_gemm_bf16_ex(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
                                ctypes.c_void_p(D.data_ptr()), M, N, K, _OUT[D.dtype], _sched(sched),
                                ctypes.byref(o), _stream_handle(stream)))


def ts_gemm_bf16_host(A_host: torch.Tensor, B_host: torch.Tensor, D_host: torch.Tensor, A: torch.Tensor,
                      B: torch.Tensor, D: torch.Tensor, sched="static", tile="auto", workspace="auto", epi_warps=0,
                      stream=None) -> None:
    """D_host = A_host @ B_host.T through the device buffers A, B, D: the copies in, the GEMM and the
    copy out are queued on ``stream`` (page-locked host tensors keep them asynchronous).  All six
    tensors are contiguous, each host tensor shaped and typed as its device one."""
    for h, d, name in ((A_host, A, "A"), (B_host, B, "B"), (D_host, D, "D")):
        if h.is_cuda or not h.is_contiguous() or not d.is_contiguous():
            raise TypeError(f"{name}_host must be a contiguous host tensor and {name} a contiguous CUDA tensor")
        if h.shape != d.shape or h.dtype != d.dtype:
            raise ValueError(f"{name}_host and {name} differ in shape or dtype")
    M, N, K, _, _, _ = _gemm_args(A, B, D)
    workspace = _resolve_workspace(M, N, K, _OUT[D.dtype], sched, workspace, 0, tile=tile, stream=stream)
    o = _opts(tile=tile, workspace=workspace, epi_warps=epi_warps)
    _check(_lib.ts_gemm_bf16_host(ctypes.c_void_p(A_host.data_ptr()), ctypes.c_void_p(B_host.data_ptr()),
                                  ctypes.c_void_p(D_host.data_ptr()), ctypes.c_void_p(A.data_ptr()),
                                  ctypes.c_void_p(B.data_ptr()), ctypes.c_void_p(D.data_ptr()), M, N, K,
                                  _OUT[D.dtype], _sched(sched), ctypes.byref(o), _stream_handle(stream)))


def ts_gemm_bf16(A: torch.Tensor, B: torch.Tensor, D: torch.Tensor, sched="static", stream=None) -> None:
    """D = A @ B.T with the default tile choice; all three tensors contiguous."""
    M, N, K, lda, ldb, ldd = _gemm_args(A, B, D)
    if (M > 1 and (lda != K or ldd != N)) or (N > 1 and ldb != K):
        raise ValueError("ts_gemm_bf16 takes dense rows; use ts_gemm_bf16_ex for strided ones")
    _check(_lib.ts_gemm_bf16(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
                             ctypes.c_void_p(D.data_ptr()), M, N, K, _OUT[D.dtype], _sched(sched),
                             _stream_handle(stream)))


def ts_gemm_bf16_checked_noalloc(A: torch.Tensor, B: torch.Tensor, D: torch.Tensor, bad_tiles: torch.Tensor,
                                 sched="static", stream=None) -> None:
    """D = A @ B.T plus a tile-coverage check, without any device allocation.

    For callers that cannot call cudaMalloc: the per-tile trace lives in a
    fixed 2 MiB array inside the library (at most 65536 output tiles) rather
    than in caller memory.  ``bad_tiles`` (one int32 on the device) receives
    the number of tiles not computed exactly once.  Calls that overlap on the
    GPU share that array and race; the first call on a device should come
    before any stream capture."""
    M, N, K, lda, ldb, ldd = _gemm_args(A, B, D)
    if (M > 1 and (lda != K or ldd != N)) or (N > 1 and ldb != K):
        raise ValueError("dense rows required")
    if bad_tiles.dtype != torch.int32 or not bad_tiles.is_cuda or bad_tiles.numel() < 1:
        raise TypeError("bad_tiles must be an int32 CUDA tensor")
    _check(_lib.ts_gemm_bf16_checked_noalloc(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
                                             ctypes.c_void_p(D.data_ptr()), M, N, K, _OUT[D.dtype], _sched(sched),
                                             ctypes.c_void_p(bad_tiles.data_ptr()), _stream_handle(stream)))


def ts_gemm_bf16_ptr(A: int, B: int, D: int, M: int, N: int, K: int, out: int, sched=0, stream=None,
                     **opts) -> int:  # no workspace unless one is passed
    """Raw-pointer call of ts_gemm_bf16_ex; returns the status without raising."""
    o = _opts(**opts)
    return _lib.ts_gemm_bf16_ex(ctypes.c_void_p(A), ctypes.c_void_p(B), ctypes.c_void_p(D), M, N, K, out,
                                _sched(sched), ctypes.byref(o), _stream_handle(stream))


def _launch_info_raw(M: int, N: int, K: int, out, sched, **opts) -> dict:
    o = _opts(**opts)
    info = LaunchInfo()
    _check(_lib.ts_gemm_launch_info(M, N, K, int(out), _sched(sched), ctypes.byref(o), ctypes.byref(info)))
    return {f: getattr(info, f) for f, _ in LaunchInfo._fields_}


def _resolve_workspace(M, N, K, out, sched, workspace, split_tail, stream=None, **opts):
    if not isinstance(workspace, str):
        return workspace
    if split_tail < 0:
        return None
    need = _launch_info_raw(M, N, K, out, sched, split_tail=split_tail, **opts)["workspace_bytes"]
    return workspace_for(need, stream=stream) if need > 0 else None


def ts_gemm_launch_info(M: int, N: int, K: int, out=TS_OUT_BF16, sched="static", workspace="auto", split_tail=0,
                        **opts) -> dict:
    """The launch ts_gemm_bf16_ex would make; ``workspace`` resolves as in that call."""
    ws = _resolve_workspace(M, N, K, out, sched, workspace, split_tail, **opts)
    return _launch_info_raw(M, N, K, out, sched, workspace=ws, split_tail=split_tail, **opts)


def ts_gemm_tile_coords(M: int, N: int, K: int, out=TS_OUT_BF16, sched="static", first=0, count=None, tile="auto",
                        raster_group=0):
    """(m_block, n_block) int32 arrays: the output tile that each tile id of the launch covers."""
    import numpy as np

    o = _opts(tile=tile, raster_group=raster_group)
    if count is None:
        if o.tile == TS_TILE_AUTO:  # the automatic choice depends on the device
            info = _launch_info_raw(M, N, K, out, sched, tile=tile, raster_group=raster_group)
            tiles = info["tiles_m"] * info["tiles_n"]
        else:
            bm = 256 if o.tile == TS_TILE_256x256_2CTA else 128
            bn = 128 if o.tile == TS_TILE_128x128 else 256
            tiles = -(-max(M, 0) // bm) * -(-max(N, 0) // bn)
        count = tiles - first
    mb = np.zeros(max(count, 0), dtype=np.int32)
    nb = np.zeros(max(count, 0), dtype=np.int32)
    _check(_lib.ts_gemm_tile_coords(M, N, K, int(out), _sched(sched), ctypes.byref(o), first, count,
                                    mb.ctypes.data, nb.ctypes.data))
    return mb, nb


def _offsets(k_offsets) -> "np.ndarray":
    import numpy as np

    off = np.ascontiguousarray(np.asarray(k_offsets, dtype=np.int64))
    if off.ndim != 1 or off.size < 2:
        raise ValueError("k_offsets must list groups + 1 offsets")
    return off


def ts_gemm_grouped_launch_info(M: int, N: int, k_offsets, out=TS_OUT_BF16, sched="static", **opts) -> dict:
    off = _offsets(k_offsets)
    o = _opts(**opts)
    info = LaunchInfo()
    _check(_lib.ts_gemm_grouped_launch_info(M, N, off.size - 1, off.ctypes.data, int(out), _sched(sched),
                                            ctypes.byref(o), ctypes.byref(info)))
    return {f: getattr(info, f) for f, _ in LaunchInfo._fields_}


def ts_gemm_grouped_order(k_offsets) -> "np.ndarray":
    """The order in which ts_gemm_bf16_grouped schedules the groups (longest K range first)."""
    import numpy as np

    off = _offsets(k_offsets)
    order = np.zeros(off.size - 1, dtype=np.int32)
    _check(_lib.ts_gemm_grouped_order(off.size - 1, off.ctypes.data, order.ctypes.data))
    return order


def ts_gemm_bf16_grouped(A: torch.Tensor, B: torch.Tensor, D: torch.Tensor, k_offsets, sched="static", tile="auto",
                         max_workers=0, timeout_s=0.0, trace=None, raster_group=0, skip_tiles=None,
                         row_sums=None, epi_warps=0, merge=0, inputs_ready=0, protocol_log=None,
                         stream=None) -> None:
    """D[g] = A[:, k_g:k_g+1] @ B[:, k_g:k_g+1].T for every group g (k_offsets: groups + 1 multiples of 64).

    A [M, >=K] and B [N, >=K] bf16 with unit column stride; D [groups, M, N]
    bf16 or fp32 whose groups are M * ldd elements apart."""
    off = _offsets(k_offsets)
    G = off.size - 1
    lda = _matrix(A, "A", torch.bfloat16)
    ldb = _matrix(B, "B", torch.bfloat16)
    if D.dtype not in _OUT or not D.is_cuda or D.dim() != 3 or D.stride(2) != 1:
        raise TypeError("D must be a [groups, M, N] bf16/fp32 CUDA tensor with unit column stride")
    M, N = A.shape[0], B.shape[0]
    if tuple(D.shape) != (G, M, N) or (G > 1 and D.stride(0) != M * D.stride(1)):
        raise ValueError(f"D must be [{G}, {M}, {N}] with groups M rows apart")
    if int(off[-1]) > min(A.shape[1], B.shape[1]):
        raise ValueError("k_offsets reach past the columns of A or B")
    o = _opts(tile, max_workers, lda if M > 1 else 0, ldb if N > 1 else 0, D.stride(1) if M > 1 else 0, timeout_s,
              trace, raster_group, skip_tiles=skip_tiles, row_sums=row_sums, epi_warps=epi_warps, merge=merge,
              inputs_ready=inputs_ready, protocol_log=protocol_log)
    _check(_lib.ts_gemm_bf16_grouped(ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
                                     ctypes.c_void_p(D.data_ptr()), M, N, G, off.ctypes.data, _OUT[D.dtype],
                                     _sched(sched), ctypes.byref(o), _stream_handle(stream)))


def ts_gemm_protocol_info(tile="256x256", out=TS_OUT_BF16, epi_warps=0, merge=0) -> dict:
    """Barrier layout and arrival counts of a kernel variant (no GPU needed)."""
    proto = GemmProtocol()
    _check(_lib.ts_gemm_protocol_info(_TILE[tile] if isinstance(tile, str) else int(tile), int(out), int(epi_warps),
                                      int(merge), ctypes.byref(proto)))
    return {f: getattr(proto, f) for f, _ in GemmProtocol._fields_}


def ts_copy_i16(src: torch.Tensor, dst: torch.Tensor, stream=None) -> None:
    """dst[i] = src[i] for contiguous int16 CUDA tensors of equal size."""
    for t, name in ((src, "src"), (dst, "dst")):
        if t.dtype != torch.int16 or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous int16 CUDA tensor")
    if src.numel() != dst.numel():
        raise ValueError("src and dst differ in size")
    _check(_lib.ts_copy_i16(ctypes.c_void_p(src.data_ptr()), ctypes.c_void_p(dst.data_ptr()), src.numel(),
                            _stream_handle(stream)))


def ts_copy_i16_ptr(src: int, dst: int, n: int, stream=None) -> int:
    return _lib.ts_copy_i16(ctypes.c_void_p(src), ctypes.c_void_p(dst), n, _stream_handle(stream))


def _rows_opts(tiles=0, rows_device=None, skip_rows=None, threads=0, max_workers=0, timeout_s=0.0, trace=None,
               chunk=0, workspace=None, pack=0):
    o = RowsOpts()
    o.tiles = int(tiles)
    o.chunk = int(chunk)
    o.pack = int(pack)
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise TypeError("workspace must be a contiguous CUDA tensor")
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    o.threads = int(threads)
    o.max_workers = int(max_workers)
    o.timeout_s = float(timeout_s)
    for name, t, dtype in (("rows_device", rows_device, torch.int64), ("skip_rows", skip_rows, torch.uint8),
                           ("trace", trace, torch.int64)):
        if t is None:
            continue
        if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous {dtype} CUDA tensor")
        setattr(o, name, t.data_ptr())
    return o


def ts_copy_rows_launch_info(n: int, rows: int, sched="clc", **opts) -> dict:
    o = _rows_opts(**{k: v for k, v in opts.items() if k in ("tiles", "threads", "max_workers", "chunk", "pack")})
    info = LaunchInfo()
    _check(_lib.ts_copy_rows_launch_info(int(n), int(rows), _sched(sched), ctypes.byref(o), ctypes.byref(info)))
    return {f: getattr(info, f) for f, _ in LaunchInfo._fields_}


def ts_copy_i16_rows(src: torch.Tensor, dst: torch.Tensor, offsets: torch.Tensor, rows=None, sched="clc", tiles=0,
                     rows_device=None, skip_rows=None, threads=0, max_workers=0, timeout_s=0.0, trace=None,
                     chunk=0, workspace=None, pack=0, stream=None) -> None:
    """Copy rows [offsets[r], offsets[r+1]) of a jagged int16 array through a work queue.

    src and dst: contiguous int16 CUDA tensors of equal size n; offsets: int64
    CUDA tensor of rows + 1 entries (rows defaults to offsets.numel() - 1).
    Tiles past the row count (tiles > rows, or rows_device below rows) and rows
    marked in skip_rows copy nothing but still take part in the queue.
    chunk > 0 cuts rows into work tiles of at most chunk elements; with
    pack=1 the rows are laid end to end and every tile copies chunk of their
    elements.  The planning workspace is allocated here unless one is passed."""
    for t, name in ((src, "src"), (dst, "dst")):
        if t.dtype != torch.int16 or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous int16 CUDA tensor")
    if src.numel() != dst.numel():
        raise ValueError("src and dst differ in size")
    if offsets.dtype != torch.int64 or not offsets.is_cuda or not offsets.is_contiguous():
        raise TypeError("offsets must be a contiguous int64 CUDA tensor")
    if rows is None:
        rows = max(offsets.numel() - 1, 0)
    if offsets.numel() < rows + 1:
        raise ValueError("offsets needs rows + 1 entries")
    if skip_rows is not None and skip_rows.numel() < rows:
        raise ValueError("skip_rows needs one byte per row")
    if chunk and workspace is None:
        need = ts_copy_rows_launch_info(src.numel(), rows, sched, tiles=tiles, chunk=chunk,
                                        pack=pack)["workspace_bytes"]
        workspace = torch.empty(need, dtype=torch.uint8, device=src.device)
    o = _rows_opts(tiles, rows_device, skip_rows, threads, max_workers, timeout_s, trace, chunk, workspace, pack)
    min_tiles = (0 if pack else int(rows)) + (-(-src.numel() // int(chunk)) if chunk else 0)
    if trace is not None and trace.numel() < 2 * max(int(tiles), min_tiles):
        raise ValueError("trace needs 2 * tiles entries")
    _check(_lib.ts_copy_i16_rows(ctypes.c_void_p(src.data_ptr()), ctypes.c_void_p(dst.data_ptr()), src.numel(),
                                 ctypes.c_void_p(offsets.data_ptr()), int(rows), _sched(sched), ctypes.byref(o),
                                 _stream_handle(stream)))


def ts_copy_i16_rows_ptr(src: int, dst: int, n: int, offsets: int, rows: int, sched=1, stream=None, **opts) -> int:
    """Raw-pointer call of ts_copy_i16_rows; returns the status without raising."""
    o = _rows_opts(**opts)
    return _lib.ts_copy_i16_rows(ctypes.c_void_p(src), ctypes.c_void_p(dst), int(n), ctypes.c_void_p(offsets),
                                 int(rows), _sched(sched), ctypes.byref(o), _stream_handle(stream))


def ts_spin(ctas: int, duration_ns: int, started: torch.Tensor, stream=None) -> None:
    """Hold ``ctas`` SMs for ``duration_ns``; ``started`` is a pinned int32 host tensor."""
    if started.dtype != torch.int32 or started.is_cuda or not started.is_pinned():
        raise TypeError("started must be a pinned int32 CPU tensor")
    _check(_lib.ts_spin(int(ctas), int(duration_ns), ctypes.c_void_p(started.data_ptr()), _stream_handle(stream)))


def ts_spin_wait_started(started: torch.Tensor, expected: int, timeout_s: float = 5.0) -> None:
    _check(_lib.ts_spin_wait_started(ctypes.c_void_p(started.data_ptr()), int(expected), float(timeout_s)))


def ts_protocol_check(program, max_states: int = 20_000_000):
    """Explore a barrier-protocol program (see tile_scheduling_gb300.protocol)."""
    from .protocol import check

    return check(program, max_states)


def ts_protocol_check_ex(program, max_states: int = 20_000_000):
    """Explore a barrier-protocol program with global counters (the split tiles' handoff); the
    program's counters and their expected reductions travel with it."""
    from .protocol import check

    return check(program, max_states)


def ts_sync_and_check(stream=None) -> None:
    """Synchronise and raise TsError for a device-side timeout (or CUDA error).

    After a timeout the cached split-tile workspaces may hold partial counters,
    so they are zeroed again before the error is raised."""
    st = _lib.ts_sync_and_check(_stream_handle(stream))
    if st == TS_ERR_TIMEOUT:
        detail = _lib.ts_last_error_detail().decode()
        for ws in _WORKSPACES.values():
            ws.zero_()
        torch.cuda.synchronize()
        raise TsError(st, detail)
    _check(st)


def ts_num_sms() -> int:
    return int(_lib.ts_num_sms())


def ts_status_string(s: int) -> str:
    return _status_name(s)


def ts_last_error_detail() -> str:
    return _lib.ts_last_error_detail().decode()
