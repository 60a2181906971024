"""CPU oracle for the tile-scheduled GEMM, the int16 copy and the jagged row copy.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline leg, never by the product path.  It shares no code
with the CUDA library.  The arithmetic lives in ``oracle.c`` (compiled with
gcc on first use); this module only marshals numpy arrays.

Functions and the passages they follow:

* ``gemm_f64``: D[i, j] = sum_k a[i, k] * b[j, k] in float64 over the bf16
  inputs, by the plain (i, j, k) loop -- the GEMM mainloop of CUTLASS TS
  "Pipeline Groups" (Overview, the Merge example gmem_ab -> smem_a/smem_b ->
  tmem_c -> gmem_d) together with the per-tile scale_d reset of TS
  "Resources" (first MMA overwrites, later MMAs accumulate).
* ``gemm_f64_blas``: the same sum with numpy's float64 matmul as the
  contraction step, for sizes the loop cannot finish in seconds.
* ``bf16_rne``: float64 -> bf16 round-to-nearest-even (IEEE 754), the
  conversion the bf16-output epilogue applies to the fp32 accumulator.
* ``grouped_gemm_f64``: the same sum per group over that group's K slice
  (TS "Schedules", Dynamic Domain: a per-tile loop bound from an offsets array).
* ``row_sums_f64``: per-row sums of A over each group's K range, the second
  output of the Fork pipeline group (TS "Pipeline Groups", Fork).
* ``copy_i16``: dst[gid] = src[gid] for gid < n (TS "Resources", the int16
  copy example; TS "Schedules", the grid-stride domain).
* ``copy_rows_i16``: the jagged row copy -- for every row r below the row
  count that the skip mask does not drop, dst[i] = src[i] for offsets[r] <= i
  < offsets[r + 1]; every other element keeps its value (TS "Schedules",
  Dynamic Domain: a per-tile loop bound from an offsets array; Skippable
  Tiles: the oversubscribed copy whose skipped tiles copy nothing).
* ``static_schedule`` / ``static_owner``: worker w takes tiles w, w+W, ...
  ("Cluster Launch Control", limits of the static persistent scheduler,
  worked example of 12 tiles on 4 workers).
* ``clc_coverage_ok``: the Cluster Launch Control invariant -- every
  coordinate is processed exactly once, and a worker that runs starts with
  the tile of its own block index.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so with gcc (OpenMP on)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f64_to_bf16_rne.restype = ctypes.c_uint16
            lib.oracle_f64_to_bf16_rne.argtypes = [ctypes.c_double]
            lib.oracle_bf16_decode.argtypes = [P, P, I64]
            lib.oracle_bf16_encode.argtypes = [P, P, I64]
            lib.oracle_gemm_f64.argtypes = [P, P, P, I64, I64, I64, I64, I64, I64, I64, I64,
                                            ctypes.c_int, ctypes.c_int]
            lib.oracle_gemm_entries_f64.argtypes = [P, P, I64, I64, I64, P, P, I64, P, P, ctypes.c_int]
            lib.oracle_copy_i16.argtypes = [P, P, I64]
            lib.oracle_copy_rows_i16.argtypes = [P, P, I64, P, I64, P]
            lib.oracle_copy_rows_i16.restype = I64
            lib.oracle_static_owner.argtypes = [I64, I64, P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _bits(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.int16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns (uint16), got {x.dtype}")
    return np.ascontiguousarray(x)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


# ---------------------------------------------------------------- bf16 codec
def bf16_to_f64(bits) -> np.ndarray:
    b = _bits(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_bf16_decode(_ptr(b), _ptr(out), b.size)
    return out


def bf16_rne(x) -> np.ndarray:
    """float64 -> bf16 bit patterns, round to nearest, ties to even."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_bf16_encode(_ptr(x), _ptr(out), x.size)
    return out


def bf16_rne_scalar(x: float) -> int:
    return int(_load().oracle_f64_to_bf16_rne(float(x)))


# ---------------------------------------------------------------------- GEMM
def gemm_f64(A_bits, B_bits, rows=None, absolute: bool = False, threads: int | None = None) -> np.ndarray:
    """Triple-loop float64 GEMM D = A . B^T over bf16 A[M, K], B[N, K].

    ``rows`` = (row0, row1) restricts the output to those rows of D.
    ``absolute`` computes sum_k |a||b| (the scale of the error bound)."""
    A = _bits(A_bits)
    B = _bits(B_bits)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("A and B disagree on K")
    r0, r1 = (0, M) if rows is None else rows
    D = np.empty((r1 - r0, N), dtype=np.float64)
    _load().oracle_gemm_f64(_ptr(A), _ptr(B), _ptr(D), M, N, K, K, K, N, r0, r1, int(absolute),
                            threads or default_threads())
    return D


def gemm_entries_f64(A_bits, B_bits, ii, jj, threads: int | None = None):
    """(D[ii[t], jj[t]], sum_k |a||b|) for individual entries, by the same loop."""
    A = _bits(A_bits)
    B = _bits(B_bits)
    K = A.shape[1]
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    out = np.empty(ii.size, dtype=np.float64)
    out_abs = np.empty(ii.size, dtype=np.float64)
    _load().oracle_gemm_entries_f64(_ptr(A), _ptr(B), K, K, K, _ptr(ii), _ptr(jj), ii.size,
                                    _ptr(out), _ptr(out_abs), threads or default_threads())
    return out, out_abs


def gemm_f64_blas(A_bits, B_bits, absolute: bool = False) -> np.ndarray:
    """D = a . b^T in float64, numpy matmul as the contraction step."""
    a = bf16_to_f64(A_bits)
    b = bf16_to_f64(B_bits)
    if absolute:
        np.abs(a, out=a)
        np.abs(b, out=b)
    return a @ b.T


def grouped_gemm_f64(A_bits, B_bits, k_offsets, absolute: bool = False, blas: bool = False) -> np.ndarray:
    """Grouped GEMM over K slices: D[g] = sum over k_offsets[g] <= k < k_offsets[g+1] of a[:, k] b[:, k]^T.

    The per-group K range is the dynamic domain of TS "Schedules" (Dynamic
    Domain: the loop bound comes from an offsets array).  Each group is the
    plain triple loop (or numpy's matmul with ``blas``) on its column slice;
    an empty group is all zeros."""
    A = _bits(A_bits)
    B = _bits(B_bits)
    off = [int(x) for x in k_offsets]
    G = len(off) - 1
    D = np.zeros((G, A.shape[0], B.shape[0]), dtype=np.float64)
    for g in range(G):
        k0, k1 = off[g], off[g + 1]
        if k1 > k0:
            a = np.ascontiguousarray(A[:, k0:k1])
            b = np.ascontiguousarray(B[:, k0:k1])
            D[g] = gemm_f64_blas(a, b, absolute) if blas else gemm_f64(a, b, absolute=absolute)
    return D


def row_sums_f64(A_bits, k_offsets) -> np.ndarray:
    """R[g][i] = sum over k_offsets[g] <= k < k_offsets[g+1] of a[i, k], by a plain loop.

    The second output of the Fork pipeline group (TS "Pipeline Groups", Fork):
    a second consumer reads the same A stages as the MMA."""
    A = _bits(A_bits)
    off = [int(x) for x in k_offsets]
    a = bf16_to_f64(A)
    R = np.zeros((len(off) - 1, A.shape[0]), dtype=np.float64)
    for g in range(len(off) - 1):
        for k in range(off[g], off[g + 1]):
            R[g] += a[:, k]
    return R


# ---------------------------------------------------------------------- copy
def copy_i16(src) -> np.ndarray:
    s = np.ascontiguousarray(np.asarray(src, dtype=np.int16))
    d = np.empty_like(s)
    _load().oracle_copy_i16(_ptr(s), _ptr(d), s.size)
    return d


def copy_rows_i16(src, dst, offsets, rows: int | None = None, skip=None) -> tuple[np.ndarray, int]:
    """The jagged row copy applied to a copy of ``dst``; returns (result, first invalid row or -1)."""
    s = np.ascontiguousarray(np.asarray(src, dtype=np.int16))
    d = np.array(dst, dtype=np.int16, copy=True)
    if d.shape != s.shape:
        raise ValueError("src and dst differ in size")
    off = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    if rows is None:
        rows = max(off.size - 1, 0)
    if off.size < rows + 1:
        raise ValueError("offsets needs rows + 1 entries")
    sk = None
    if skip is not None:
        sk = np.ascontiguousarray(np.asarray(skip, dtype=np.uint8))
        if sk.size < rows:
            raise ValueError("skip needs one entry per row")
    bad = _load().oracle_copy_rows_i16(_ptr(s), _ptr(d), s.size, _ptr(off), int(rows),
                                       _ptr(sk) if sk is not None else None)
    return d, int(bad)


# ---------------------------------------------------------------- scheduling
def static_owner(num_tiles: int, num_workers: int) -> np.ndarray:
    owner = np.full(num_tiles, -1, dtype=np.int64)
    _load().oracle_static_owner(num_tiles, num_workers, _ptr(owner))
    return owner


def static_schedule(num_tiles: int, num_workers: int) -> list[list[int]]:
    """Per worker, the tiles it takes under the grid-stride rule, in order."""
    owner = static_owner(num_tiles, num_workers)
    return [[int(t) for t in np.nonzero(owner == w)[0]] for w in range(num_workers)]


def clc_coverage_ok(visits: np.ndarray, owner: np.ndarray) -> tuple[bool, str]:
    """Every tile visited exactly once; each worker that ran owns the tile of its own index."""
    visits = np.asarray(visits)
    owner = np.asarray(owner)
    if visits.size and not np.all(visits == 1):
        bad = np.nonzero(visits != 1)[0]
        return False, f"{bad.size} tiles not visited exactly once (first {bad[:8].tolist()})"
    ran = np.unique(owner)
    if ran.size and (ran.min() < 0 or ran.max() >= owner.size):
        return False, "owner index out of range"
    if not np.all(owner[ran] == ran):
        bad = ran[owner[ran] != ran]
        return False, f"workers {bad[:8].tolist()} did not start on their own tile"
    return True, "ok"
