"""Seeded synthetic inputs shared by the CUDA path's tests/bench and by the oracle.

This module only draws random numbers and rounds them to the input storage
format (bf16 bit patterns, int16).  It holds none of the GEMM or copy
arithmetic, so both sides can consume the same bits without sharing any code
that decides a result.

Generator: SplitMix64 in counter form, z_i = mix(seed + (i + 1) * 0x9E3779B97F4A7C15),
with the published finaliser (Steele, Lea, Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014).  Values:

* uniform in [-1, 1):  u = ((z >> 40) - 2**23) / 2**23  (24-bit, exact in fp32)
* standard normal:     Box-Muller on two 53-bit uniforms, then scaled
* small integers:      lo + (z mod (hi - lo + 1))
* int16:               the low 16 bits of z

The draws are made by synth.c (compiled with gcc on first use); splitmix64()
here is the same generator in numpy, kept as the readable reference form.
Rounding to bf16 uses torch's float32 -> bfloat16 conversion (round to
nearest even); the normal draws go float64 -> float32 -> bfloat16.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 23

# seeds of the five workloads (A uses base + index, B adds 0x100)
SEED_BASE = 0x74530000


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """n SplitMix64 outputs for counters offset+1 .. offset+n (uint64 array), numpy reference form."""
    out = np.empty(n, dtype=np.uint64)
    s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        for c0 in range(0, n, _CHUNK):
            c1 = min(n, c0 + _CHUNK)
            ctr = np.arange(offset + c0 + 1, offset + c1 + 1, dtype=np.uint64)
            z = s + ctr * _GOLDEN
            z = (z ^ (z >> np.uint64(30))) * _M1
            z = (z ^ (z >> np.uint64(27))) * _M2
            out[c0:c1] = z ^ (z >> np.uint64(31))
    return out


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


# ------------------------------------------------------------ C generator
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile synth.c (gcc, OpenMP) into synth/_build/libsynth.so."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"],
                   check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _c():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I64, U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
            lib.synth_splitmix64.argtypes = [U64, I64, I64, P]
            lib.synth_uniform_pm1_f32.argtypes = [U64, I64, P]
            lib.synth_normal_f32.argtypes = [U64, I64, ctypes.c_double, P]
            lib.synth_int_uniform_f32.argtypes = [U64, I64, ctypes.c_int32, ctypes.c_int32, P]
            lib.synth_int16.argtypes = [U64, I64, P]
            _lib = lib
    return _lib


def _seed(seed: int) -> int:
    return seed & 0xFFFFFFFFFFFFFFFF


def splitmix64_fast(seed: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _c().synth_splitmix64(_seed(seed), offset, n, out.ctypes.data)
    return out


def uniform_pm1_bf16(seed: int, shape) -> np.ndarray:
    """bf16 bit patterns of uniform draws in [-1, 1), row-major ``shape``."""
    n = int(np.prod(shape))
    f = np.empty(n, dtype=np.float32)
    _c().synth_uniform_pm1_f32(_seed(seed), n, f.ctypes.data)
    return _f32_to_bf16_bits(f).reshape(shape)


def normal_bf16(seed: int, shape, scale: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of N(0, 1) * scale draws (Box-Muller, cosine branch)."""
    n = int(np.prod(shape))
    f = np.empty(n, dtype=np.float32)
    _c().synth_normal_f32(_seed(seed), n, float(scale), f.ctypes.data)
    return _f32_to_bf16_bits(f).reshape(shape)


def int_uniform_bf16(seed: int, shape, lo: int = -4, hi: int = 4) -> np.ndarray:
    """bf16 bit patterns of integers uniform in [lo, hi] (exact in bf16 for |v| <= 256)."""
    n = int(np.prod(shape))
    f = np.empty(n, dtype=np.float32)
    _c().synth_int_uniform_f32(_seed(seed), n, lo, hi, f.ctypes.data)
    return _f32_to_bf16_bits(f).reshape(shape)


def int16_uniform(seed: int, n: int) -> np.ndarray:
    """n int16 values from the low 16 bits of the generator."""
    out = np.empty(n, dtype=np.int16)
    _c().synth_int16(_seed(seed), n, out.ctypes.data)
    return out


def one_hot_rows_bf16(n_rows: int, n_cols: int, cols: np.ndarray) -> np.ndarray:
    """Rows with a single 1.0 at column cols[r] (bf16 bits; 0x3F80 is 1.0)."""
    out = np.zeros((n_rows, n_cols), dtype=np.uint16)
    out[np.arange(n_rows), cols] = 0x3F80
    return out


@dataclass(frozen=True)
class GemmWorkload:
    name: str
    M: int
    N: int
    K: int
    out: str  # "bf16" or "f32"
    dist: str  # "uniform" or "normal"
    tile: str  # "128x128", "128x256", "256x256"
    sched: tuple  # schedulers exercised
    seed_a: int
    seed_b: int

    def inputs(self):
        if self.dist == "normal":
            s = 1.0 / math.sqrt(self.K)
            return normal_bf16(self.seed_a, (self.M, self.K), s), normal_bf16(self.seed_b, (self.N, self.K), s)
        return uniform_pm1_bf16(self.seed_a, (self.M, self.K)), uniform_pm1_bf16(self.seed_b, (self.N, self.K))


def _w(i, name, M, N, K, out, dist, tile, sched):
    return GemmWorkload(name, M, N, K, out, dist, tile, sched, SEED_BASE + i, SEED_BASE + i + 0x100)


# The GEMM workloads (indices follow the workload list; index 1 is the copy).
GEMM_256 = _w(0, "gemm 256x256x256 fp32-out 128x128 static", 256, 256, 256, "f32", "uniform", "128x128", ("static",))
GEMM_4096 = _w(2, "gemm 4096x4096x4096 bf16-out 128x256 static/clc", 4096, 4096, 4096, "bf16", "uniform", "128x256",
               ("static", "clc"))
GEMM_8192 = _w(3, "gemm 8192x8192x8192 bf16-out 2-CTA 256x256 clc", 8192, 8192, 8192, "bf16", "normal", "256x256",
               ("clc",))
GEMM_RAGGED = _w(4, "gemm 8191x6143x4096 fp32-out ragged contended", 8191, 6143, 4096, "f32", "uniform", "128x256",
                 ("static", "clc"))
# K = 64 is one k-block per tile: the 134 MB bf16 output dominates the traffic (HBM-bound GEMM).
GEMM_SMALLK = _w(10, "gemm 8192x8192x64 bf16-out small-K (output-write bound)", 8192, 8192, 64, "bf16", "uniform",
                 "256x256", ("static", "clc"))
COPY_N = 1 << 28
COPY_SEED = SEED_BASE + 1


@dataclass(frozen=True)
class GroupedWorkload:
    """A grouped GEMM whose groups differ in K (e.g. per-expert weight gradients)."""

    name: str
    M: int
    N: int
    groups: int
    seed: int

    def k_offsets(self) -> list:
        # group sizes in 64-column blocks: 1 + floor(127 u^2) -- skewed towards small groups
        z = splitmix64(self.seed, self.groups)
        u = (z >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        blocks = 1 + np.floor(127.0 * u * u).astype(np.int64)
        return [0] + [int(x) for x in np.cumsum(blocks * 64)]

    def inputs(self):
        K = self.k_offsets()[-1]
        return (uniform_pm1_bf16(self.seed + 1, (self.M, K)), uniform_pm1_bf16(self.seed + 2, (self.N, K)))


GROUPED = GroupedWorkload("grouped gemm 16 groups 2048x2048, K per group 64..8192 (skewed)", 2048, 2048, 16,
                          SEED_BASE + 5)


@dataclass(frozen=True)
class RowsWorkload:
    """A jagged int16 array whose row lengths span several decades (log-uniform)."""

    name: str
    rows: int
    min_len: int
    max_len: int
    seed: int

    def offsets(self) -> np.ndarray:
        # length = floor(min_len * (max_len / min_len) ** u), u uniform in [0, 1), in generator order
        z = splitmix64(self.seed, self.rows)
        u = (z >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        lengths = np.floor(self.min_len * (self.max_len / self.min_len) ** u).astype(np.int64)
        return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)

    def inputs(self):
        off = self.offsets()
        return int16_uniform(self.seed + 1, int(off[-1])), off


ROWS = RowsWorkload("jagged int16 copy, 8192 rows of 64..262144 elements (log-uniform)", 8192, 64, 262144,
                    SEED_BASE + 8)
