"""Seeded sweep over shapes and launch options, bit-exact against the oracle.

Each case draws M, N, K (ragged tails in every dimension, K a multiple of 8 so
that rows start on 16-byte boundaries), the output type, tile, scheduler,
epilogue warps, barrier layout, raster group, static worker cap and
dependency mode, and multiplies integer-valued matrices in [-4, 4], whose
products are exact in fp32 and in the oracle's float64.  Every element of D
is compared, and nothing outside D (a sentinel band of the buffer) may change.
A few cases have K >= 4096 and more tiles than fit at once, so that the plan
splits tiles along K.  The scheduler is static persistent, CLC or
non-persistent.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_bit_exact, to_device_bf16

pytestmark = pytest.mark.gpu

SEED = 0x7E57
N_CASES = 48


def _cases():
    rng = np.random.default_rng(SEED)
    out = []
    for i in range(N_CASES):
        big = i % 12 == 11  # a 10 x 10 grid of pair tiles with K >= 4096: the plan splits tiles along K
        if big:
            M, N = (int(x) for x in rng.integers(2305, 2561, 2))
            K = int(rng.choice([4096, 4160, 5120]))
        else:
            M, N = (int(x) for x in rng.integers(1, 2100, 2))
            K = int(8 * rng.integers(1, 257))
        out_t = str(rng.choice(["f32", "bf16"]))
        merge = int(rng.random() < 0.2)
        tile = "256x256" if big else str(rng.choice(["auto", "128x128", "128x256", "256x256"]))
        ew = 0
        if not merge:
            ew = int(rng.choice([0, 4, 8])) if big else int(rng.choice([0, 4, 8, 16]))
            if ew == 16 and tile not in ("128x256", "256x256"):
                tile = str(rng.choice(["128x256", "256x256"]))
        sched = str(rng.choice(["static", "clc", "nonpersistent"]))
        cap = int(rng.choice([0, 0, 1, 7, 100])) if sched == "static" and not big else 0
        raster = int(rng.choice([0, 1, 3, 16]))
        ready = int(rng.random() < 0.5)
        out.append((i, M, N, K, out_t, tile, sched, ew, merge, cap, raster, ready))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: "case%02d_%dx%dx%d_%s_%s_%s_ew%d_mg%d_cap%d_r%d_ready%d" % c)
def test_random_shape_and_options_bit_exact(lib, case):
    i, M, N, K, out_t, tile, sched, ew, merge, cap, raster, ready = case
    A = synth.int_uniform_bf16(SEED + 2 * i, (M, K))
    B = synth.int_uniform_bf16(SEED + 2 * i + 1, (N, K))
    dt = torch.float32 if out_t == "f32" else torch.bfloat16
    # D sits inside a larger buffer whose sentinel band must survive: even cases with a pitch and
    # an offset that allow TMA stores, odd ones with an odd pitch (plain stores)
    if i % 2 == 0:
        pr, pc = 2, 8
        pitch = -(-(N + 2 * pc) // 8) * 8
    else:
        pr, pc = 3, 3
        pitch = N + 2 * pc
    buf = torch.full((M + 2 * pr, pitch), -7.0, dtype=dt, device="cuda")
    D = buf[pr:pr + M, pc:pc + N]
    lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched=sched, tile=tile, epi_warps=ew, merge=merge,
                        max_workers=cap, raster_group=raster, inputs_ready=ready)
    lib.ts_sync_and_check()
    assert_bit_exact(D, oracle.gemm_f64_blas(A, B), f"case {case}")
    band = buf.clone()
    band[pr:pr + M, pc:pc + N] = -7.0
    assert bool((band == -7.0).all()), f"case {case}: a write outside D"


def test_sweep_covers_split_tiles_and_both_modes(lib):
    cases = _cases()
    split = 0
    for i, M, N, K, out_t, tile, sched, ew, merge, cap, raster, ready in cases:
        info = lib.ts_gemm_launch_info(M, N, K, lib.TS_OUT_F32 if out_t == "f32" else lib.TS_OUT_BF16, sched,
                                       tile=tile, epi_warps=ew, merge=merge, max_workers=cap)
        split += info["split_tiles"] > 0
    assert split >= 1
    assert {c[11] for c in cases} == {0, 1} and {c[6] for c in cases} == {"static", "clc", "nonpersistent"}


def _grouped_cases():
    rng = np.random.default_rng(SEED + 1)
    out = []
    for i in range(24):
        G = int(rng.integers(1, 17))
        widths = [int(64 * rng.choice([0, 1, 2, 5, 16, 40])) for _ in range(G)]
        base = int(64 * rng.integers(0, 3))
        off = [base + int(x) for x in np.concatenate([[0], np.cumsum(widths)])]
        M, N = (int(x) for x in rng.integers(1, 1200, 2))
        out_t = str(rng.choice(["f32", "bf16"]))
        tile = str(rng.choice(["auto", "128x128", "128x256", "256x256"]))
        merge = int(rng.random() < 0.2)
        ew = 0 if merge else int(rng.choice([0, 4, 8]))
        sched = str(rng.choice(["static", "clc", "nonpersistent"]))
        ready = int(rng.random() < 0.5)
        out.append((i, tuple(off), M, N, out_t, tile, sched, ew, merge, ready))
    return out


@pytest.mark.parametrize("case", _grouped_cases(), ids=lambda c: "grouped%02d_g%d_%dx%d_%s_%s_%s_ew%d_mg%d_ready%d" % (
    c[0], len(c[1]) - 1, c[2], c[3], c[4], c[5], c[6], c[7], c[8], c[9]))
def test_random_grouped_bit_exact(lib, case):
    # groups of 0 to 2560 columns (empty groups included), offsets not starting at 0
    i, off, M, N, out_t, tile, sched, ew, merge, ready = case
    Kt = max(off[-1], 8)
    A = synth.int_uniform_bf16(SEED + 100 + 2 * i, (M, Kt))
    B = synth.int_uniform_bf16(SEED + 101 + 2 * i, (N, Kt))
    dt = torch.float32 if out_t == "f32" else torch.bfloat16
    G = len(off) - 1
    D = torch.full((G, M, N), float("nan"), dtype=dt, device="cuda")
    lib.ts_gemm_bf16_grouped(to_device_bf16(A), to_device_bf16(B), D, list(off), sched=sched, tile=tile, epi_warps=ew,
                             merge=merge, inputs_ready=ready)
    lib.ts_sync_and_check()
    ref = oracle.grouped_gemm_f64(A, B, list(off), blas=True)
    for g in range(G):
        assert_bit_exact(D[g], ref[g], f"case {case} group {g}")
