"""GPU parity of ts_gemm_bf16 against the CPU oracle (called through the C ABI).

Random inputs must satisfy the error bound in tests/parity.py; integer-valued,
identity and one-hot inputs must match bit for bit.  Sizes small enough for the
triple-loop oracle span several tiles and a ragged tail; the full-size
workloads are checked against the oracle's BLAS route (whole output) or on
sampled rows.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import as_f64, assert_bit_exact, assert_within_bound, bf16_bits, tile_layouts, to_device_bf16

pytestmark = pytest.mark.gpu

TILES = ["128x128", "128x256", "256x256"]
SCHEDS = ["static", "clc"]
OUTS = [torch.float32, torch.bfloat16]


def _run(ts, A_bits, B_bits, out, **kw):
    A = to_device_bf16(A_bits)
    B = to_device_bf16(B_bits)
    D = torch.full((A.shape[0], B.shape[0]), float("nan"), dtype=out, device="cuda")
    ts.ts_gemm_bf16_ex(A, B, D, **kw)
    ts.ts_sync_and_check()
    return D


# -------------------------------------------------------------- workload 0
def test_gemm_256_fp32_static_128x128(lib):
    w = synth.GEMM_256
    A, B = w.inputs()
    info = lib.ts_gemm_launch_info(w.M, w.N, w.K, lib.TS_OUT_F32, "static", tile="128x128")
    assert info["num_tiles"] == 4 and info["workers"] == 4 and info["grid_ctas"] == 4
    D = _run(lib, A, B, torch.float32, sched="static", tile="128x128")
    ref = oracle.gemm_f64(A, B)
    S = oracle.gemm_f64(A, B, absolute=True)
    assert_within_bound(as_f64(D), ref, S, torch.float32, "256^3")


# ------------------------------------------------------ exact-value cases
@pytest.mark.parametrize("tile,ew,merge", tile_layouts(TILES))
@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("out", OUTS)
def test_gemm_integer_bit_exact(lib, tile, sched, out, ew, merge):
    M, N, K = 600, 520, 328  # ragged in M, N and K
    A = synth.int_uniform_bf16(101, (M, K))
    B = synth.int_uniform_bf16(102, (N, K))
    D = _run(lib, A, B, out, sched=sched, tile=tile, epi_warps=ew, merge=merge)
    assert_bit_exact(D, oracle.gemm_f64(A, B), f"integer {tile} {sched} {ew} epilogue warps, merge {merge}")


def test_gemm_epilogue_warps_automatic_choice(lib):
    # sixteen epilogue warps for the shortest K loops on 256-column tiles, eight
    # for short ones, four for a long one; a grouped GEMM by its longest group
    for K, ew in ((64, 16), (128, 16), (192, 8), (256, 8)):
        assert lib.ts_gemm_launch_info(4096, 4096, K, lib.TS_OUT_BF16, "clc")["epi_warps"] == ew
        assert lib.ts_gemm_launch_info(4096, 4096, K, lib.TS_OUT_BF16, "static", tile="128x256")["epi_warps"] == ew
    assert lib.ts_gemm_launch_info(4096, 4096, 64, lib.TS_OUT_BF16, "clc", tile="128x128")["epi_warps"] == 8
    with pytest.raises(lib.TsError):
        lib.ts_gemm_launch_info(4096, 4096, 64, lib.TS_OUT_BF16, "clc", tile="128x128", epi_warps=16)
    assert lib.ts_gemm_launch_info(4096, 4096, 320, lib.TS_OUT_BF16, "clc")["epi_warps"] == 4
    assert lib.ts_gemm_launch_info(4096, 4096, 64, lib.TS_OUT_BF16, "clc", epi_warps=4)["epi_warps"] == 4
    assert lib.ts_gemm_grouped_launch_info(512, 512, [0, 64, 128])["epi_warps"] == 8  # 128 x 128 tiles
    for widths, ew in (([64] * 16, 16), ([128, 64] * 8, 16), ([256, 0] * 8, 8), ([64] * 15 + [320], 4)):
        off = [0] + list(np.cumsum(widths))
        info = lib.ts_gemm_grouped_launch_info(2048, 2048, off, lib.TS_OUT_BF16, "clc")
        assert info["cluster"] == 2 and info["epi_warps"] == ew, (widths[:2], info["epi_warps"])
    # the Merge layout is built with four
    info = lib.ts_gemm_launch_info(4096, 4096, 64, lib.TS_OUT_BF16, "clc", merge=1)
    assert info["epi_warps"] == 4 and info["merge"] == 1
    with pytest.raises(lib.TsError):
        lib.ts_gemm_launch_info(4096, 4096, 64, lib.TS_OUT_BF16, "clc", epi_warps=2)


@pytest.mark.parametrize("G", [1, 2, 3, 5, 8, 16, 64])
@pytest.mark.parametrize("tile,sched", [("128x128", "clc"), ("128x256", "static"), ("256x256", "clc"),
                                        ("256x256", "static")])
def test_gemm_raster_groups_cover_every_tile(lib, G, tile, sched):
    # tile rows not a multiple of the raster group, so the last group is shorter;
    # every tile id must land on a distinct tile (NaN-filled D shows a missed one)
    M, N, K = 1100, 1300, 128
    A = synth.int_uniform_bf16(141 + G, (M, K))
    B = synth.int_uniform_bf16(241 + G, (N, K))
    D = _run(lib, A, B, torch.float32, sched=sched, tile=tile, raster_group=G)
    assert_bit_exact(D, oracle.gemm_f64(A, B), f"raster group {G} {tile} {sched}")


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("sched", SCHEDS)
def test_gemm_one_hot_selects_columns(lib, tile, sched):
    M, N, K = 300, 270, 200
    rng = np.random.default_rng(3)
    cols = rng.integers(0, K, size=N)
    A = synth.uniform_pm1_bf16(111, (M, K))
    B = synth.one_hot_rows_bf16(N, K, cols)
    D = _run(lib, A, B, torch.bfloat16, sched=sched, tile=tile)
    assert np.array_equal(bf16_bits(D), A[:, cols])


@pytest.mark.parametrize("tile", TILES)
def test_gemm_identity_returns_a(lib, tile):
    M, K = 257, 192
    A = synth.uniform_pm1_bf16(121, (M, K))
    B = synth.one_hot_rows_bf16(K, K, np.arange(K))
    D = _run(lib, A, B, torch.float32, sched="static", tile=tile)
    assert np.array_equal(as_f64(D), oracle.bf16_to_f64(A))


# Extreme aspect ratios: a K loop of 1024 k-blocks (every ring barrier wraps
# its phase over a hundred times inside one tile), a single tile row 2048
# tiles wide, and a single tile column 8193 tiles tall whose D pitch (3
# elements) rules out TMA stores.  Integer entries keep every partial sum exact.
@functools.lru_cache(maxsize=None)
def _aspect_case(M, N, K):
    A = synth.int_uniform_bf16(141, (M, K))
    B = synth.int_uniform_bf16(142, (N, K))
    return A, B, oracle.gemm_f64(A, B)


@pytest.mark.parametrize("M,N,K", [(2, 300, 1 << 16), (1, 1 << 18, 64), ((1 << 20) + 7, 3, 64)])
@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("sched", SCHEDS)
def test_gemm_extreme_aspect_integer(lib, M, N, K, tile, sched):
    A, B, ref = _aspect_case(M, N, K)
    for out in OUTS:
        D = _run(lib, A, B, out, sched=sched, tile=tile)
        assert_bit_exact(D, ref, f"{M}x{N}x{K} {tile} {sched} {out}")


# Host buffers: the copies in, the GEMM and the copy out in one call.
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("M,N,K", [(600, 520, 328), (1, 300, 64), (257, 1, 72), (300, 260, 0)])
@pytest.mark.parametrize("out", OUTS)
def test_gemm_host_buffers_integer_exact(lib, pinned, M, N, K, out):
    A_bits = synth.int_uniform_bf16(151, (M, K))
    B_bits = synth.int_uniform_bf16(152, (N, K))
    A_h = torch.from_numpy(A_bits.view(np.int16)).view(torch.bfloat16)
    B_h = torch.from_numpy(B_bits.view(np.int16)).view(torch.bfloat16)
    D_h = torch.full((M, N), float("nan"), dtype=out)
    if pinned:
        A_h, B_h, D_h = A_h.pin_memory(), B_h.pin_memory(), D_h.pin_memory()
    A = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    D = torch.empty((M, N), dtype=out, device="cuda")
    lib.ts_gemm_bf16_host(A_h, B_h, D_h, A, B, D, sched="clc")
    torch.cuda.synchronize()
    lib.ts_sync_and_check()
    assert_bit_exact(D_h, oracle.gemm_f64(A_bits, B_bits), f"host buffers {M}x{N}x{K} {out} pinned={pinned}")


def test_gemm_host_buffers_checks_before_copying(lib):
    A_h = torch.ones((64, 64), dtype=torch.bfloat16)
    B_h = torch.ones((64, 64), dtype=torch.bfloat16)
    D_h = torch.full((64, 64), 7.0, dtype=torch.float32)
    A = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(lib.TsError):
        lib.ts_gemm_bf16_host(A_h, B_h, D_h, A, B, D, tile="128x128", epi_warps=16)  # no such variant
    torch.cuda.synchronize()
    assert torch.count_nonzero(A) == 0 and torch.all(D_h == 7.0)  # nothing was copied either way


# ---------------------------------------------------------- random inputs
@pytest.mark.parametrize("M,N,K", [(1, 1, 8), (127, 129, 64), (129, 127, 72), (255, 255, 200), (1, 255, 8),
                                   (255, 1, 136), (384, 640, 1024)])
@pytest.mark.parametrize("tile", TILES)
def test_gemm_small_odd_shapes(lib, M, N, K, tile):
    A = synth.uniform_pm1_bf16(131 + M, (M, K))
    B = synth.uniform_pm1_bf16(231 + N, (N, K))
    ref = oracle.gemm_f64(A, B)
    S = oracle.gemm_f64(A, B, absolute=True)
    for sched in SCHEDS:
        for out in OUTS:
            D = _run(lib, A, B, out, sched=sched, tile=tile)
            assert_within_bound(as_f64(D), ref, S, out, f"{M}x{N}x{K} {tile} {sched} {out}")


@pytest.mark.parametrize("tile", TILES)
def test_gemm_strided_operands(lib, tile):
    M, N, K = 300, 200, 136
    Af = synth.uniform_pm1_bf16(141, (M, K + 24))
    Bf = synth.uniform_pm1_bf16(142, (N, K + 40))
    A = to_device_bf16(Af)[:, :K]
    B = to_device_bf16(Bf)[:, :K]
    Dfull = torch.zeros((M, N + 8), dtype=torch.float32, device="cuda")
    D = Dfull[:, :N]
    lib.ts_gemm_bf16_ex(A, B, D, sched="clc", tile=tile)
    lib.ts_sync_and_check()
    ref = oracle.gemm_f64(np.ascontiguousarray(Af[:, :K]), np.ascontiguousarray(Bf[:, :K]))
    S = oracle.gemm_f64(np.ascontiguousarray(Af[:, :K]), np.ascontiguousarray(Bf[:, :K]), absolute=True)
    assert_within_bound(as_f64(D), ref, S, torch.float32, "strided")
    assert torch.all(Dfull[:, N:] == 0)


@pytest.mark.parametrize("out", OUTS)
@pytest.mark.parametrize("tile", TILES)
def test_gemm_guard_regions_untouched(lib, out, tile):
    # D lives inside a larger buffer; rows/columns around it hold a sentinel
    # N = 301: the right edge is ragged at 16-byte granularity for both dtypes.
    # pitch N + 64 + pad: pad 0 -> 365 (unaligned, plain-store epilogue);
    # pad 3 -> 368 and pad 11 -> 376 (16-byte pitch, TMA stores + ragged edge)
    M, N, K = 200, 301, 64
    A = synth.int_uniform_bf16(151, (M, K))
    B = synth.int_uniform_bf16(152, (N, K))
    for pitch_pad in (0, 3, 11):
        big = torch.full((M + 64, N + 64 + pitch_pad), 3072.0, dtype=out, device="cuda")
        D = big[32:32 + M, 32:32 + N]
        lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched="static", tile=tile)
        lib.ts_sync_and_check()
        assert_bit_exact(D, oracle.gemm_f64(A, B), f"guard pad={pitch_pad}")
        mask = torch.ones_like(big, dtype=torch.bool)
        mask[32:32 + M, 32:32 + N] = False
        assert torch.all(big[mask] == 3072.0), f"write outside D (pad={pitch_pad})"


def test_gemm_unaligned_pitch_fp32_contiguous(lib):
    # fp32 with N = 6143-like odd width: pitch not a multiple of 16 bytes
    M, N, K = 130, 131, 64
    info = lib.ts_gemm_launch_info(M, N, K, lib.TS_OUT_F32, "static", tile="128x256")
    assert info["tma_store"] == 0
    A = synth.uniform_pm1_bf16(161, (M, K))
    B = synth.uniform_pm1_bf16(162, (N, K))
    D = _run(lib, A, B, torch.float32, sched="clc", tile="128x256")
    assert_within_bound(as_f64(D), oracle.gemm_f64(A, B), oracle.gemm_f64(A, B, absolute=True), torch.float32,
                        "odd pitch")


# ----------------------------------------------------------- edge cases
def test_gemm_k_zero_fills_zero(lib):
    A = torch.empty((0,), dtype=torch.bfloat16, device="cuda")
    for out in OUTS:
        D = torch.full((70, 90), 7.0, dtype=out, device="cuda")
        st = lib.ts_gemm_bf16_ptr(A.data_ptr(), A.data_ptr(), D.data_ptr(), 70, 90, 0,
                                  lib.TS_OUT_F32 if out == torch.float32 else lib.TS_OUT_BF16)
        assert st == lib.TS_OK
        lib.ts_sync_and_check()
        assert torch.all(D == 0)


def test_gemm_empty_m_or_n_is_noop(lib):
    D = torch.full((4, 4), 3.0, device="cuda")
    assert lib.ts_gemm_bf16_ptr(0, 0, D.data_ptr(), 0, 4, 64, lib.TS_OUT_F32) == lib.TS_OK
    assert lib.ts_gemm_bf16_ptr(0, 0, D.data_ptr(), 4, 0, 64, lib.TS_OUT_F32) == lib.TS_OK
    lib.ts_sync_and_check()
    assert torch.all(D == 3.0)


def test_gemm_rejects_unaligned_rows(lib):
    A = torch.zeros((64, 12), dtype=torch.bfloat16, device="cuda")  # 24-byte rows
    B = torch.zeros((64, 12), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((64, 64), device="cuda")
    with pytest.raises(lib.TsError) as e:
        lib.ts_gemm_bf16(A, B, D)
    assert e.value.status == lib.TS_ERR_UNSUPPORTED


def test_gemm_rejects_overlap(lib):
    buf = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    st = lib.ts_gemm_bf16_ptr(buf.data_ptr(), buf.data_ptr(), buf.data_ptr() + 512, 64, 64, 64, lib.TS_OUT_BF16)
    assert st == lib.TS_ERR_INVALID_ARG


# ----------------------------------------------------- full-size workloads
@pytest.mark.slow
@pytest.mark.parametrize("sched", SCHEDS)
def test_gemm_4096_bf16_128x256(lib, sched):
    w = synth.GEMM_4096
    A, B = w.inputs()
    D = _run(lib, A, B, torch.bfloat16, sched=sched, tile="128x256")
    ref = oracle.gemm_f64_blas(A, B)
    S = oracle.gemm_f64_blas(A, B, absolute=True)
    assert_within_bound(as_f64(D), ref, S, torch.bfloat16, f"4096^3 {sched}")


@pytest.mark.slow
@pytest.mark.parametrize("merge", [0, 1])
def test_gemm_8192_bf16_2cta_clc_sampled_rows(lib, merge):
    w = synth.GEMM_8192
    A, B = w.inputs()
    D = _run(lib, A, B, torch.bfloat16, sched="clc", tile="256x256", merge=merge)
    rng = np.random.default_rng(8192)
    rows = np.unique(np.concatenate([rng.integers(0, w.M, 96), [0, 255, 256, w.M - 1]]))
    ref = oracle.gemm_f64_blas(A[rows], B)
    S = oracle.gemm_f64_blas(A[rows], B, absolute=True)
    got = oracle.bf16_to_f64(bf16_bits(D[torch.as_tensor(rows, device="cuda")]))
    assert_within_bound(got, ref, S, torch.bfloat16, "8192^3 sampled rows")
    # every tile column/row block is exercised by the sampled rows' full width; add sampled columns too
    cols = rng.integers(0, w.N, 64)
    ii = rng.integers(0, w.M, 64)
    e, ea = oracle.gemm_entries_f64(A, B, ii, cols)
    got2 = oracle.bf16_to_f64(bf16_bits(D[torch.as_tensor(ii, device="cuda"), torch.as_tensor(cols, device="cuda")]))
    assert_within_bound(got2, e, ea, torch.bfloat16, "8192^3 sampled entries")


@pytest.mark.slow
@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("tile", ["128x256", "256x256"])
@pytest.mark.parametrize("ew", [4, 8, 16])
def test_gemm_small_k_sampled(lib, sched, tile, ew):
    # 8192x8192x64: one k-block per tile, the output-write-bound launch the bench times
    w = synth.GEMM_SMALLK
    A, B = w.inputs()
    D = _run(lib, A, B, torch.bfloat16, sched=sched, tile=tile, epi_warps=ew)
    rng = np.random.default_rng(64)
    rows = np.unique(np.concatenate([rng.integers(0, w.M, 128), [0, 127, 128, 255, 256, w.M - 1]]))
    assert_within_bound(oracle.bf16_to_f64(bf16_bits(D[torch.as_tensor(rows, device="cuda")])),
                        oracle.gemm_f64_blas(A[rows], B), oracle.gemm_f64_blas(A[rows], B, absolute=True),
                        torch.bfloat16, f"8192x8192x64 {sched} {tile} sampled rows")
    ii = rng.integers(0, w.M, 256)
    jj = rng.integers(0, w.N, 256)
    e, ea = oracle.gemm_entries_f64(A, B, ii, jj)
    got = oracle.bf16_to_f64(bf16_bits(D[torch.as_tensor(ii, device="cuda"), torch.as_tensor(jj, device="cuda")]))
    assert_within_bound(got, e, ea, torch.bfloat16, f"8192x8192x64 {sched} {tile} sampled entries")
    assert not torch.isnan(D).any()  # every output tile was written


@pytest.mark.slow
@pytest.mark.parametrize("sched", SCHEDS)
@pytest.mark.parametrize("pitch", [6144, 6143])
def test_gemm_ragged_fp32(lib, sched, pitch):
    w = synth.GEMM_RAGGED
    A, B = w.inputs()
    Dbuf = torch.full((w.M, pitch), float("nan"), dtype=torch.float32, device="cuda")
    D = Dbuf[:, :w.N]
    lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched=sched)
    lib.ts_sync_and_check()
    ref = oracle.gemm_f64_blas(A, B)
    S = oracle.gemm_f64_blas(A, B, absolute=True)
    assert_within_bound(as_f64(D), ref, S, torch.float32, f"ragged {sched} pitch {pitch}")
    if pitch > w.N:
        assert torch.isnan(Dbuf[:, w.N:]).all()
