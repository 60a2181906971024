"""GPU parity of the grouped GEMM (per-group K from an offsets array) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import as_f64, assert_bit_exact, assert_within_bound, to_device_bf16, tile_layouts

pytestmark = pytest.mark.gpu

TILES = ["128x128", "128x256", "256x256"]
OFFSETS = [0, 64, 64, 320, 448, 1024]  # slices of 64, 0, 256, 128 and 576 columns


def _run(lib, A_bits, B_bits, off, out, **kw):
    G = len(off) - 1
    D = torch.full((G, A_bits.shape[0], B_bits.shape[0]), float("nan"), dtype=out, device="cuda")
    lib.ts_gemm_bf16_grouped(to_device_bf16(A_bits), to_device_bf16(B_bits), D, off, **kw)
    lib.ts_sync_and_check()
    return D


@pytest.mark.parametrize("tile,ew,merge", tile_layouts(TILES))
@pytest.mark.parametrize("sched", ["static", "clc"])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_grouped_integer_bit_exact(lib, tile, sched, out, ew, merge):
    M, N = 300, 520
    A = synth.int_uniform_bf16(601, (M, 1024))
    B = synth.int_uniform_bf16(602, (N, 1024))
    D = _run(lib, A, B, OFFSETS, out, sched=sched, tile=tile, epi_warps=ew, merge=merge)
    ref = oracle.grouped_gemm_f64(A, B, OFFSETS, blas=True)
    for g in range(len(OFFSETS) - 1):
        assert_bit_exact(D[g], ref[g], f"group {g} {tile} {sched}")


@pytest.mark.parametrize("tile", TILES)
def test_grouped_random_within_bound_and_trace(lib, tile):
    M, N = 1024, 768
    off = [0, 640, 704, 2048, 2112, 4096]
    A = synth.uniform_pm1_bf16(611, (M, 4096))
    B = synth.uniform_pm1_bf16(612, (N, 4096))
    ref = oracle.grouped_gemm_f64(A, B, off, blas=True)
    S = oracle.grouped_gemm_f64(A, B, off, absolute=True, blas=True)
    for sched in ("static", "clc"):
        info = lib.ts_gemm_grouped_launch_info(M, N, off, lib.TS_OUT_BF16, sched, tile=tile)
        assert info["num_units"] == info["num_tiles"] == (len(off) - 1) * info["tiles_m"] * info["tiles_n"]
        trace = torch.zeros(4 * info["num_units"], dtype=torch.int64, device="cuda")
        D = _run(lib, A, B, off, torch.bfloat16, sched=sched, tile=tile, trace=trace)
        assert_within_bound(as_f64(D), ref, S, torch.bfloat16, f"grouped {tile} {sched}")
        tr = trace.view(-1, 4).cpu().numpy()
        if sched == "static":
            assert np.all(tr[:, 0] == 1)
            assert np.array_equal(tr[:, 1], oracle.static_owner(info["num_units"], info["workers"]))
        else:
            ok, why = oracle.clc_coverage_ok(tr[:, 0], tr[:, 1])
            assert ok, why


def test_grouped_offsets_not_starting_at_zero_and_strided_a(lib):
    M, N, Kcols = 200, 300, 640
    A_full = synth.int_uniform_bf16(621, (M, Kcols + 64))
    B = synth.int_uniform_bf16(622, (N, Kcols))
    off = [128, 256, 640]
    A = to_device_bf16(A_full)[:, :Kcols]  # row stride Kcols + 64
    D = torch.full((2, M, N), float("nan"), dtype=torch.float32, device="cuda")
    lib.ts_gemm_bf16_grouped(A, to_device_bf16(B), D, off, sched="clc")
    lib.ts_sync_and_check()
    ref = oracle.grouped_gemm_f64(np.ascontiguousarray(A_full[:, :Kcols]), B, off)
    for g in range(2):
        assert_bit_exact(D[g], ref[g], f"offset group {g}")


def test_grouped_all_empty_is_zero(lib):
    A = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    D = torch.full((3, 64, 64), 5.0, dtype=torch.float32, device="cuda")
    lib.ts_gemm_bf16_grouped(A, B, D, [0, 0, 0, 0])
    lib.ts_sync_and_check()
    assert torch.all(D == 0)


def test_grouped_rejects_bad_offsets(lib):
    A = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((2, 64, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(lib.TsError) as e:
        lib.ts_gemm_bf16_grouped(A, B, D, [0, 100, 256])
    assert e.value.status == lib.TS_ERR_INVALID_ARG
    with pytest.raises(lib.TsError) as e:
        lib.ts_gemm_bf16_grouped(A, B, D, [0, 192, 128])
    assert e.value.status == lib.TS_ERR_INVALID_ARG
    big = torch.zeros((300, 64, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(lib.TsError) as e:
        lib.ts_gemm_bf16_grouped(A, B, big, [0] * 301)
    assert e.value.status == lib.TS_ERR_UNSUPPORTED


@pytest.mark.slow
def test_grouped_workload_sampled(lib):
    w = synth.GROUPED
    off = w.k_offsets()
    A, B = w.inputs()
    for sched in ("static", "clc"):
        D = _run(lib, A, B, off, torch.bfloat16, sched=sched)
        rng = np.random.default_rng(5)
        for g in rng.choice(w.groups, 4, replace=False):
            rows = rng.integers(0, w.M, 16)
            k0, k1 = off[g], off[g + 1]
            a, b = A[rows, k0:k1], B[:, k0:k1]
            got = as_f64(D[int(g)][torch.as_tensor(rows, device="cuda")])
            assert_within_bound(got, oracle.gemm_f64_blas(a, b), oracle.gemm_f64_blas(a, b, absolute=True),
                                torch.bfloat16, f"grouped workload g{g}")


@pytest.mark.parametrize("tile,sched", [("128x256", "clc"), ("256x256", "static")])
def test_grouped_inputs_ready_back_to_back(lib, tile, sched):
    # grouped launches back to back into one D with inputs_ready (A and B never written): the
    # groups' first units run ahead of the previous launch, every D write waits for it
    M, N = 300, 520
    A = synth.int_uniform_bf16(603, (M, 1024))
    B = synth.int_uniform_bf16(604, (N, 1024))
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    G = len(OFFSETS) - 1
    D = torch.full((G, M, N), float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(4):
        lib.ts_gemm_bf16_grouped(Ad, Bd, D, OFFSETS, sched=sched, tile=tile, inputs_ready=1)
    lib.ts_sync_and_check()
    ref = oracle.grouped_gemm_f64(A, B, OFFSETS, blas=True)
    for g in range(G):
        assert_bit_exact(D[g], ref[g], f"group {g} {tile} {sched} inputs_ready")


def test_grouped_units_follow_the_longest_first_order(lib):
    # One static worker runs the units one after another in unit order.  Groups of 1, 64 and 1
    # k-blocks: the 64-block group is scheduled first, so the first four units (its 2 x 2 tiles)
    # are the long ones, and the gaps between consecutive unit ends show it.
    M, N = 256, 256
    off = [0, 64, 4160, 4224]
    assert list(lib.ts_gemm_grouped_order(off)) == [1, 0, 2]
    A = synth.int_uniform_bf16(631, (M, off[-1]))
    B = synth.int_uniform_bf16(632, (N, off[-1]))
    info = lib.ts_gemm_grouped_launch_info(M, N, off, lib.TS_OUT_F32, "static", tile="128x128", max_workers=1)
    assert info["workers"] == 1 and info["num_units"] == 12
    trace = torch.zeros(4 * info["num_units"], dtype=torch.int64, device="cuda")
    D = _run(lib, A, B, off, torch.float32, sched="static", tile="128x128", max_workers=1, trace=trace)
    ref = oracle.grouped_gemm_f64(A, B, off, blas=True)
    for g in range(3):
        assert_bit_exact(D[g], ref[g], f"group {g}")
    tr = trace.view(-1, 4).cpu().numpy()
    assert np.all(tr[:, 0] == 1) and np.all(tr[:, 1] == 0)
    gaps = np.diff(tr[:, 3]).astype(np.float64)  # gaps[i]: end of unit i + 1 after the end of unit i
    long_gaps, short_gaps = gaps[0:3], gaps[4:11]
    assert long_gaps.mean() > 3 * short_gaps.mean(), (long_gaps, short_gaps)


def test_automatic_tile_counts_every_group(lib):
    # the automatic tile choice counts the tiles of every group: sixteen groups of 2048 x 2048 fill
    # the GPU with 2-CTA 256 x 256 tiles, while one group alone takes the 128 x 128 tile
    off16 = [64 * i for i in range(17)]
    info = lib.ts_gemm_grouped_launch_info(2048, 2048, off16, lib.TS_OUT_BF16, "clc")
    assert (info["cluster"], info["tile_m"], info["tile_n"]) == (2, 256, 256)
    info = lib.ts_gemm_grouped_launch_info(2048, 2048, [0, 64], lib.TS_OUT_BF16, "clc")
    assert (info["cluster"], info["tile_m"], info["tile_n"]) == (1, 128, 128)
