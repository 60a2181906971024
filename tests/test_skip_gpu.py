"""Skippable tiles: masked tiles are neither computed nor stored, yet every role still
hands them out and advances the queue (CUTLASS TS "Schedules", Skippable Tiles)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_bit_exact, to_device_bf16, tile_layouts

pytestmark = pytest.mark.gpu

SENTINEL = 3072.0  # exact in bf16


def _mask_rows_cols(mask, tm, tn, M, N):
    """Expand a [tiles_m, tiles_n] tile mask to an [M, N] element mask."""
    return np.repeat(np.repeat(mask, tm, axis=0), tn, axis=1)[:M, :N]


def _causal(tiles_m, tiles_n, tm, tn):
    mb = np.arange(tiles_m)[:, None]
    nb = np.arange(tiles_n)[None, :]
    return (nb * tn > mb * tm + tm - 1).astype(np.uint8)  # tiles entirely above the diagonal


@pytest.mark.parametrize("tile,ew,merge", tile_layouts(["128x128", "128x256", "256x256"]))
@pytest.mark.parametrize("sched", ["static", "clc"])
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
def test_skipped_tiles_untouched_others_exact(lib, tile, sched, out, ew, merge):
    M, N, K = 1500, 1400, 320
    A = synth.int_uniform_bf16(701, (M, K))
    B = synth.int_uniform_bf16(702, (N, K))
    info = lib.ts_gemm_launch_info(M, N, K, lib.TS_OUT_F32 if out == torch.float32 else lib.TS_OUT_BF16, sched,
                                   tile=tile, workspace=None)
    mask = _causal(info["tiles_m"], info["tiles_n"], info["tile_m"], info["tile_n"])
    assert 0 < mask.sum() < mask.size
    trace = torch.zeros(4 * info["num_units"], dtype=torch.int64, device="cuda")
    D = torch.full((M, N), SENTINEL, dtype=out, device="cuda")
    lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched=sched, tile=tile, workspace=None,
                        trace=trace, skip_tiles=torch.from_numpy(mask.reshape(-1)).cuda(), epi_warps=ew, merge=merge)
    lib.ts_sync_and_check()
    skipped = _mask_rows_cols(mask, info["tile_m"], info["tile_n"], M, N).astype(bool)
    ref = oracle.gemm_f64(A, B)
    ref[skipped] = SENTINEL
    assert_bit_exact(D, ref, f"skip {tile} {sched}")
    tr = trace.view(-1, 4).cpu().numpy()
    if sched == "static":  # the queue still advances over skipped tiles
        assert np.all(tr[:, 0] == 1)
        assert np.array_equal(tr[:, 1], oracle.static_owner(info["num_units"], info["workers"]))
    else:
        ok, why = oracle.clc_coverage_ok(tr[:, 0], tr[:, 1])
        assert ok, why


@pytest.mark.parametrize("tile,ew,merge", tile_layouts(["128x256", "256x256"]))
def test_skipped_tiles_with_lazy_clc_requests(lib, tile, ew, merge):
    # K = 2048 (32 k-blocks): CLC requests wait for the producer to near the end of its unit; a
    # skipped tile has no k-block, so its producer signals at once and the queue keeps moving
    M, N, K = 2048, 1792, 2048
    A = synth.int_uniform_bf16(721, (M, K))
    B = synth.int_uniform_bf16(722, (N, K))
    info = lib.ts_gemm_launch_info(M, N, K, lib.TS_OUT_F32, "clc", tile=tile, workspace=None)
    mask = _causal(info["tiles_m"], info["tiles_n"], info["tile_m"], info["tile_n"])
    trace = torch.zeros(4 * info["num_units"], dtype=torch.int64, device="cuda")
    D = torch.full((M, N), SENTINEL, dtype=torch.float32, device="cuda")
    lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched="clc", tile=tile, workspace=None,
                        trace=trace, skip_tiles=torch.from_numpy(mask.reshape(-1)).cuda(), epi_warps=ew, merge=merge)
    lib.ts_sync_and_check()
    skipped = _mask_rows_cols(mask, info["tile_m"], info["tile_n"], M, N).astype(bool)
    ref = oracle.gemm_f64_blas(A, B)
    ref[skipped] = SENTINEL
    assert_bit_exact(D, ref, f"skip + lazy CLC {tile}")
    ok, why = oracle.clc_coverage_ok(trace.view(-1, 4)[:, 0].cpu().numpy(), trace.view(-1, 4)[:, 1].cpu().numpy())
    assert ok, why


def test_every_tile_skipped_leaves_d_alone(lib):
    M, N, K = 512, 512, 128
    A = to_device_bf16(synth.int_uniform_bf16(711, (M, K)))
    B = to_device_bf16(synth.int_uniform_bf16(712, (N, K)))
    info = lib.ts_gemm_launch_info(M, N, K, lib.TS_OUT_F32, "clc", tile="128x128")
    D = torch.full((M, N), SENTINEL, device="cuda")
    lib.ts_gemm_bf16_ex(A, B, D, sched="clc", tile="128x128",
                        skip_tiles=torch.ones(info["num_tiles"], dtype=torch.uint8, device="cuda"))
    lib.ts_sync_and_check()
    assert torch.all(D == SENTINEL)


def test_skip_in_grouped_gemm(lib):
    M, N = 300, 400
    off = [0, 128, 384]
    A = synth.int_uniform_bf16(721, (M, 384))
    B = synth.int_uniform_bf16(722, (N, 384))
    info = lib.ts_gemm_grouped_launch_info(M, N, off, lib.TS_OUT_F32, "clc", tile="128x128")
    T1 = info["tiles_m"] * info["tiles_n"]
    mask = np.zeros((2, info["tiles_m"], info["tiles_n"]), np.uint8)
    mask[0, 0, :] = 1  # group 0: first tile row
    mask[1, :, 1] = 1  # group 1: second tile column
    D = torch.full((2, M, N), SENTINEL, dtype=torch.float32, device="cuda")
    lib.ts_gemm_bf16_grouped(to_device_bf16(A), to_device_bf16(B), D, off, sched="clc", tile="128x128",
                             skip_tiles=torch.from_numpy(mask.reshape(-1)).cuda())
    lib.ts_sync_and_check()
    ref = oracle.grouped_gemm_f64(A, B, off)
    for g in range(2):
        ref[g][_mask_rows_cols(mask[g], 128, 128, M, N).astype(bool)] = SENTINEL
        assert_bit_exact(D[g], ref[g], f"grouped skip g{g}")
    assert mask.size == 2 * T1


def test_skip_mask_disables_the_split_tail(lib):
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    m = torch.zeros(512, dtype=torch.uint8, device="cuda")
    info = lib.ts_gemm_launch_info(4096, 4096, 1024, lib.TS_OUT_BF16, "static", tile="128x256", workspace=ws,
                                   skip_tiles=m)
    assert info["split_tiles"] == 0
