"""The Fork pipeline group: the ring's A stages feed the MMA and a second consumer task
that writes per-row sums of A (CUTLASS TS "Pipeline Groups", Fork)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_bit_exact, as_f64, assert_within_bound, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("tile,ew", [("128x128", 4), ("128x128", 8), ("128x256", 4), ("128x256", 8), ("128x256", 16)])
@pytest.mark.parametrize("sched", ["static", "clc"])
def test_fork_integer_exact(lib, tile, sched, ew):
    M, N, K = 700, 600, 640
    A = synth.int_uniform_bf16(801, (M, K))
    B = synth.int_uniform_bf16(802, (N, K))
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    R = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched=sched, tile=tile, row_sums=R, epi_warps=ew)
    lib.ts_sync_and_check()
    assert_bit_exact(D, oracle.gemm_f64(A, B), f"fork D {tile} {sched} {ew}")
    assert np.array_equal(R.cpu().numpy().astype(np.float64), oracle.row_sums_f64(A, [0, K])[0])


@pytest.mark.parametrize("sched", ["static", "clc"])
def test_fork_random_row_sums_within_fp32_bound(lib, sched):
    M, N, K = 1000, 512, 4096
    A = synth.uniform_pm1_bf16(811, (M, K))
    B = synth.uniform_pm1_bf16(812, (N, K))
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    R = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched=sched, row_sums=R)
    lib.ts_sync_and_check()
    ref = oracle.row_sums_f64(A, [0, K])[0]
    absum = np.abs(oracle.bf16_to_f64(A)).sum(1)
    # K sequential fp32 additions: |error| <= K * 2^-24 * sum |a|
    assert np.all(np.abs(R.cpu().numpy() - ref) <= K * 2.0 ** -24 * absum)
    assert_within_bound(as_f64(D), oracle.gemm_f64(A, B), oracle.gemm_f64(A, B, absolute=True), torch.bfloat16,
                        "fork D")


def test_fork_grouped_and_skipped(lib):
    M, N = 300, 400
    off = [0, 128, 128, 384]
    A = synth.int_uniform_bf16(821, (M, 384))
    B = synth.int_uniform_bf16(822, (N, 384))
    info = lib.ts_gemm_grouped_launch_info(M, N, off, lib.TS_OUT_F32, "clc", tile="128x128")
    mask = np.zeros((3, info["tiles_m"], info["tiles_n"]), np.uint8)
    mask[0, 1, 0] = 1  # group 0, tile row 1, first column: its rows' sums stay untouched
    D = torch.zeros((3, M, N), dtype=torch.float32, device="cuda")
    R = torch.full((3, M), -7.0, dtype=torch.float32, device="cuda")
    lib.ts_gemm_bf16_grouped(to_device_bf16(A), to_device_bf16(B), D, off, sched="clc", tile="128x128",
                             skip_tiles=torch.from_numpy(mask.reshape(-1)).cuda(), row_sums=R)
    lib.ts_sync_and_check()
    want = oracle.row_sums_f64(A, off)
    want[0, 128:256] = -7.0
    assert np.array_equal(R.cpu().numpy().astype(np.float64), want)


def test_fork_needs_a_one_cta_tile(lib):
    A = torch.zeros((512, 128), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((512, 512), dtype=torch.float32, device="cuda")
    R = torch.zeros(512, dtype=torch.float32, device="cuda")
    with pytest.raises(lib.TsError) as e:
        lib.ts_gemm_bf16_ex(A, A, D, tile="256x256", row_sums=R)
    assert e.value.status == lib.TS_ERR_UNSUPPORTED
    info = lib.ts_gemm_launch_info(8192, 8192, 1024, lib.TS_OUT_BF16, "clc", row_sums=R)
    assert info["cluster"] == 1 and info["split_tiles"] == 0
