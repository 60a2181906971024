"""The allocation-free, self-checking GEMM entry point, compared with the existing one.

ts_gemm_bf16_checked_noalloc serves callers that cannot call cudaMalloc (for
instance a plugin whose host process owns all device memory): its per-tile
trace sits in a fixed array inside the library instead of caller memory.  The
file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import as_f64, assert_bit_exact, assert_within_bound, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("sched", ["static", "clc", "nonpersistent"])
def test_no_alloc_entry_point_matches_existing_entry_point(lib, sched):
    M, N, K = 1000, 1200, 320
    A_bits = synth.uniform_pm1_bf16(901, (M, K))
    B_bits = synth.uniform_pm1_bf16(902, (N, K))
    A, B = to_device_bf16(A_bits), to_device_bf16(B_bits)
    ref = oracle.gemm_f64(A_bits, B_bits)
    S = oracle.gemm_f64(A_bits, B_bits, absolute=True)

    D_old = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    info = lib.ts_gemm_launch_info(M, N, K, lib.TS_OUT_F32, sched)
    trace = torch.zeros(4 * info["num_units"], dtype=torch.int64, device="cuda")
    lib.ts_gemm_bf16_ex(A, B, D_old, sched=sched, trace=trace)
    lib.ts_sync_and_check()
    assert np.all(trace.view(-1, 4)[:, 0].cpu().numpy() == 1)

    bad = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):  # the shared scratch keeps the previous call's contents
        D_new = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        bad.fill_(-1)
        lib.ts_gemm_bf16_checked_noalloc(A, B, D_new, bad, sched=sched)
        lib.ts_sync_and_check()
        assert int(bad.item()) == 0, f"call {call}: {int(bad.item())} tiles not computed exactly once"
        assert_within_bound(as_f64(D_new), as_f64(D_old), S, torch.float32, f"no-alloc vs existing, call {call}")
        assert_within_bound(as_f64(D_new), ref, S, torch.float32, f"no-alloc vs oracle, call {call}")


def test_no_alloc_entry_point_rejects_oversized_problems(lib):
    # 65536 tiles is the scratch limit; the default tile choice gives 300 x 300 tiles here
    M, N, K = 256 * 300, 256 * 300, 64
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = lib._lib.ts_gemm_bf16_checked_noalloc(None, None, None, M, N, K, lib.TS_OUT_BF16, lib.TS_SCHED_STATIC,
                                               bad.data_ptr(), None)
    assert st == lib.TS_ERR_UNSUPPORTED
    assert "65536" in lib.ts_last_error_detail()


def test_no_alloc_entry_point_on_the_cta_pair_tile_after_a_larger_call(lib):
    # the default tile choice here is the 2-CTA pair (only rank 0 of a pair writes the
    # trace); a smaller call after a larger one must not count entries the larger call
    # left past its own tiles
    big = (3072, 3072, 128)
    small = (2304, 2304, 64)
    bad = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for (M, N, K), seed in ((big, 911), (small, 913), (small, 915)):
        info = lib.ts_gemm_launch_info(M, N, K, lib.TS_OUT_BF16, "clc")
        assert info["cluster"] == 2
        A_bits = synth.int_uniform_bf16(seed, (M, K))
        B_bits = synth.int_uniform_bf16(seed + 1, (N, K))
        D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        bad.fill_(-1)
        lib.ts_gemm_bf16_checked_noalloc(to_device_bf16(A_bits), to_device_bf16(B_bits), D, bad, sched="clc")
        lib.ts_sync_and_check()
        assert int(bad.item()) == 0, f"{(M, N, K)}: {int(bad.item())} tiles not computed exactly once"
        assert_bit_exact(D, oracle.gemm_f64(A_bits, B_bits), f"no-alloc 2-CTA {(M, N, K)}")


def test_no_alloc_entry_point_with_k_zero(lib):
    # K = 0: D is the empty sum (zero-filled), no tile is scheduled and none is counted bad
    M, N = 300, 200
    A = torch.zeros((M, 8), dtype=torch.bfloat16, device="cuda")[:, :0]
    B = torch.zeros((N, 8), dtype=torch.bfloat16, device="cuda")[:, :0]
    D = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    bad = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    st = lib._lib.ts_gemm_bf16_checked_noalloc(None, None, ctypes.c_void_p(D.data_ptr()), M, N, 0, lib.TS_OUT_F32,
                                               lib.TS_SCHED_CLC, ctypes.c_void_p(bad.data_ptr()), None)
    assert st == lib.TS_OK
    lib.ts_sync_and_check()
    assert int(bad.item()) == 0
    assert torch.all(D == 0)
