"""Tile-scheduler coverage on the GPU, from the kernel's per-tile trace.

Static: the owner of every tile is the one the grid-stride rule gives
(oracle.static_owner, pinned by the 12-tile / 4-worker worked example).
Cluster Launch Control: every tile is visited exactly once, and every worker
that ran started on the tile of its own block index; results stay identical
while part of the GPU is held by another kernel.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import as_f64, assert_bit_exact, assert_within_bound, to_device_bf16, tile_layouts

pytestmark = pytest.mark.gpu


def _traced(lib, A_bits, B_bits, out, tile, sched, **kw):
    M, N = A_bits.shape[0], B_bits.shape[0]
    info = lib.ts_gemm_launch_info(M, N, A_bits.shape[1], lib.TS_OUT_F32 if out == torch.float32 else lib.TS_OUT_BF16,
                                   sched, tile=tile, **kw)
    trace = torch.zeros(4 * info["num_units"], dtype=torch.int64, device="cuda")
    D = torch.full((M, N), float("nan"), dtype=out, device="cuda")
    lib.ts_gemm_bf16_ex(to_device_bf16(A_bits), to_device_bf16(B_bits), D, sched=sched, tile=tile, trace=trace,
                        **kw)
    lib.ts_sync_and_check()
    return info, trace.view(-1, 4).cpu().numpy(), D


@pytest.mark.parametrize("tile,ew,merge", tile_layouts(["128x128", "128x256", "256x256"]))
@pytest.mark.parametrize("max_workers", [0, 7, 1])
def test_static_owner_follows_grid_stride_rule(lib, tile, max_workers, ew, merge):
    M, N, K = 1500, 1300, 128
    A = synth.int_uniform_bf16(301, (M, K))
    B = synth.int_uniform_bf16(302, (N, K))
    info, tr, D = _traced(lib, A, B, torch.float32, tile, "static", max_workers=max_workers, epi_warps=ew,
                          merge=merge)
    assert info["epi_warps"] == ew
    if max_workers:
        assert info["workers"] == min(max_workers, info["num_units"])
    assert np.all(tr[:, 0] == 1), "a work unit was not visited exactly once"
    assert np.array_equal(tr[:, 1], oracle.static_owner(info["num_units"], info["workers"]))
    assert np.all(tr[:, 3] >= tr[:, 2])
    assert_bit_exact(D, oracle.gemm_f64(A, B), f"static {tile}")


@pytest.mark.parametrize("tile,ew,merge", tile_layouts(["128x128", "128x256", "256x256"]))
def test_clc_covers_every_tile_once(lib, tile, ew, merge):
    M, N, K = 4000, 3000, 64  # many more tiles than resident workers
    A = synth.int_uniform_bf16(311, (M, K))
    B = synth.int_uniform_bf16(312, (N, K))
    info, tr, D = _traced(lib, A, B, torch.bfloat16, tile, "clc", epi_warps=ew, merge=merge)
    assert info["grid_ctas"] == info["num_units"] * info["cluster"]
    ok, why = oracle.clc_coverage_ok(tr[:, 0], tr[:, 1])
    assert ok, why
    # work stealing happened: fewer workers ran than there are units
    assert np.unique(tr[:, 1]).size < info["num_units"]
    ref = oracle.gemm_f64_blas(A, B)
    assert_bit_exact(D, ref, f"clc {tile}")


@pytest.mark.parametrize("sched", ["static", "clc"])
def test_results_identical_while_sms_are_held(lib, sched):
    M, N, K = 2048, 2048, 1024
    A = synth.int_uniform_bf16(321, (M, K))
    B = synth.int_uniform_bf16(322, (N, K))
    ref = oracle.gemm_f64_blas(A, B)
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    side = torch.cuda.Stream()
    started = torch.zeros(1, dtype=torch.int32).pin_memory()
    ctas = 32
    info = lib.ts_gemm_launch_info(M, N, K, lib.TS_OUT_F32, sched, tile="128x256")
    trace = torch.zeros(4 * info["num_units"], dtype=torch.int64, device="cuda")
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    lib.ts_spin(ctas, 20_000_000, started, stream=side)
    lib.ts_spin_wait_started(started, ctas, 5.0)
    lib.ts_gemm_bf16_ex(Ad, Bd, D, sched=sched, tile="128x256", trace=trace)
    torch.cuda.synchronize()
    lib.ts_sync_and_check()
    assert started.item() == ctas
    assert_bit_exact(D, ref, f"contended {sched}")
    tr = trace.view(-1, 4).cpu().numpy()
    if sched == "clc":
        ok, why = oracle.clc_coverage_ok(tr[:, 0], tr[:, 1])
        assert ok, why
    else:
        assert np.array_equal(tr[:, 1], oracle.static_owner(info["num_units"], info["workers"]))


def test_spin_rejects_bad_arguments(lib):
    started = torch.zeros(1, dtype=torch.int32).pin_memory()
    with pytest.raises(lib.TsError):
        lib.ts_spin(0, 1000, started)
    with pytest.raises(lib.TsError):
        lib.ts_spin(1, -5, started)
    with pytest.raises(TypeError):
        lib.ts_spin(1, 1000, torch.zeros(1, dtype=torch.int32))


@pytest.mark.parametrize("tile,ew,merge", tile_layouts(["128x256", "256x256"]))
@pytest.mark.parametrize("held", [0, 32])
def test_lazy_clc_claims_balance_few_long_units(lib, tile, ew, merge, held):
    # 2560 x 2560 x 8192: few units per worker and long K loops, so the scheduler's requests
    # wait until the producer has nearly loaded its unit.  Every unit once, every running
    # worker starts on its own block's unit, the result bit-exact, with and without SMs held;
    # no worker ends up with two more whole tiles than another.
    M, N, K = 2560, 2560, 8192
    A = synth.int_uniform_bf16(331, (M, K))
    B = synth.int_uniform_bf16(332, (N, K))
    started = torch.zeros(1, dtype=torch.int32).pin_memory()
    if held:
        side = torch.cuda.Stream()
        lib.ts_spin(held, 100_000, started, stream=side)
        lib.ts_spin_wait_started(started, held, 5.0)
    info, tr, D = _traced(lib, A, B, torch.float32, tile, "clc", epi_warps=ew, merge=merge)
    torch.cuda.synchronize()
    ok, why = oracle.clc_coverage_ok(tr[:, 0], tr[:, 1])
    assert ok, why
    assert_bit_exact(D, oracle.gemm_f64_blas(A, B), f"lazy CLC {tile} held {held}")
    if not held:
        kb = 128  # k-blocks of a whole tile
        work = {}
        for u in range(info["num_units"]):
            w = int(tr[u, 1])
            part = u < info["split_tiles"] * info["split_parts"]
            work[w] = work.get(w, 0) + (kb // info["split_parts"] if part else kb)
        assert max(work.values()) - min(work.values()) <= kb + kb // max(info["split_parts"], 1)


@pytest.mark.parametrize("tile,M,N", [("128x128", 2048, 2048), ("128x256", 2048, 4096), ("256x256", 4096, 2048)])
def test_random_results_identical_across_schedulers_and_caps(lib, tile, M, N):
    # More units than fit at once, so the second wave's units walk their K range
    # downwards.  Which way a unit walks depends only on its index and the plan's
    # resident worker count, so on non-integer inputs (where the summation order
    # shows in the fp32 result) static, CLC and a capped static grid agree bit for
    # bit, and each lies within the error bound of the oracle's product.
    K = 512
    A = synth.uniform_pm1_bf16(341, (M, K))
    B = synth.uniform_pm1_bf16(342, (N, K))
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    info = lib.ts_gemm_launch_info(M, N, K, lib.TS_OUT_F32, "static", tile=tile)
    assert info["num_units"] > info["resident"] and info["split_tiles"] == 0
    outs = []
    for sched, cap in (("static", 0), ("clc", 0), ("static", 7)):
        D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        lib.ts_gemm_bf16_ex(Ad, Bd, D, sched=sched, tile=tile, max_workers=cap)
        lib.ts_sync_and_check()
        outs.append(D)
    for D, what in zip(outs[1:], ("clc", "static capped at 7 workers")):
        assert torch.equal(outs[0], D), f"{tile}: {what} differs from static"
    assert_within_bound(as_f64(outs[0]), oracle.gemm_f64_blas(A, B), oracle.gemm_f64_blas(A, B, absolute=True),
                        torch.float32, f"random {tile}")


@pytest.mark.parametrize("tile,ew,merge", tile_layouts(["128x128", "128x256", "256x256"]))
@pytest.mark.parametrize("ready", [0, 1])
def test_nonpersistent_each_block_computes_its_own_unit(lib, tile, ew, merge, ready):
    # the pages' non-persistent scheduling shape: one CTA (cluster) per unit, no queue
    M, N, K = 1500, 1300, 192
    A = synth.int_uniform_bf16(351, (M, K))
    B = synth.int_uniform_bf16(352, (N, K))
    info, tr, D = _traced(lib, A, B, torch.float32, tile, "nonpersistent", epi_warps=ew, merge=merge,
                          inputs_ready=ready)
    assert info["workers"] == info["num_units"] and info["grid_ctas"] == info["num_units"] * info["cluster"]
    assert np.all(tr[:, 0] == 1), "a work unit was not visited exactly once"
    assert np.array_equal(tr[:, 1], np.arange(info["num_units"])), "a block computed another block's unit"
    assert_bit_exact(D, oracle.gemm_f64(A, B), f"non-persistent {tile}")


@pytest.mark.parametrize("tile", ["128x256", "256x256"])
def test_nonpersistent_with_split_tiles(lib, tile):
    M, N, K = 2560, 2560, 4096
    A = synth.int_uniform_bf16(361, (M, K))
    B = synth.int_uniform_bf16(362, (N, K))
    info, tr, D = _traced(lib, A, B, torch.float32, tile, "nonpersistent")
    assert info["split_tiles"] > 0
    assert np.all(tr[:, 0] == 1) and np.array_equal(tr[:, 1], np.arange(info["num_units"]))
    assert_bit_exact(D, oracle.gemm_f64_blas(A, B), f"non-persistent split {tile}")
