"""Split tiles: the tiles that would leave the last wave partly empty, split along K.

Their parts are the first work units, so that the partial writes and the
reduction run in the epilogue while the mainloop already computes the next
tiles.  Each part writes an fp32 partial to the workspace; the warp that
finishes a 32-row slab last sums the parts in part order and stores D, then
re-arms the slab counter.  Integer inputs must stay bit-exact, random inputs within the
bound, the result must not depend on which part finished last, and the
workspace must come back zeroed.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import as_f64, assert_bit_exact, assert_within_bound, bf16_bits, to_device_bf16, LAYOUTS

pytestmark = pytest.mark.gpu

# (tile, M, N, K): each leaves a partial last wave on a 152-SM GB300, with
# K long enough for parts of at least 32 k-blocks
CASES = [("128x256", 2048, 2560, 4096), ("256x256", 2560, 2560, 4096), ("128x128", 1664, 1664, 4096)]


def _info(lib, M, N, K, out, sched, tile, ws):
    return lib.ts_gemm_launch_info(M, N, K, out, sched, tile=tile, workspace=ws)


@functools.lru_cache(maxsize=None)
def _integer_case(M, N, K):
    A = synth.int_uniform_bf16(801, (M, K))
    B = synth.int_uniform_bf16(802, (N, K))
    return A, B, oracle.gemm_f64_blas(A, B)


@functools.lru_cache(maxsize=None)
def _random_case(M, N, K):
    A = synth.uniform_pm1_bf16(811, (M, K))
    B = synth.uniform_pm1_bf16(812, (N, K))
    return A, B, oracle.gemm_f64_blas(A, B), oracle.gemm_f64_blas(A, B, absolute=True)


@pytest.mark.parametrize("tile,M,N,K", CASES)
@pytest.mark.parametrize("sched", ["static", "clc"])
@pytest.mark.parametrize("ew,merge", LAYOUTS)
def test_split_tail_integer_bit_exact_and_workspace_rearmed(lib, tile, M, N, K, sched, ew, merge):
    A, B, ref = _integer_case(M, N, K)
    need = _info(lib, M, N, K, lib.TS_OUT_F32, sched, tile, None)["workspace_bytes"]
    assert need > 0, "case must leave a partial last wave"
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    info = _info(lib, M, N, K, lib.TS_OUT_F32, sched, tile, ws)
    assert info["split_tiles"] > 0 and info["split_parts"] >= 2
    assert info["num_units"] == info["num_tiles"] + info["split_tiles"] * (info["split_parts"] - 1)
    trace = torch.zeros(4 * info["num_units"], dtype=torch.int64, device="cuda")
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched=sched, tile=tile, workspace=ws, trace=trace,
                        epi_warps=ew, merge=merge)
    lib.ts_sync_and_check()
    assert_bit_exact(D, ref, f"split {tile} {sched} {ew} epilogue warps")
    tr = trace.view(-1, 4).cpu().numpy()
    if sched == "static":
        assert np.all(tr[:, 0] == 1)
        assert np.array_equal(tr[:, 1], oracle.static_owner(info["num_units"], info["workers"]))
    else:
        ok, why = oracle.clc_coverage_ok(tr[:, 0], tr[:, 1])
        assert ok, why
    # counters re-armed: the workspace's counter region (first 8 KiB) is zero again
    assert torch.all(ws[:8192] == 0)


@pytest.mark.parametrize("tile,M,N,K", CASES)
@pytest.mark.parametrize("out", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("ew,merge", LAYOUTS)
def test_split_tail_random_within_bound_and_deterministic(lib, tile, M, N, K, out, ew, merge):
    A, B, ref, S = _random_case(M, N, K)
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    results = []
    for sched in ("clc", "static", "clc"):
        D = torch.full((M, N), float("nan"), dtype=out, device="cuda")
        lib.ts_gemm_bf16_ex(Ad, Bd, D, sched=sched, tile=tile, epi_warps=ew, merge=merge)  # cached workspace
        lib.ts_sync_and_check()
        assert_within_bound(as_f64(D), ref, S, out, f"split {tile} {sched} {out}")
        results.append(bf16_bits(D) if out == torch.bfloat16 else D.cpu().numpy())
    # same units, same summation order: repeatable bit for bit
    assert np.array_equal(results[0], results[2])
    # without a workspace the tail is not split; the result stays within the bound
    D = torch.full((M, N), float("nan"), dtype=out, device="cuda")
    lib.ts_gemm_bf16_ex(Ad, Bd, D, sched="static", tile=tile, workspace=None)
    lib.ts_sync_and_check()
    assert_within_bound(as_f64(D), ref, S, out, f"unsplit {tile} {out}")


@pytest.mark.parametrize("tile,M,N,K", CASES[:2])
def test_sixteen_epilogue_warps_do_not_split(lib, tile, M, N, K):
    # the 16-warp variants have no reduction path: the plan keeps whole tiles
    A, B, ref = _integer_case(M, N, K)
    need = _info(lib, M, N, K, lib.TS_OUT_F32, "clc", tile, None)["workspace_bytes"]
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    info = lib.ts_gemm_launch_info(M, N, K, lib.TS_OUT_F32, "clc", tile=tile, workspace=ws, epi_warps=16)
    assert info["split_tiles"] == 0 and info["num_units"] == info["num_tiles"] and info["epi_warps"] == 16
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched="clc", tile=tile, workspace=ws, epi_warps=16)
    lib.ts_sync_and_check()
    assert_bit_exact(D, ref, f"{tile} 16 epilogue warps, whole tiles")


def test_split_needs_enough_k(lib):
    # 32 k-blocks cannot be split into parts of at least 32 k-blocks
    info = lib.ts_gemm_launch_info(2048, 2560, 2048, lib.TS_OUT_BF16, "static", tile="128x256")
    assert info["split_tiles"] == 0 and info["workspace_bytes"] == 0
    info = lib.ts_gemm_launch_info(2048, 2560, 4096, lib.TS_OUT_BF16, "static", tile="128x256")
    assert info["split_tiles"] > 0 and info["split_parts"] == 2


def test_split_disabled_by_option(lib):
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    info = lib.ts_gemm_launch_info(2048, 2560, 4096, lib.TS_OUT_BF16, "static", tile="128x256", workspace=ws,
                                   split_tail=-1)
    assert info["split_tiles"] == 0 and info["num_units"] == info["num_tiles"]


@pytest.mark.parametrize("sched", ["static", "clc"])
def test_split_parts_are_the_first_units(lib, sched):
    # units 0 .. split_tiles * parts - 1 are the K parts of tiles 0 .. split_tiles - 1
    M, N, K = 2560, 2560, 4096
    A, B, ref = _integer_case(M, N, K)
    need = _info(lib, M, N, K, lib.TS_OUT_F32, sched, "256x256", None)["workspace_bytes"]
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    info = _info(lib, M, N, K, lib.TS_OUT_F32, sched, "256x256", ws)
    S, P = info["split_tiles"], info["split_parts"]
    assert S > 0
    trace = torch.zeros(4 * info["num_units"], dtype=torch.int64, device="cuda")
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched=sched, tile="256x256", workspace=ws,
                        trace=trace)
    lib.ts_sync_and_check()
    assert_bit_exact(D, ref, f"split-first {sched}")
    tr = trace.view(-1, 4).cpu().numpy()
    if sched == "static":
        # every split part runs as the first unit of its worker
        owner = tr[:, 1]
        assert len(set(owner[:S * P].tolist())) == S * P
        first = {}
        for u in range(info["num_units"]):
            first.setdefault(int(owner[u]), u)
        assert all(first[int(owner[u])] == u for u in range(S * P))


def test_automatic_workspaces_are_per_stream(lib):
    # split-tile launches on two streams at once, each with the binding's automatic workspace: the
    # streams get workspaces of their own, and both results are exact
    tile, M, N, K = "256x256", 2560, 2560, 4096
    A, B, ref = _integer_case(M, N, K)
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    assert _info(lib, M, N, K, lib.TS_OUT_F32, "clc", tile, "auto")["split_tiles"] > 0
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    need = _info(lib, M, N, K, lib.TS_OUT_F32, "clc", tile, None)["workspace_bytes"]
    assert lib.workspace_for(need, stream=s1).data_ptr() != lib.workspace_for(need, stream=s2).data_ptr()
    assert lib.workspace_for(need, stream=s1.cuda_stream).data_ptr() == lib.workspace_for(need, stream=s1).data_ptr()
    D1 = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    D2 = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        lib.ts_gemm_bf16_ex(Ad, Bd, D1, sched="clc", tile=tile, stream=s1)
        lib.ts_gemm_bf16_ex(Ad, Bd, D2, sched="static", tile=tile, stream=s2)
    torch.cuda.synchronize()
    lib.ts_sync_and_check()
    assert_bit_exact(D1, ref, "stream 1")
    assert_bit_exact(D2, ref, "stream 2")
