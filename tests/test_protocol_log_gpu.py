"""The barrier-protocol model checked against the kernel's own operations.

tile_scheduling_gb300/protocol.py restates the kernel's role loops by hand, and the explicit-state
checker explores every interleaving of that model.  Here the protocol-logging build of the kernel
(ts_gemm_opts.protocol_log) runs real launches and records, per CTA and role, every barrier
operation in program order: waits with their parity, arrivals, TMA loads, MMA k-blocks, tcgen05
commits, CLC requests and the dependent-launch wait.  For every worker that ran, the model is built
for the units that worker's producer logged, and each modelled role must have done exactly the
model's operations, in the model's order.  A reordering in the kernel that the model does not
follow, or the reverse, fails here.  The results of the logged launches are checked against the
oracle as well.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import tile_scheduling_gb300.protocol as pc
from parity import assert_bit_exact, to_device_bf16

pytestmark = pytest.mark.gpu

CAP = 2048


def _logged(lib, M, N, K, sched, tile, merge=0, max_workers=0, fork=False, skip=None, inputs_ready=0, offsets=None,
            seed=0x910, ew=4):
    Kt = offsets[-1] if offsets is not None else K
    A = synth.int_uniform_bf16(seed, (M, max(Kt, 8)))
    B = synth.int_uniform_bf16(seed + 1, (N, max(Kt, 8)))
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    kw = dict(sched=sched, tile=tile, merge=merge, max_workers=max_workers, epi_warps=ew, inputs_ready=inputs_ready)
    if offsets is not None:
        info = lib.ts_gemm_grouped_launch_info(M, N, offsets, lib.TS_OUT_F32, sched, tile=tile, merge=merge,
                                               max_workers=max_workers, epi_warps=ew)
    else:
        info = lib.ts_gemm_launch_info(M, N, K, lib.TS_OUT_F32, sched, tile=tile, merge=merge,
                                       max_workers=max_workers, epi_warps=ew,
                                       split_tail=-1 if (fork or skip is not None) else 0)
    log = torch.zeros((info["grid_ctas"], pc.LOG_ROLES, CAP + 1), dtype=torch.int32, device="cuda")
    R = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda") if fork else None
    if inputs_ready:  # a previous kernel in the stream for the dependent launch to wait on
        lib.ts_copy_i16(torch.zeros(1 << 22, dtype=torch.int16, device="cuda"),
                        torch.empty(1 << 22, dtype=torch.int16, device="cuda"))
    if offsets is not None:
        D = torch.full((len(offsets) - 1, M, N), float("nan"), dtype=torch.float32, device="cuda")
        lib.ts_gemm_bf16_grouped(Ad, Bd, D, offsets, protocol_log=log, **kw)
        lib.ts_sync_and_check()
        ref = oracle.grouped_gemm_f64(A, B, offsets, blas=True)
        for g in range(len(offsets) - 1):
            assert_bit_exact(D[g], ref[g], f"logged grouped launch, group {g}")
    else:
        D = torch.full((M, N), -3.0, dtype=torch.float32, device="cuda")
        lib.ts_gemm_bf16_ex(Ad, Bd, D, protocol_log=log, skip_tiles=skip, row_sums=R, **kw)
        lib.ts_sync_and_check()
        want = oracle.gemm_f64_blas(A, B).astype(np.float32)
        if skip is not None:
            tm, tn = info["tiles_m"], info["tiles_n"]
            keep = skip.cpu().numpy().reshape(tm, tn) != 0
            mask = np.repeat(np.repeat(keep, info["tile_m"], 0), info["tile_n"], 1)[:M, :N]
            want[mask] = -3.0
        assert np.array_equal(D.cpu().numpy(), want), "logged launch result"
        if fork:
            assert np.array_equal(R.cpu().numpy().astype(np.float64), oracle.row_sums_f64(A, [0, K])[0])
    return info, log.cpu().numpy()


def _check_workers(lib, info, log, tile, sched, merge=0, fork=False, early=False, mutate=None, ew=4):
    proto = lib.ts_gemm_protocol_info(tile, lib.TS_OUT_F32, ew, merge)
    cg = proto["cluster"]
    lazy = bool(info["clc_lazy"])
    ran, problems = 0, []
    for w in range(info["grid_ctas"] // cg):
        ctas = [w * cg + c for c in range(cg)]
        if log[ctas[0], 0, 0] == 0:
            continue  # a launch that a running worker took over (CLC) never ran
        _, units = pc.decode_log(log[ctas[0], 0])
        P = pc.build_program(proto, units, "clc" if sched == "clc" else "static", fork=fork, lazy=lazy,
                             lazy_lead=16, early=early, mutate=mutate)
        problems += [f"worker {w} units {units}: {p}" for p in pc.compare_with_log(P, log, ctas, lazy)]
        ran += 1
    return ran, problems


CASES = [
    # tile, sched, M, N, K, max_workers, merge
    ("128x128", "static", 384, 256, 512, 2, 0),    # 6 tiles on 2 persistent workers
    ("128x128", "static", 384, 256, 4096, 4, 0),   # split tiles first (long K parts)
    ("128x128", "clc", 2048, 2048, 512, 0, 0),     # more tiles than resident CTAs
    ("128x128", "clc", 2048, 2048, 4096, 0, 0),    # lazy CLC requests
    ("128x128", "nonpersistent", 512, 512, 512, 0, 0),
    ("128x128", "static", 384, 256, 512, 2, 1),    # Merge layout: A and B producers apart
    ("128x128", "clc", 2048, 2048, 512, 0, 1),
    ("256x256", "static", 1024, 1024, 512, 2, 0),  # CTA pairs
    ("256x256", "clc", 4096, 4096, 512, 0, 0),
    ("256x256", "clc", 4096, 4096, 4096, 0, 0),
]


@pytest.mark.parametrize("ready", [0, 1])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "%s_%s_%dx%dx%d_w%d_m%d" % c)
def test_kernel_operations_follow_the_model(lib, case, ready):
    tile, sched, M, N, K, mw, merge = case
    info, log = _logged(lib, M, N, K, sched, tile, merge=merge, max_workers=mw, inputs_ready=ready)
    if K == 4096 and sched == "static":
        assert info["split_tiles"] > 0
    if K == 4096 and sched == "clc":
        assert info["clc_lazy"] == 1
    ran, problems = _check_workers(lib, info, log, tile, sched, merge=merge, early=bool(ready))
    assert ran >= 1 and not problems, "\n".join(problems[:5])
    if sched == "clc":
        assert ran < info["grid_ctas"] // info["cluster"], "some worker should have taken over another's launch"


@pytest.mark.parametrize("ready", [0, 1])
@pytest.mark.parametrize("sched", ["static", "clc"])
@pytest.mark.parametrize("tile,ew,K", [("128x128", 8, 256), ("128x256", 16, 64), ("128x256", 16, 128)])
def test_more_epilogue_warps_follow_the_model(lib, tile, ew, K, sched, ready):
    # eight warps (two per TMEM lane quarter) and sixteen (four), the short-K epilogues
    M, N = 2048, 4096
    info, log = _logged(lib, M, N, K, sched, tile, max_workers=16 if sched == "static" else 0, inputs_ready=ready,
                        ew=ew)
    assert info["epi_warps"] == ew
    ran, problems = _check_workers(lib, info, log, tile, sched, early=bool(ready), ew=ew)
    assert ran >= 1 and not problems, "\n".join(problems[:5])


@pytest.mark.parametrize("sched", ["static", "clc"])
def test_fork_consumer_follows_the_model(lib, sched):
    info, log = _logged(lib, 1024, 512, 512, sched, "128x128", max_workers=4 if sched == "static" else 0,
                        fork=True)
    ran, problems = _check_workers(lib, info, log, "128x128", sched, fork=True)
    assert ran >= 1 and not problems, "\n".join(problems[:5])


@pytest.mark.parametrize("sched", ["static", "clc"])
def test_skipped_tiles_and_empty_groups_follow_the_model(lib, sched):
    # a causal skip mask, and a grouped launch whose first group has K = 0
    M = N = 2048
    tm = tn = 16
    skip = torch.from_numpy((np.arange(tn)[None, :] > np.arange(tm)[:, None]).astype(np.uint8).ravel()).cuda()
    info, log = _logged(lib, M, N, 512, sched, "128x128", max_workers=8 if sched == "static" else 0, skip=skip)
    ran, problems = _check_workers(lib, info, log, "128x128", sched)
    assert ran >= 1 and not problems, "\n".join(problems[:5])
    units = [u for w in range(info["grid_ctas"]) for u in pc.decode_log(log[w, 0])[1]]
    assert pc.SKIP in units
    info, log = _logged(lib, 512, 512, 0, sched, "128x128", max_workers=3 if sched == "static" else 0,
                        offsets=[0, 0, 256, 320])
    ran, problems = _check_workers(lib, info, log, "128x128", sched)
    assert ran >= 1 and not problems, "\n".join(problems[:5])
    units = [u for w in range(info["grid_ctas"]) for u in pc.decode_log(log[w, 0])[1]]
    assert 0 in units


def test_a_planted_model_mistake_does_not_match_the_kernel(lib):
    # the same logs against models with one planted mistake each: the comparison must object
    info, log = _logged(lib, 2048, 2048, 512, "clc", "128x128")
    for mutate in ("producer_wait_parity", "epilogue_release_before_read", "mma_skip_stage_release",
                   "tmem_empty_count_low"):
        ran, problems = _check_workers(lib, info, log, "128x128", "clc", mutate=mutate)
        if mutate == "tmem_empty_count_low":
            # a miscounted barrier changes no role's operations: the log cannot show it (the
            # checker's search does, and the counts come from the kernel's own constants)
            assert not problems
        else:
            assert problems, f"{mutate} went unnoticed"


def test_protocol_log_rejects_shapes_without_a_logging_build(lib):
    A = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((256, 256), dtype=torch.float32, device="cuda")
    log = torch.zeros((4, pc.LOG_ROLES, 9), dtype=torch.int32, device="cuda")
    with pytest.raises(lib.TsError) as e:
        lib.ts_gemm_bf16_ex(A, A, D, tile="128x256", protocol_log=log)
    assert e.value.status == lib.TS_ERR_UNSUPPORTED
