"""Failure detection without a GPU fault: bounded barrier waits.

A one-microsecond wait limit is far shorter than the time a tile's data takes
to arrive, so the kernel's waits run out.  The kernel must record the timeout
in the library's status word, let every role leave its loop, wait (with its
own limit) for copies and MMAs in flight, free TMEM and return: the host sees
TS_ERR_TIMEOUT from ts_sync_and_check, and the next launch on the same
context computes the right answer.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import as_f64, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("tile,sched", [("128x256", "static"), ("128x128", "clc"), ("256x256", "clc"),
                                        ("256x256", "static")])
@pytest.mark.parametrize("ready", [0, 1])
def test_wait_timeout_reported_then_context_still_works(lib, tile, sched, ready):
    # ready = 1: the timed-out launch follows a normal one with inputs_ready, so its roles time
    # out in their first unit, ahead of the dependent-launch barrier, and still leave cleanly
    M, N, K = 2048, 2048, 4096
    A_bits = synth.int_uniform_bf16(701, (M, K))
    B_bits = synth.int_uniform_bf16(702, (N, K))
    A, B = to_device_bf16(A_bits), to_device_bf16(B_bits)
    D = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    if ready:
        lib.ts_gemm_bf16_ex(A, B, D, sched=sched, tile=tile)
    lib.ts_gemm_bf16_ex(A, B, D, sched=sched, tile=tile, timeout_s=1e-6, inputs_ready=ready)
    with pytest.raises(lib.TsError) as e:
        lib.ts_sync_and_check()
    assert e.value.status == lib.TS_ERR_TIMEOUT
    assert "timed out" in e.value.detail
    # the status word was cleared and the context is healthy
    lib.ts_sync_and_check()
    D.zero_()
    lib.ts_gemm_bf16_ex(A, B, D, sched=sched, tile=tile)
    lib.ts_sync_and_check()
    rows = np.arange(0, M, 97)
    ref = oracle.gemm_f64(A_bits[rows], B_bits)
    assert np.array_equal(as_f64(D)[rows], ref)
