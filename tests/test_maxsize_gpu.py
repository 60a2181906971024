"""Problems whose outputs hold more than 2^31 elements: every offset past 2^31 needs 64-bit arithmetic.

The GEMM writes a 65541 x 32772 fp32 D (2.15e9 elements, 8.6 GB), through TMA stores at a pitch of
32772 elements and through plain stores at an odd pitch of 32773; the rows on both sides of element
2^31, the first and last rows and a seeded sample of others are compared bit for bit with the oracle
(integer inputs in [-4, 4], K = 64: every sum is exact), and the padding column of the odd pitch
must stay untouched.  The copy moves 2^31 + 37 int16 elements at relative offsets that take the
32-byte, the 16-byte and the shifted-vector paths; the whole destination is compared with the
source on the device, a sample of it with the oracle's copy, and the elements around it must keep
their sentinel.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_bit_exact, to_device_bf16

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.mark.parametrize("sched", ["static", "clc"])
@pytest.mark.parametrize("pitch", [32772, 32773])
def test_gemm_output_beyond_2_31_elements(lib, pitch, sched):
    M, N, K = 65541, 32772, 64
    assert M * N > 2 ** 31
    A = synth.int_uniform_bf16(0x3A1, (M, K))
    B = synth.int_uniform_bf16(0x3A2, (N, K))
    Dbuf = torch.full((M, pitch), -7.0, dtype=torch.float32, device="cuda")
    D = Dbuf[:, :N]
    lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched=sched)
    lib.ts_sync_and_check()
    cross = (2 ** 31) // pitch  # the row holding element 2^31 of the buffer
    rng = np.random.default_rng(0x3A3)
    rows = np.unique(np.concatenate([[0, 1, cross - 1, cross, cross + 1, M - 2, M - 1],
                                     rng.integers(0, M, 24)]))
    got = D[torch.as_tensor(rows, device="cuda")]
    assert_bit_exact(got, oracle.gemm_f64(A[rows], B), f"rows {rows.tolist()} pitch {pitch} {sched}")
    if pitch > N:
        assert bool((Dbuf[:, N:] == -7.0).all()), "a write into the padding column"


def _pattern(t: torch.Tensor, seed: int) -> None:
    # a seeded hash of the element index, written chunk by chunk (no index tensor of the full size)
    chunk = 1 << 27
    for c0 in range(0, t.numel(), chunk):
        i = torch.arange(c0, min(c0 + chunk, t.numel()), dtype=torch.int64, device=t.device)
        h = (i + seed) * 0x9E3779B1
        h = (h ^ (h >> 15)) * 0x85EBCA77
        t[c0:c0 + i.numel()] = ((h ^ (h >> 13)) & 0xFFFF).to(torch.int32).sub(32768).to(torch.int16)


@pytest.mark.parametrize("src_off,dst_off", [(0, 0), (0, 8), (0, 3)])
def test_copy_beyond_2_31_elements(lib, src_off, dst_off):
    n = (1 << 31) + 37
    src = torch.empty(n + 64, dtype=torch.int16, device="cuda")
    _pattern(src, 0x5EED)
    dst = torch.full((n + 64,), -1, dtype=torch.int16, device="cuda")
    lib.ts_copy_i16(src[src_off:src_off + n], dst[dst_off:dst_off + n])
    lib.ts_sync_and_check()
    assert torch.equal(dst[dst_off:dst_off + n], src[src_off:src_off + n])
    assert bool((dst[:dst_off] == -1).all()) and bool((dst[dst_off + n:] == -1).all())
    rng = np.random.default_rng(0x5EEE)
    idx = np.unique(np.concatenate([rng.integers(0, n, 1 << 14), np.arange((1 << 31) - 40, n)]))
    sample = src[src_off:src_off + n][torch.as_tensor(idx, device="cuda")].cpu().numpy()
    got = dst[dst_off:dst_off + n][torch.as_tensor(idx, device="cuda")].cpu().numpy()
    assert np.array_equal(got, oracle.copy_i16(sample))
