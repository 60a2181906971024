"""Full-size parity at the exact shapes and launch choices the benchmark times, bit for bit.

Entries are integers in [-4, 4] (exact in bf16).  Every partial sum is an
integer of magnitude at most 16 * K <= 131072 < 2^24, so the fp32 tensor-core
accumulation is exact in any order and the bf16 output is the round to nearest
even of the exact value; the oracle's float64 BLAS route is exact on the same
inputs for the same reason.  Every element of D is compared, not a sample.
The workloads: 4096^3 (128x256 tile and the automatic choice, static and CLC),
8192^3 on the 2-CTA 256x256 tile under CLC with the split tiles planned and
applied, the ragged 8191 x 6143 x 4096 fp32 GEMM at pitches 6144 (TMA stores)
and 6143 (plain stores) alone and with 32 SMs held by the spin kernel, and the
small-K 8192 x 8192 x 64 GEMM.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_bit_exact, to_device_bf16

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

_REF = {}


def _int_inputs(M, N, K, seed):
    return synth.int_uniform_bf16(seed, (M, K)), synth.int_uniform_bf16(seed + 1, (N, K))


def _ref(key, A, B):
    """The oracle's exact float64 product, cached per shape (the inputs are seeded per shape)."""
    if key not in _REF:
        _REF.clear()
        _REF[key] = oracle.gemm_f64_blas(A, B)
    return _REF[key]


@pytest.mark.parametrize("tile", ["128x256", "auto"])
@pytest.mark.parametrize("sched", ["static", "clc"])
def test_4096_integer_every_element(lib, tile, sched):
    M = N = K = 4096
    A, B = _int_inputs(M, N, K, 4096)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched=sched, tile=tile)
    lib.ts_sync_and_check()
    assert_bit_exact(D, _ref("4096", A, B), f"4096^3 integer {tile} {sched}")


@pytest.mark.parametrize("sched", ["clc", "static"])
def test_8192_integer_2cta_split_tail_every_element(lib, sched):
    M = N = K = 8192
    info = lib.ts_gemm_launch_info(M, N, K, lib.TS_OUT_BF16, sched, tile="256x256")
    # the launch the benchmark times: 2-CTA pair tiles with the last partial wave split along K
    assert info["cluster"] == 2 and info["split_tiles"] > 0 and info["split_parts"] >= 2
    A, B = _int_inputs(M, N, K, 8192)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched=sched, tile="256x256")
    lib.ts_sync_and_check()
    assert_bit_exact(D, _ref("8192", A, B), f"8192^3 integer 2-CTA {sched}")


@pytest.mark.parametrize("spin", [False, True])
@pytest.mark.parametrize("pitch", [6144, 6143])
@pytest.mark.parametrize("sched", ["static", "clc"])
def test_ragged_integer_fp32_every_element(lib, sched, pitch, spin):
    M, N, K = 8191, 6143, 4096
    A, B = _int_inputs(M, N, K, 8191)
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    Dbuf = torch.full((M, pitch), float("nan"), dtype=torch.float32, device="cuda")
    D = Dbuf[:, :N]
    if spin:
        # the contended launch: a spin kernel on a second stream holds 32 SMs while the GEMM starts
        started = torch.zeros(1, dtype=torch.int32).pin_memory()
        side = torch.cuda.Stream()
        lib.ts_spin(32, 150_000, started, stream=side)
        lib.ts_spin_wait_started(started, 32, 5.0)
    lib.ts_gemm_bf16_ex(Ad, Bd, D, sched=sched, tile="256x256")
    torch.cuda.synchronize()
    lib.ts_sync_and_check()
    assert_bit_exact(D, _ref("ragged", A, B), f"ragged integer {sched} pitch {pitch} spin {spin}")
    if pitch > N:
        assert torch.isnan(Dbuf[:, N:]).all()


@pytest.mark.parametrize("tile", ["256x256", "128x256"])
@pytest.mark.parametrize("sched", ["static", "clc"])
def test_small_k_integer_every_element(lib, tile, sched):
    M, N, K = 8192, 8192, 64
    A, B = _int_inputs(M, N, K, 64)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched=sched, tile=tile)
    lib.ts_sync_and_check()
    assert_bit_exact(D, _ref("smallk", A, B), f"8192x8192x64 integer {tile} {sched}")
