"""Stream order across back-to-back launches (GEMMs are programmatic dependents).

Each GEMM launch may start its prologue while the previous kernel in the
stream is still running, and waits (griddepcontrol) before touching global
memory.  These chains would read stale data or lose writes if it did not:
every case is integer-valued so the results are exact.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import assert_bit_exact, bf16_bits, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("tile,sched", [("128x256", "static"), ("256x256", "clc"), ("128x128", "clc")])
def test_gemm_chain_reads_the_previous_output(lib, tile, sched):
    # D1 = A B^T (bf16, exact small integers), then D2 = D1 C^T, D3 = D2 E^T, launched back to back
    M, K = 1024, 128
    A = synth.int_uniform_bf16(901, (M, K))
    B = synth.one_hot_rows_bf16(K, K, np.random.default_rng(1).permutation(K))  # D1 = a column permutation of A
    C = synth.one_hot_rows_bf16(K, K, np.random.default_rng(2).permutation(K))
    E = synth.int_uniform_bf16(903, (256, K))
    d_a, d_b, d_c, d_e = (to_device_bf16(x) for x in (A, B, C, E))
    D1 = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    D2 = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    D3 = torch.full((M, 256), float("nan"), dtype=torch.float32, device="cuda")
    for _ in range(3):  # repeated so that later launches overlap earlier ones' tails
        lib.ts_gemm_bf16_ex(d_a, d_b, D1, sched=sched, tile=tile)
        lib.ts_gemm_bf16_ex(D1, d_c, D2, sched=sched, tile=tile)
        lib.ts_gemm_bf16_ex(D2, d_e, D3, sched=sched, tile=tile)
    lib.ts_sync_and_check()
    d1 = oracle.gemm_f64(A, B)
    assert np.array_equal(bf16_bits(D1), oracle.bf16_rne(d1))
    d2_bits = oracle.bf16_rne(oracle.gemm_f64(oracle.bf16_rne(d1), C))
    assert np.array_equal(bf16_bits(D2), d2_bits)
    assert_bit_exact(D3, oracle.gemm_f64(d2_bits, E), f"chain {tile} {sched}")


def test_gemm_overwrites_in_stream_order(lib):
    # two GEMMs write the same D back to back: the second one's values remain
    M, N, K = 2048, 2048, 64
    A1, A2 = synth.int_uniform_bf16(911, (M, K)), synth.int_uniform_bf16(912, (M, K))
    B = synth.int_uniform_bf16(913, (N, K))
    d_a1, d_a2, d_b = to_device_bf16(A1), to_device_bf16(A2), to_device_bf16(B)
    D = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    for _ in range(4):
        lib.ts_gemm_bf16_ex(d_a1, d_b, D, sched="clc")
        lib.ts_gemm_bf16_ex(d_a2, d_b, D, sched="static")
    lib.ts_sync_and_check()
    assert_bit_exact(D, oracle.gemm_f64(A2, B), "write after write")


def test_copy_then_gemm_then_copy(lib):
    # the GEMM reads what the copy kernel just wrote; the next copy reads the GEMM's output
    M, N, K = 512, 768, 192
    A = synth.int_uniform_bf16(921, (M, K))
    B = synth.int_uniform_bf16(922, (N, K))
    src = to_device_bf16(A).view(torch.int16).reshape(-1)
    a_copy = torch.zeros_like(src)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(M * N, dtype=torch.int16, device="cuda")
    lib.ts_copy_i16(src, a_copy)
    lib.ts_gemm_bf16_ex(a_copy.view(torch.bfloat16).view(M, K), to_device_bf16(B), D, sched="clc")
    lib.ts_copy_i16(D.view(torch.int16).reshape(-1), out)
    lib.ts_sync_and_check()
    want = oracle.bf16_rne(oracle.gemm_f64(A, B))
    assert np.array_equal(bf16_bits(D), want)
    assert np.array_equal(out.cpu().numpy().view(np.uint16).reshape(M, N), want)


@pytest.mark.parametrize("pack", [0, 1])
def test_row_copy_between_gemms_with_offsets_written_just_before(lib, pack):
    # GEMM -> (a kernel writes the offsets) -> planned row copy of the GEMM's output -> GEMM on the copy:
    # the planning kernels and the copy are programmatic dependents and must see every earlier write
    M, N, K = 512, 512, 128
    A = synth.int_uniform_bf16(931, (M, K))
    B = synth.int_uniform_bf16(932, (N, K))
    E = synth.int_uniform_bf16(933, (256, N))
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    D2 = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    D3 = torch.full((M, 256), float("nan"), dtype=torch.float32, device="cuda")
    lengths = (synth.splitmix64(934, M) % np.uint64(2 * N)).astype(np.int64)
    bounds = np.minimum(np.concatenate([[0], np.cumsum(lengths)]), M * N).astype(np.int64)
    bounds[-1] = M * N  # the rows cover the whole output
    off = torch.zeros(M + 1, dtype=torch.int64, device="cuda")
    ws = torch.empty(lib.ts_copy_rows_launch_info(M * N, M, "clc", chunk=4096, pack=pack)["workspace_bytes"],
                     dtype=torch.uint8, device="cuda")
    for _ in range(3):
        off.zero_()
        lib.ts_gemm_bf16_ex(to_device_bf16(A), to_device_bf16(B), D, sched="clc")
        off.copy_(torch.from_numpy(bounds).cuda(non_blocking=False))
        lib.ts_copy_i16_rows(D.view(torch.int16).reshape(-1), D2.view(torch.int16).reshape(-1), off, sched="clc",
                             chunk=4096, pack=pack, workspace=ws)
        lib.ts_gemm_bf16_ex(D2, to_device_bf16(E), D3, sched="static")
    lib.ts_sync_and_check()
    d_bits = oracle.bf16_rne(oracle.gemm_f64(A, B))
    assert np.array_equal(bf16_bits(D2), d_bits)
    assert_bit_exact(D3, oracle.gemm_f64(d_bits, E), f"row copy between GEMMs, pack {pack}")


def test_cuda_graph_replay(lib):
    # a GEMM, a copy and a planned row copy captured once and replayed with new inputs
    M, N, K = 512, 768, 192
    B = synth.int_uniform_bf16(941, (N, K))
    d_b = to_device_bf16(B)
    A_in = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(M * N, dtype=torch.int16, device="cuda")
    rows_out = torch.zeros(M * N, dtype=torch.int16, device="cuda")
    off = torch.from_numpy(np.arange(0, M * N + 1, N, dtype=np.int64)).cuda()
    ws = torch.empty(lib.ts_copy_rows_launch_info(M * N, M, "clc", chunk=1000)["workspace_bytes"], dtype=torch.uint8,
                     device="cuda")
    gemm_ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")

    def step():
        lib.ts_gemm_bf16_ex(A_in, d_b, D, sched="clc", workspace=gemm_ws)
        lib.ts_copy_i16(D.view(torch.int16).reshape(-1), out)
        lib.ts_copy_i16_rows(out, rows_out, off, sched="clc", chunk=1000, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # first calls outside the capture: per-device set-up
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for r in range(3):
        A = synth.int_uniform_bf16(950 + r, (M, K))
        A_in.copy_(to_device_bf16(A))
        g.replay()
        torch.cuda.synchronize()
        lib.ts_sync_and_check()
        want = oracle.bf16_rne(oracle.gemm_f64(A, B))
        assert np.array_equal(bf16_bits(D), want), f"replay {r}: GEMM"
        assert np.array_equal(rows_out.cpu().numpy().view(np.uint16).reshape(M, N), want), f"replay {r}: copies"


# inputs_ready = 1: the caller states that A, B (and the skip mask) were final before the previous
# kernel in the stream began; every task but the epilogue then runs its first work unit ahead of the
# dependent-launch barrier, and the epilogue waits on it before writing anything.  The chains below
# keep that contract.

@pytest.mark.parametrize("tile,sched", [("128x256", "clc"), ("128x256", "static"), ("256x256", "clc"),
                                        ("256x256", "static"), ("128x128", "clc")])
def test_inputs_ready_gemms_overwrite_in_stream_order(lib, tile, sched):
    # back-to-back GEMMs on operands that nothing writes, all into the same D: the early loads
    # overlap the previous launch, but the last launch's values remain (write after write)
    M, N, K = 2048, 2048, 64
    A1, A2 = synth.int_uniform_bf16(961, (M, K)), synth.int_uniform_bf16(962, (M, K))
    B = synth.int_uniform_bf16(963, (N, K))
    d_a1, d_a2, d_b = to_device_bf16(A1), to_device_bf16(A2), to_device_bf16(B)
    D = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(6):
        lib.ts_gemm_bf16_ex(d_a1, d_b, D, sched=sched, tile=tile, inputs_ready=1)
        lib.ts_gemm_bf16_ex(d_a2, d_b, D, sched=sched, tile=tile, inputs_ready=1)
    lib.ts_sync_and_check()
    assert_bit_exact(D, oracle.gemm_f64(A2, B), f"inputs_ready write after write {tile} {sched}")


@pytest.mark.parametrize("tile,sched", [("128x256", "static"), ("256x256", "clc")])
def test_inputs_ready_mixed_chain(lib, tile, sched):
    # D1 = A B^T (A, B static: ready), D2 = D1 C^T (D1 written by the previous kernel: not ready),
    # D3 = A E^T (ready), D4 = D2 E^T (D2 was written while D3's predecessor ran: not ready)
    M, K = 1024, 128
    A = synth.int_uniform_bf16(971, (M, K))
    B = synth.one_hot_rows_bf16(K, K, np.random.default_rng(7).permutation(K))
    C = synth.one_hot_rows_bf16(K, K, np.random.default_rng(8).permutation(K))
    E = synth.int_uniform_bf16(973, (256, K))
    d_a, d_b, d_c, d_e = (to_device_bf16(x) for x in (A, B, C, E))
    D1 = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    D2 = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    D3 = torch.full((M, 256), float("nan"), dtype=torch.float32, device="cuda")
    D4 = torch.full((M, 256), float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        lib.ts_gemm_bf16_ex(d_a, d_b, D1, sched=sched, tile=tile, inputs_ready=1)
        lib.ts_gemm_bf16_ex(D1, d_c, D2, sched=sched, tile=tile)
        lib.ts_gemm_bf16_ex(d_a, d_e, D3, sched=sched, tile=tile, inputs_ready=1)
        lib.ts_gemm_bf16_ex(D2, d_e, D4, sched=sched, tile=tile)
    lib.ts_sync_and_check()
    d1 = oracle.bf16_rne(oracle.gemm_f64(A, B))
    assert np.array_equal(bf16_bits(D1), d1)
    d2 = oracle.bf16_rne(oracle.gemm_f64(d1, C))
    assert np.array_equal(bf16_bits(D2), d2)
    assert_bit_exact(D3, oracle.gemm_f64(A, E), "D3")
    assert_bit_exact(D4, oracle.gemm_f64(d2, E), f"inputs_ready chain {tile} {sched}")


@pytest.mark.parametrize("sched", ["static", "clc"])
def test_inputs_ready_with_split_tiles_row_sums_skip_and_trace(lib, sched):
    # every output a task writes waits for the previous kernel: split partials and counters (2-CTA,
    # planned split), the Fork task's row sums, D around a skip mask, and the producer's trace
    M, N, K = 2560, 2560, 8192
    A = synth.int_uniform_bf16(981, (M, K))
    B = synth.int_uniform_bf16(982, (N, K))
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    ref = oracle.gemm_f64_blas(A, B)
    info = lib.ts_gemm_launch_info(M, N, K, lib.TS_OUT_F32, sched, tile="256x256")
    assert info["split_tiles"] > 0
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        lib.ts_gemm_bf16_ex(Ad, Bd, D, sched=sched, tile="256x256", inputs_ready=1)
    lib.ts_sync_and_check()
    assert_bit_exact(D, ref, f"inputs_ready split tiles {sched}")

    Ms, Ks = 1024, 1024
    As = synth.int_uniform_bf16(983, (Ms, Ks))
    Bs = synth.int_uniform_bf16(984, (N, Ks))
    R = torch.full((Ms,), float("nan"), dtype=torch.float32, device="cuda")
    Dr = torch.full((Ms, N), float("nan"), dtype=torch.float32, device="cuda")
    lib.ts_gemm_bf16_ex(to_device_bf16(As), to_device_bf16(Bs), Dr, sched=sched, tile="128x256", row_sums=R,
                        inputs_ready=1)
    lib.ts_sync_and_check()
    assert_bit_exact(Dr, oracle.gemm_f64(As, Bs), "inputs_ready with row sums: D")
    assert np.array_equal(R.cpu().numpy().astype(np.float64), oracle.row_sums_f64(As, [0, Ks])[0])

    tiles_m, tiles_n = Ms // 128, N // 256
    skip = torch.from_numpy((np.arange(tiles_m * tiles_n) % 3 == 1).astype(np.uint8)).cuda()
    Dk = torch.full((Ms, N), -1.0, dtype=torch.float32, device="cuda")
    trace = torch.zeros(4 * tiles_m * tiles_n, dtype=torch.int64, device="cuda")
    lib.ts_gemm_bf16_ex(to_device_bf16(As), to_device_bf16(Bs), Dk, sched=sched, tile="128x256", skip_tiles=skip,
                        trace=trace, inputs_ready=1)
    lib.ts_sync_and_check()
    want = oracle.gemm_f64(As, Bs).astype(np.float32)
    keep = np.repeat(np.repeat(skip.cpu().numpy().reshape(tiles_m, tiles_n) != 0, 128, 0), 256, 1)
    want[keep] = -1.0
    assert np.array_equal(Dk.cpu().numpy(), want)
    tr = trace.view(-1, 4).cpu().numpy()
    assert np.all(tr[:, 0] == 1)
    # a computed tile's epilogue ends after its producer began it; a skipped tile moves no data
    # between the two, so its stamps are not ordered
    mb, nb = lib.ts_gemm_tile_coords(Ms, N, Ks, lib.TS_OUT_F32, sched, tile="128x256")
    computed = skip.cpu().numpy()[mb * tiles_n + nb] == 0
    assert computed.any() and np.all(tr[computed, 3] >= tr[computed, 2])


def test_inputs_ready_waits_do_not_time_out_behind_a_long_kernel(lib):
    # A long static GEMM on half of the SMs lets the next launch start beside it.  That launch (8
    # units on each of 8 workers) runs each role's first unit ahead of its dependent-launch
    # barrier; every wait that depends on the epilogue (the MMA's third unit needs an accumulator
    # back) comes after the role's own wait on the barrier, so none of the 0.1 ms wait limits is
    # reached while the first launch runs, and both results are exact.
    M = N = 8192
    K = 4096
    A = synth.int_uniform_bf16(991, (M, K))
    B = synth.int_uniform_bf16(992, (N, K))
    Ms, Ns, Ks = 1024, 2048, 512
    As = synth.int_uniform_bf16(993, (Ms, Ks))
    Bs = synth.int_uniform_bf16(994, (Ns, Ks))
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    Ds = torch.full((Ms, Ns), float("nan"), dtype=torch.float32, device="cuda")
    Ad, Bd, Asd, Bsd = (to_device_bf16(x) for x in (A, B, As, Bs))
    half = lib.ts_num_sms() // 2

    def long_gemm():
        lib.ts_gemm_bf16_ex(Ad, Bd, D, sched="static", tile="128x256", max_workers=half, workspace=None)

    long_gemm()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    long_gemm()
    e1.record()
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) > 0.3  # ms: far longer than the 0.1 ms limit below
    info = lib.ts_gemm_launch_info(Ms, Ns, Ks, lib.TS_OUT_F32, "static", tile="128x256", max_workers=8)
    assert info["workers"] == 8 and info["num_units"] >= 3 * 8
    long_gemm()
    lib.ts_gemm_bf16_ex(Asd, Bsd, Ds, sched="static", tile="128x256", max_workers=8, timeout_s=1e-4,
                        inputs_ready=1)
    torch.cuda.synchronize()
    lib.ts_sync_and_check()
    assert_bit_exact(Ds, oracle.gemm_f64(As, Bs), "the launch behind the long one")
    assert_bit_exact(D, oracle.gemm_f64_blas(A, B), "the long launch")
