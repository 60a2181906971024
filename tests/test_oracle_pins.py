"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test ties one oracle function to something independent: hand-derived
bf16 bit patterns, a library conversion routine, exact rational arithmetic,
closed forms (identity / one-hot / integer products), or the worked example
printed in "Cluster Launch Control".  The ``planted`` tests feed the pins a
deliberately wrong variant of the oracle to show that they would catch it.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_value(tok: str) -> float:
    if tok in ("inf", "-inf", "nan"):
        return float(tok)
    return float.fromhex(tok)


def _golden_bf16():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_rne.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split(None, 2)
            rows.append((parts[0], _parse_value(parts[0]), int(parts[1], 16), parts[2]))
    return rows


# --------------------------------------------------------------- generator
def test_splitmix64_published_first_output():
    # SplitMix64 seeded with 0: first output 0xE220A8397B1DCDAF (reference
    # implementation by Vigna, splitmix64.c).
    assert int(synth.splitmix64(0, 1)[0]) == 0xE220A8397B1DCDAF


def test_c_generator_matches_numpy_reference_form():
    assert np.array_equal(synth.splitmix64(5, 1000, offset=37), synth.splitmix64_fast(5, 1000, offset=37))


def test_uniform_range_and_exactness():
    a = synth.uniform_pm1_bf16(7, (64, 64))
    v = oracle.bf16_to_f64(a)
    assert v.min() >= -1.0 and v.max() <= 1.0
    assert abs(v.mean()) < 0.05


# ------------------------------------------------------------------- bf16
@pytest.mark.parametrize("tok,value,bits,reason", _golden_bf16(), ids=lambda x: str(x)[:24])
def test_bf16_rne_golden(tok, value, bits, reason):
    assert oracle.bf16_rne_scalar(value) == bits, reason


def test_bf16_rne_matches_library_conversion():
    # torch's float32 -> bfloat16 conversion rounds to nearest even; on
    # float32 inputs (exact in float64) the oracle must agree bit for bit.
    import torch

    rng = np.random.default_rng(1)
    raw = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    f = raw.view(np.float32)
    f = f[np.isfinite(f)]
    lib = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = oracle.bf16_rne(f.astype(np.float64))
    assert np.array_equal(lib, mine)


def test_bf16_decode_encode_roundtrip_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = oracle.bf16_to_f64(bits)
    back = oracle.bf16_rne(v)
    nan = np.isnan(v)
    assert np.array_equal(back[~nan], bits[~nan])
    assert np.all((back[nan] & 0x7FFF) == 0x7FC0)


def test_bf16_decode_closed_form():
    # bit pattern s|e|m  ->  (-1)^s * 2^(e-127) * (1 + m/128) for normal e
    for b in (0x3F80, 0x4049, 0xC2F7, 0x0080, 0x7F7F):
        s, e, m = b >> 15, (b >> 7) & 0xFF, b & 0x7F
        want = (-1) ** s * 2.0 ** (e - 127) * (1 + m / 128)
        assert oracle.bf16_to_f64(np.array([b], np.uint16))[0] == want


# ------------------------------------------------------------------- GEMM
def _exact_gemm(A_bits, B_bits):
    a = [[Fraction(float(x)) for x in row] for row in oracle.bf16_to_f64(A_bits)]
    b = [[Fraction(float(x)) for x in row] for row in oracle.bf16_to_f64(B_bits)]
    return [[sum(ai[k] * bj[k] for k in range(len(ai))) for bj in b] for ai in a]


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 1), (3, 5, 7, 2), (8, 8, 16, 3), (5, 2, 13, 4)])
def test_gemm_against_exact_rationals(M, N, K, seed):
    A = synth.uniform_pm1_bf16(seed, (M, K))
    B = synth.normal_bf16(seed + 50, (N, K), 3.0)
    exact = _exact_gemm(A, B)
    D = oracle.gemm_f64(A, B)
    S = oracle.gemm_f64(A, B, absolute=True)
    for i in range(M):
        for j in range(N):
            err = abs(Fraction(D[i, j]) - exact[i][j])
            assert err <= Fraction(K * 2.0 ** -52) * Fraction(S[i, j]) + Fraction(2.0 ** -1074)


def test_gemm_identity_b_returns_a():
    M, K = 37, 48
    A = synth.uniform_pm1_bf16(11, (M, K))
    Bid = synth.one_hot_rows_bf16(K, K, np.arange(K))
    D = oracle.gemm_f64(A, Bid)
    assert np.array_equal(D, oracle.bf16_to_f64(A))


def test_gemm_one_hot_selects_columns():
    # B[j, k] = [k == c_j]  =>  D[i, j] = A[i, c_j]; non-square, so a swapped
    # operand or a transposed index cannot pass.
    M, N, K = 9, 13, 21
    rng = np.random.default_rng(5)
    cols = rng.integers(0, K, size=N)
    A = synth.uniform_pm1_bf16(12, (M, K))
    B = synth.one_hot_rows_bf16(N, K, cols)
    D = oracle.gemm_f64(A, B)
    assert np.array_equal(D, oracle.bf16_to_f64(A)[:, cols])


def test_gemm_integer_matches_integer_matmul():
    M, N, K = 33, 29, 70
    A = synth.int_uniform_bf16(21, (M, K))
    B = synth.int_uniform_bf16(22, (N, K))
    ai = oracle.bf16_to_f64(A).astype(np.int64)
    bi = oracle.bf16_to_f64(B).astype(np.int64)
    D = oracle.gemm_f64(A, B)
    assert np.array_equal(D, (ai @ bi.T).astype(np.float64))


def test_gemm_blas_route_matches_loop():
    A = synth.uniform_pm1_bf16(31, (64, 200))
    B = synth.uniform_pm1_bf16(32, (48, 200))
    D1 = oracle.gemm_f64(A, B)
    D2 = oracle.gemm_f64_blas(A, B)
    S = oracle.gemm_f64(A, B, absolute=True)
    assert np.all(np.abs(D1 - D2) <= 200 * 2.0 ** -52 * S)
    assert np.allclose(oracle.gemm_f64_blas(A, B, absolute=True), S, rtol=1e-13, atol=0)


def test_gemm_row_subset_and_entries_agree_with_full():
    A = synth.uniform_pm1_bf16(41, (20, 30))
    B = synth.uniform_pm1_bf16(42, (17, 30))
    D = oracle.gemm_f64(A, B)
    assert np.array_equal(oracle.gemm_f64(A, B, rows=(5, 12)), D[5:12])
    ii = np.array([0, 19, 7, 3])
    jj = np.array([16, 0, 8, 3])
    e, ea = oracle.gemm_entries_f64(A, B, ii, jj)
    assert np.array_equal(e, D[ii, jj])
    assert np.array_equal(ea, oracle.gemm_f64(A, B, absolute=True)[ii, jj])


def test_gemm_k_zero_is_zero():
    A = np.zeros((4, 0), np.uint16)
    B = np.zeros((3, 0), np.uint16)
    assert np.array_equal(oracle.gemm_f64(A, B), np.zeros((4, 3)))


def test_grouped_single_group_is_the_plain_gemm():
    A = synth.uniform_pm1_bf16(51, (17, 128))
    B = synth.uniform_pm1_bf16(52, (13, 128))
    assert np.array_equal(oracle.grouped_gemm_f64(A, B, [0, 128])[0], oracle.gemm_f64(A, B))


def test_grouped_groups_sum_to_the_full_product():
    # linearity over disjoint K slices (integer inputs: every sum is exact)
    A = synth.int_uniform_bf16(53, (19, 448))
    B = synth.int_uniform_bf16(54, (11, 448))
    off = [0, 64, 64, 256, 448]
    D = oracle.grouped_gemm_f64(A, B, off)
    assert np.array_equal(D.sum(axis=0), oracle.gemm_f64(A, B))
    assert np.array_equal(D[1], np.zeros((19, 11)))  # the empty group


def test_grouped_slices_match_integer_matmul():
    A = synth.int_uniform_bf16(55, (9, 320))
    B = synth.int_uniform_bf16(56, (7, 320))
    off = [64, 128, 320]
    ai = oracle.bf16_to_f64(A).astype(np.int64)
    bi = oracle.bf16_to_f64(B).astype(np.int64)
    D = oracle.grouped_gemm_f64(A, B, off)
    for g in range(2):
        k0, k1 = off[g], off[g + 1]
        assert np.array_equal(D[g], (ai[:, k0:k1] @ bi[:, k0:k1].T).astype(np.float64))
    assert np.array_equal(oracle.grouped_gemm_f64(A, B, off, blas=True), D)


def test_row_sums_equal_a_product_with_a_row_of_ones():
    # sum_k a[i, k] = (A . 1^T)[i]: the row sums are the GEMM against a row of ones
    A = synth.uniform_pm1_bf16(57, (23, 192))
    ones = np.full((1, 192), 0x3F80, np.uint16)
    R = oracle.row_sums_f64(A, [0, 192])
    D = oracle.gemm_f64(A, ones)
    assert np.all(np.abs(R[0] - D[:, 0]) <= 192 * 2.0 ** -52 * oracle.gemm_f64(A, ones, absolute=True)[:, 0])


def test_row_sums_integer_groups_exact():
    A = synth.int_uniform_bf16(58, (11, 256))
    ai = oracle.bf16_to_f64(A).astype(np.int64)
    R = oracle.row_sums_f64(A, [0, 64, 64, 256])
    assert np.array_equal(R[0], ai[:, :64].sum(1)) and np.array_equal(R[2], ai[:, 64:].sum(1))
    assert np.array_equal(R[1], np.zeros(11))


# ------------------------------------------------------------------- copy
@pytest.mark.parametrize("n", [0, 1, 7, 8, 1000, 4097])
def test_copy_is_identity(n):
    src = synth.int16_uniform(99 + n, n)
    assert np.array_equal(oracle.copy_i16(src), src)


def _golden_rows():
    meta, cases = {}, []
    with open(os.path.join(GOLDEN, "copy_rows_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, vals = line.split(":")
            if key.startswith("case"):
                _, rows, mode = key.split()
                cases.append((int(rows), mode == "skip", np.array(vals.split(), dtype=np.int16)))
            else:
                meta[key] = np.array(vals.split(), dtype=np.int64)
    return meta, cases


def test_copy_rows_golden():
    meta, cases = _golden_rows()
    n = int(meta["n"][0])
    for rows, use_skip, want in cases:
        got, bad = oracle.copy_rows_i16(meta["src"].astype(np.int16), np.full(n, -1, np.int16), meta["offsets"],
                                        rows, meta["skip"] if use_skip else None)
        assert bad == -1
        assert np.array_equal(got, want), (rows, use_skip, got)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_copy_rows_over_a_partition_is_the_plain_copy(seed):
    # rows that tile [0, n) exactly, none skipped: the jagged copy is the whole copy
    rng = np.random.default_rng(seed)
    n = 5000
    cuts = np.sort(rng.integers(0, n + 1, size=40))
    offsets = np.concatenate([[0], cuts, [n]])
    src = synth.int16_uniform(300 + seed, n)
    got, bad = oracle.copy_rows_i16(src, np.zeros(n, np.int16), offsets)
    assert bad == -1 and np.array_equal(got, oracle.copy_i16(src))


def test_copy_rows_skipping_everything_changes_nothing():
    src = synth.int16_uniform(7, 100)
    dst0 = synth.int16_uniform(8, 100)
    offsets = np.array([0, 10, 50, 100])
    got, _ = oracle.copy_rows_i16(src, dst0, offsets, skip=np.ones(3, np.uint8))
    assert np.array_equal(got, dst0)
    got, _ = oracle.copy_rows_i16(src, dst0, offsets, rows=0)
    assert np.array_equal(got, dst0)


def test_copy_rows_reports_the_first_invalid_row():
    src = np.arange(1, 11, dtype=np.int16)
    # row 1 decreases, row 2 ends past n; row 0 is still copied
    got, bad = oracle.copy_rows_i16(src, np.zeros(10, np.int16), [1, 3, 2, 11])
    assert bad == 1 and np.array_equal(got, [0, 2, 3, 0, 0, 0, 0, 0, 0, 0])
    assert oracle.copy_rows_i16(src, np.zeros(10, np.int16), [-1, 3])[1] == 0
    assert oracle.copy_rows_i16(src, np.zeros(10, np.int16), [0, 10, 11])[1] == 1


# ------------------------------------------------------------- scheduling
def test_static_schedule_worked_example():
    want = {}
    with open(os.path.join(GOLDEN, "static_schedule_12x4.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                w, tiles = line.split(":")
                want[int(w)] = [int(t) for t in tiles.split()]
    got = oracle.static_schedule(12, 4)
    assert got == [want[w] for w in range(4)]


@pytest.mark.parametrize("tiles,workers", [(1, 1), (5, 8), (152, 152), (1000, 148), (7, 3)])
def test_static_schedule_partitions_tiles(tiles, workers):
    sched = oracle.static_schedule(tiles, workers)
    flat = sorted(t for w in sched for t in w)
    assert flat == list(range(tiles))
    for w, ts in enumerate(sched):
        assert ts == list(range(w, tiles, workers))


def test_clc_coverage_checker():
    owner = np.array([0, 1, 2, 0, 1, 0])
    assert oracle.clc_coverage_ok(np.ones(6), owner)[0]
    assert not oracle.clc_coverage_ok(np.array([1, 1, 2, 1, 1, 1]), owner)[0]
    assert not oracle.clc_coverage_ok(np.array([1, 1, 0, 1, 1, 1]), owner)[0]
    # worker 3 ran but did not start on tile 3
    assert not oracle.clc_coverage_ok(np.ones(6), np.array([0, 1, 2, 1, 3, 0]))[0]


# ------------------------------------------------- planted mistakes (CPU)
def _wrong_transposed(A, B):
    # reads B as [K, N] (a swapped operand) -- only defined when shapes allow
    a = oracle.bf16_to_f64(A)
    b = oracle.bf16_to_f64(B).reshape(-1)[: a.shape[1] * B.shape[0]].reshape(a.shape[1], B.shape[0])
    return a @ b


def _wrong_dropped_last_k(A, B):
    return oracle.gemm_f64(A[:, :-1], B[:, :-1])


def _wrong_sign(A, B):
    return -oracle.gemm_f64(A, B)


@pytest.mark.parametrize("wrong", [_wrong_transposed, _wrong_dropped_last_k, _wrong_sign])
def test_planted_mistakes_fail_the_pins(wrong):
    M, N, K = 9, 13, 21
    rng = np.random.default_rng(5)
    cols = rng.integers(0, K, size=N)
    A = synth.int_uniform_bf16(12, (M, K))
    B = synth.one_hot_rows_bf16(N, K, cols)
    want = oracle.bf16_to_f64(A)[:, cols]
    assert not np.array_equal(wrong(A, B), want)


def test_planted_bad_rounding_fails_golden():
    # truncation instead of round-to-nearest-even
    def trunc(x):
        f = np.array([x], np.float32).view(np.uint32)[0]
        return int(f >> 16)

    mism = [tok for tok, v, bits, _ in _golden_bf16() if not math.isnan(v) and trunc(v) != bits]
    assert mism, "the golden cases must distinguish RNE from truncation"


@pytest.mark.parametrize("wrong", ["inclusive_end", "ignores_skip", "ignores_row_count"])
def test_planted_row_copy_mistakes_fail_golden(wrong):
    meta, cases = _golden_rows()
    src, off, skip = meta["src"].astype(np.int16), meta["offsets"], meta["skip"]

    def variant(rows, use_skip):
        d = np.full(src.size, -1, np.int16)
        for r in range(off.size - 1 if wrong == "ignores_row_count" else rows):
            if use_skip and skip[r] and wrong != "ignores_skip":
                continue
            e = off[r + 1] + (1 if wrong == "inclusive_end" else 0)
            d[off[r]:min(e, src.size)] = src[off[r]:min(e, src.size)]
        return d

    assert any(not np.array_equal(variant(rows, use_skip), want) for rows, use_skip, want in cases)
