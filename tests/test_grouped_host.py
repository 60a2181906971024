"""The grouped GEMM's unit order (host only, no GPU): groups longest K range first."""
import numpy as np
import pytest


def _lpt(off):
    # longest processing time first, ties in index order (Graham's LPT list order)
    G = len(off) - 1
    return sorted(range(G), key=lambda g: (-(off[g + 1] - off[g]), g))


@pytest.mark.parametrize("off", [
    [0, 64],
    [0, 64, 64, 320, 448, 1024],            # 64, 0, 256, 128, 576 columns
    [128, 256, 640],                        # offsets not starting at 0
    [0, 0, 0, 0],                           # every group empty: index order
    [0, 128, 256, 384, 512],                # all equal: index order
])
def test_order_is_longest_first_ties_by_index(ts, off):
    assert list(ts.ts_gemm_grouped_order(off)) == _lpt(off)


def test_order_of_random_and_maximal_group_counts(ts):
    rng = np.random.default_rng(0x0D3)
    for G in (1, 2, 17, 255, 256):
        for _ in range(5):
            widths = 64 * rng.choice([0, 1, 2, 3, 50, 127], size=G)  # many ties
            off = [int(x) for x in np.concatenate([[0], np.cumsum(widths)])]
            order = ts.ts_gemm_grouped_order(off)
            assert sorted(order) == list(range(G))
            assert list(order) == _lpt(off)
            lengths = np.diff(off)[order]
            assert np.all(lengths[:-1] >= lengths[1:])


def test_order_rejects_what_the_grouped_gemm_rejects(ts):
    with pytest.raises(ts.TsError):
        ts.ts_gemm_grouped_order([0, 128, 64])  # decreasing
    with pytest.raises(ts.TsError):
        ts.ts_gemm_grouped_order([0, 100])  # not a multiple of 64
    with pytest.raises(ts.TsError):
        ts.ts_gemm_grouped_order([0] * 258)  # 257 groups
    off = np.array([0, 64], dtype=np.int64)
    assert ts._lib.ts_gemm_grouped_order(1, off.ctypes.data, None) == ts.TS_ERR_INVALID_ARG


def test_lpt_order_shortens_the_simulated_schedule():
    # list scheduling of the benchmark's 16 skewed groups (64 tiles each) on 76 workers, each unit
    # costing its k-blocks plus 2 of overhead: the longest-first order ends sooner than index
    # order, both for greedy (CLC-like) assignment and for the static round-robin deal
    import heapq

    import synth

    off = synth.GROUPED.k_offsets()
    kb = [(off[g + 1] - off[g]) // 64 for g in range(len(off) - 1)]

    def greedy(order):
        h = [0.0] * 76
        for g in order:
            for _ in range(64):
                heapq.heappush(h, heapq.heappop(h) + kb[g] + 2)
        return max(h)

    def round_robin(order):
        loads = [0.0] * 76
        units = [kb[g] + 2 for g in order for _ in range(64)]
        for i, u in enumerate(units):
            loads[i % 76] += u
        return max(loads)

    natural, lpt = list(range(len(kb))), _lpt(off)
    assert greedy(lpt) < greedy(natural) and round_robin(lpt) < round_robin(natural)
