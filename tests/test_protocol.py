"""The host-side barrier-protocol checker (no GPU needed).

The kernel's role loops, modelled with the arrival counts the kernel itself
uses (ts_gemm_protocol_info), must be free of deadlocks and races for every
compiled variant and both schedulers; every planted protocol mistake must be
caught; and the engine's mbarrier semantics are pinned on tiny hand-written
programs.
"""
import itertools

import pytest

from tile_scheduling_gb300 import protocol as pc

OP = pc


@pytest.fixture(scope="module")
def ts():
    import tile_scheduling_gb300 as ts

    return ts


# ------------------------------------------------------------ engine semantics
def _prog(bars, roles, nbufs=1):
    P = pc.Program()
    for i, n in enumerate(bars):
        P.bar(f"b{i}", n)
    for i in range(nbufs):
        P.buf(f"x{i}")
    for name, ops in roles:
        P.roles.append((name, None, [list(o) + [-1] * (8 - len(o)) for o in ops]))
    return P


def test_engine_fresh_barrier_passes_parity_one_only():
    ok = _prog([1], [("r", [(OP.OP_WAIT, 0, 1)])])
    assert pc.check(ok).ok
    stuck = _prog([1], [("r", [(OP.OP_WAIT, 0, 0)])])
    r = pc.check(stuck)
    assert not r.ok and "deadlock" in r.message


def test_engine_transaction_bytes_may_land_before_expect_tx():
    # the copy's complete-tx can overtake the expect-tx; the phase still completes once
    prog = _prog([1], [("producer", [(OP.OP_TMA, 0, 7, 0, 64), (OP.OP_ARRIVE, 0, 64)]),
                       ("consumer", [(OP.OP_WAIT, 0, 0), (OP.OP_TREAD, 0, 7)])])
    assert pc.check(prog).ok


def test_engine_reports_reading_before_the_copy_landed():
    prog = _prog([1], [("producer", [(OP.OP_ARRIVE, 0, 0), (OP.OP_TMA, 0, 7, 0, 0)]),
                       ("consumer", [(OP.OP_WAIT, 0, 0), (OP.OP_TREAD, 0, 7)])])
    r = pc.check(prog)
    assert not r.ok and "read of x0" in r.message


def test_engine_reports_over_arrival():
    prog = _prog([1], [("a", [(OP.OP_ARRIVE, 0, 5)]), ("b", [(OP.OP_ARRIVE, 0, 0)])])
    r = pc.check(prog)
    assert not r.ok and "more arrivals" in r.message


# ------------------------------------------------------------ kernel protocol
def test_exported_counts_match_the_role_structure(ts):
    for tile, out, ew in itertools.product(("128x128", "128x256", "256x256"), (ts.TS_OUT_BF16, ts.TS_OUT_F32), (4, 8)):
        p = ts.ts_gemm_protocol_info(tile, out, ew)
        cg, e = p["cluster"], p["epilogue_warps"]
        assert e == ew
        assert p["tx_bytes"] == p["stage_bytes"] * cg
        assert p["tmem_empty_arrivals"] == e * cg
        # producer, MMA, scheduler and epilogue warps of the even CTA; producer,
        # scheduler and epilogue warps of the odd CTA
        assert p["clc_empty_arrivals"] == (3 + e) + (2 + e if cg == 2 else 0)
        assert p["full_arrivals"] == p["empty_arrivals"] == p["tmem_full_arrivals"] == 1


@pytest.mark.parametrize("tile", ["128x128", "128x256", "256x256"])
@pytest.mark.parametrize("units", [[1], [2, 3], [3, 1, 2]])
def test_static_protocol_verified(tile, units):
    r = pc.check_variant(tile, units, "static", stages=2)
    assert r.ok, r.message


@pytest.mark.parametrize("tile", ["128x256", "256x256"])
def test_static_protocol_verified_at_the_kernels_ring_depth(tile):
    r = pc.check_variant(tile, [2, 3], "static")
    assert r.ok, r.message


@pytest.mark.parametrize("units", [[1], [2, 1], [1, 2, 1]])
def test_clc_protocol_verified_one_cta(units):
    r = pc.check_variant("128x256", units, "clc")
    assert r.ok, r.message


@pytest.mark.parametrize("units", [[1], [2, 1], [1, 1, 2]])
def test_clc_protocol_verified_cta_pair(units):
    # one epilogue warp per CTA modelled; the barriers expect the others' arrivals fewer
    r = pc.check_variant("256x256", units, "clc", stages=2, epilogue_warps=1)
    assert r.ok, r.message


@pytest.mark.slow
def test_clc_protocol_verified_cta_pair_two_epilogue_warps_per_cta():
    # two epilogue warps per CTA of the pair, interleaved with each other and with the odd
    # CTA's: ~9.6 million states, about 10 s
    r = pc.check_variant("256x256", [1, 1], "clc", stages=2, epilogue_warps=2, max_states=30_000_000)
    assert r.ok, r.message


@pytest.mark.exhaustive
def test_merge_protocol_verified_cta_pair_two_units():
    # the Merge layout on the CTA pair under CLC, two one-k-block units: ~4.1e7 states, about a
    # minute (run with --exhaustive)
    r = pc.check_variant("256x256", [1, 1], "clc", stages=2, epilogue_warps=1, variant_merge=1,
                         max_states=100_000_000)
    assert r.ok, r.message


@pytest.mark.exhaustive
def test_clc_protocol_verified_cta_pair_three_epilogue_warps_per_cta():
    # three epilogue warps per CTA of the pair: ~1.2e8 states, about 5 minutes and 4 GB of host
    # memory (run with --exhaustive)
    r = pc.check_variant("256x256", [1, 1], "clc", stages=2, epilogue_warps=3, max_states=150_000_000)
    assert r.ok, r.message


@pytest.mark.parametrize("mutation", [m for m in pc.MUTATIONS
                                      if not m.startswith(("fork", "merge")) and m not in pc.ZERO_K_MUTATIONS])
@pytest.mark.parametrize("tile,sched,warps", [("128x256", "clc", None), ("256x256", "clc", 1),
                                              ("256x256", "static", 2)])
def test_planted_mistakes_are_caught(mutation, tile, sched, warps):
    r = pc.check_variant(tile, [2, 1, 2], sched, stages=2, epilogue_warps=warps, mutate=mutation)
    if mutation == "clc_empty_count_low" and sched == "static":
        assert r.ok  # the static scheduler never touches the CLC barriers
    else:
        assert not r.ok and r.status == 1, (mutation, r)


@pytest.mark.parametrize("sched", ["static", "clc"])
@pytest.mark.parametrize("tile", ["128x128", "128x256"])
def test_fork_protocol_verified(tile, sched):
    # the ring's second consumer (row sums of A) beside the MMA issuer
    r = pc.check_variant(tile, [2, 1, 2], sched, stages=2, fork=True)
    assert r.ok, r.message


@pytest.mark.parametrize("sched", ["static", "clc"])
def test_fork_mistake_is_caught(sched):
    r = pc.check_variant("128x256", [2, 1, 2], sched, stages=2, fork=True,
                         mutate="fork_producer_ignores_second_consumer")
    assert not r.ok and r.status == 1, r


def test_fork_exports_its_arrivals(ts):
    assert ts.ts_gemm_protocol_info("128x256", 0)["aux_empty_arrivals"] == 1
    with pytest.raises(ValueError):
        pc.build_program(ts.ts_gemm_protocol_info("256x256", 0), [1], fork=True)


def test_protocol_info_epilogue_warp_choices(ts):
    assert ts.ts_gemm_protocol_info("128x256", 0)["epilogue_warps"] == 4  # 0 = the four-warp variant
    with pytest.raises(ts.TsError):
        ts.ts_gemm_protocol_info("128x256", 0, 6)
    with pytest.raises(ts.TsError):
        ts.ts_gemm_protocol_info("128x128", 0, 16)  # sixteen only on 256-column tiles
    for tile, out in itertools.product(("128x256", "256x256"), (ts.TS_OUT_BF16, ts.TS_OUT_F32)):
        p, p8 = ts.ts_gemm_protocol_info(tile, out, 16), ts.ts_gemm_protocol_info(tile, out, 8)
        cg = p["cluster"]
        assert p["epilogue_warps"] == 16 and p["tmem_empty_arrivals"] == 16 * cg
        assert p["clc_empty_arrivals"] == p8["clc_empty_arrivals"] + 8 * cg
        # 64 KB of staging instead of 32 KB: one stage fewer
        assert p["stages"] == p8["stages"] - 1


# Eight epilogue warps: two per TMEM lane quarter, each releasing the
# accumulator after its own subtiles.  Each warp still runs one read and one
# release per unit, so the model is the same with twice the arrivals expected;
# models of fewer warps count the rest as arrived.
@pytest.mark.parametrize("tile,sched,warps,units", [("128x256", "clc", 2, [2, 1]), ("128x128", "static", 3, [1, 2]),
                                                    ("256x256", "clc", 1, [1, 2]), ("256x256", "static", 2, [2, 1])])
def test_eight_warp_protocol_verified(tile, sched, warps, units):
    r = pc.check_variant(tile, units, sched, stages=2, variant_epi_warps=8, epilogue_warps=warps)
    assert r.ok, r.message


@pytest.mark.parametrize("mutation", ["epilogue_release_before_read", "tmem_empty_count_low"])
def test_eight_warp_planted_mistakes_are_caught(mutation):
    assert mutation in pc.MUTATIONS
    r = pc.check_variant("256x256", [2, 1, 2], "clc", stages=2, variant_epi_warps=8, epilogue_warps=1,
                         mutate=mutation)
    assert not r.ok and r.status == 1, (mutation, r)


# Merge barrier layout ("Pipeline Groups", Merge): A and B loaded by two
# producer warps onto their own full barriers, one shared empty barrier, the
# MMA waiting on both.
def test_merge_exports_its_layout(ts):
    for tile, out in itertools.product(("128x128", "128x256", "256x256"), (ts.TS_OUT_BF16, ts.TS_OUT_F32)):
        fused, p = ts.ts_gemm_protocol_info(tile, out, 4, 0), ts.ts_gemm_protocol_info(tile, out, 4, 1)
        cg, e = p["cluster"], p["epilogue_warps"]
        assert fused["merge"] == 0 and p["merge"] == 1 and e == 4
        assert p["a_stage_bytes"] == 128 * 64 * 2  # 128 rows of A, one 128-byte swizzle row each
        assert p["stage_bytes"] == fused["stage_bytes"] and p["stages"] == fused["stages"]
        # the B producer of each CTA consumes every CLC response too
        assert p["clc_empty_arrivals"] == fused["clc_empty_arrivals"] + cg
    with pytest.raises(ts.TsError):
        ts.ts_gemm_protocol_info("128x256", 0, 8, 1)  # Merge is built with four epilogue warps
    with pytest.raises(ts.TsError):
        ts.ts_gemm_protocol_info("128x256", 0, 4, 2)
    with pytest.raises(ValueError):
        pc.build_program(ts.ts_gemm_protocol_info("128x256", 0, 4, 1), [1], fork=True)


@pytest.mark.parametrize("tile,sched,warps,units", [("128x128", "static", None, [2, 1, 2]),
                                                    ("128x256", "clc", None, [2, 1, 2]),
                                                    ("128x128", "clc", 2, [1, 3]),
                                                    ("256x256", "static", 2, [2, 1, 2]),
                                                    ("256x256", "clc", 1, [1]),
                                                    ("256x256", "clc", 1, [3])])
def test_merge_protocol_verified(tile, sched, warps, units):
    r = pc.check_variant(tile, units, sched, stages=2, variant_merge=1, epilogue_warps=warps)
    assert r.ok, r.message


@pytest.mark.parametrize("mutation", [m for m in pc.MUTATIONS if not m.startswith("fork") and m not in pc.ZERO_K_MUTATIONS])
@pytest.mark.parametrize("tile,sched,warps", [("128x256", "clc", 2), ("256x256", "static", 1)])
def test_merge_planted_mistakes_are_caught(mutation, tile, sched, warps):
    r = pc.check_variant(tile, [2, 1, 2], sched, stages=2, variant_merge=1, epilogue_warps=warps, mutate=mutation)
    if mutation == "clc_empty_count_low" and sched == "static":
        assert r.ok
    else:
        assert not r.ok and r.status == 1, (mutation, r)


# Sixteen epilogue warps: four per TMEM lane quarter, each releasing the
# accumulator after its own subtiles; the model keeps a few of them.
@pytest.mark.parametrize("tile,sched,warps,units", [("128x256", "clc", 2, [2, 1]), ("128x256", "static", 3, [1, 2, 1]),
                                                    ("256x256", "clc", 1, [1, 2]), ("256x256", "static", 2, [2, 1])])
def test_sixteen_warp_protocol_verified(tile, sched, warps, units):
    r = pc.check_variant(tile, units, sched, stages=2, variant_epi_warps=16, epilogue_warps=warps)
    assert r.ok, r.message


@pytest.mark.parametrize("mutation", ["epilogue_release_before_read", "tmem_empty_count_high", "clc_empty_count_low"])
def test_sixteen_warp_planted_mistakes_are_caught(mutation):
    r = pc.check_variant("256x256", [2, 1, 2], "clc", stages=2, variant_epi_warps=16, epilogue_warps=1,
                         mutate=mutation)
    assert not r.ok and r.status == 1, (mutation, r)


# --------------------------------------------- units with no k-blocks (skip, K = 0)
# A skipped tile (TS "Schedules", Skippable Tiles) is taken from the queue by every
# role but loads nothing and takes no accumulator; a K = 0 group of a grouped GEMM
# takes an accumulator that the MMA commits with no MMA issued and the epilogue
# reads (discarding it) and releases.
MIXED = [[2, pc.SKIP, 0, 2], [0, 1, pc.SKIP, 1], [pc.SKIP, pc.SKIP, 1, 0, 1], [0, 0, 1], [pc.SKIP, 0, pc.SKIP]]


@pytest.mark.parametrize("units", MIXED)
@pytest.mark.parametrize("tile", ["128x128", "128x256", "256x256"])
@pytest.mark.parametrize("sched", ["static", "clc"])
def test_units_without_k_blocks_verified_on_every_tile(tile, units, sched):
    r = pc.check_variant(tile, units, sched, stages=2, epilogue_warps=1)
    assert r.ok, r.message


@pytest.mark.parametrize("units", MIXED[:2])
@pytest.mark.parametrize("ew", [2, 4])
def test_units_without_k_blocks_verified_with_more_epilogue_warps(units, ew):
    r = pc.check_variant("128x256", units, "clc", stages=2, epilogue_warps=min(ew, 4), variant_epi_warps=ew * 2
                         if ew == 4 else 4)
    assert r.ok, r.message


@pytest.mark.parametrize("units", MIXED[:2])
def test_units_without_k_blocks_verified_fork_and_merge(units):
    assert pc.check_variant("128x256", units, "clc", stages=2, fork=True).ok
    assert pc.check_variant("256x256", units, "static", stages=2, epilogue_warps=1, variant_merge=1).ok


ZERO_K_CASES = {"mma_takes_skipped_accumulator": [1, pc.SKIP, 1, 1], "epilogue_waits_skipped_tile": [1, pc.SKIP, 1],
                "zero_k_mma_no_commit": [1, 0, 1], "zero_k_epilogue_no_release": [0, 1, 1]}


@pytest.mark.parametrize("mutation", pc.ZERO_K_MUTATIONS)
@pytest.mark.parametrize("tile", ["128x128", "128x256", "256x256"])
@pytest.mark.parametrize("sched", ["static", "clc"])
def test_zero_k_mistakes_are_caught(mutation, tile, sched):
    r = pc.check_variant(tile, ZERO_K_CASES[mutation], sched, stages=2, epilogue_warps=1, mutate=mutation)
    assert not r.ok and r.status == 1, (mutation, r)
    # the same sequence without the mistake is clean
    assert pc.check_variant(tile, ZERO_K_CASES[mutation], sched, stages=2, epilogue_warps=1).ok


# ------------------------------------------- the split tiles' counter handoff
@pytest.mark.parametrize("parts", [2, 3, 4])
@pytest.mark.parametrize("launches", [1, 2, 3])
def test_split_handoff_verified(parts, launches):
    r = pc.check(pc.build_split_program(parts, launches))
    assert r.ok, r.message


@pytest.mark.parametrize("mutation", pc.SPLIT_MUTATIONS)
@pytest.mark.parametrize("parts", [2, 3, 4])
def test_split_handoff_mistakes_are_caught(mutation, parts):
    r = pc.check(pc.build_split_program(parts, 2, mutate=mutation))
    assert not r.ok and r.status == 1, (mutation, r)


def test_engine_ticket_counts_reductions_and_rearm():
    # two roles draw tickets 0 and 1 of a counter whose last ticket is 1; the last re-arms
    P = pc.Program()
    c = P.counter(1)
    P.buf("x0")
    P.roles.append(("a", None, [[OP.OP_TICKET, c, 1, 0, 0, 0, 1, -1]]))
    P.roles.append(("b", None, [[OP.OP_TICKET, c, 1, 0, 0, 0, 1, -1]]))
    assert pc.check(P).ok
    P.counters[0] = 2  # expected two reductions: only one happens
    r = pc.check(P)
    assert not r.ok and "after 1 reductions" in r.message


def test_engine_fence_waits_for_own_stores_only():
    # b's fence does not wait for a's store, so b may read x0 before it lands
    P = pc.Program()
    P.buf("x0")
    P.roles.append(("a", None, [[OP.OP_GWRITE, 0, 5, -1, -1, -1, -1, -1], [OP.OP_FENCE] + [-1] * 7]))
    P.roles.append(("b", None, [[OP.OP_FENCE] + [-1] * 7, [OP.OP_TICKET, -1, -1, -1, -1, -1, -1, -1]]))
    P.roles[1] = ("b", None, [[OP.OP_FENCE] + [-1] * 7])
    assert pc.check(P).ok
    c = P.counter(1)
    P.roles[0] = ("a", None, [[OP.OP_GWRITE, 0, 5, -1, -1, -1, -1, -1], [OP.OP_FENCE] + [-1] * 7,
                              [OP.OP_TICKET, c, 0, 0, 1, 5, 1, -1]])
    assert pc.check(P).ok  # a's own fence orders its store before its ticket's read
    P.roles[0] = ("a", None, [[OP.OP_GWRITE, 0, 5, -1, -1, -1, -1, -1], [OP.OP_TICKET, c, 0, 0, 1, 5, 1, -1]])
    r = pc.check(P)
    assert not r.ok and "holding tag -1" in r.message


# ------------------------------------------------- lazy CLC requests (long K loops)
# The scheduler's request k waits until the producer has nearly loaded unit k (a barrier
# the producer arrives on once per unit, `lazy_lead` k-blocks before the unit's end), so
# a worker claims its next unit shortly before it needs it.
@pytest.mark.parametrize("tile,warps,units", [("128x256", None, [2, 1, 2]), ("128x128", None, [1, pc.SKIP, 0, 1]),
                                              ("256x256", 1, [3, 1]), ("256x256", 1, [1, pc.SKIP, 0, 1])])
def test_lazy_clc_protocol_verified(tile, warps, units):
    r = pc.check_variant(tile, units, "clc", stages=2, epilogue_warps=warps, lazy=True)
    assert r.ok, r.message
    # the signal at the first k-block of every unit (a lead as long as the unit)
    r = pc.check_variant(tile, units, "clc", stages=2, epilogue_warps=warps, lazy=True, lazy_lead=8)
    assert r.ok, r.message


def test_lazy_clc_protocol_verified_fork_and_merge():
    assert pc.check_variant("128x256", [2, 1], "clc", stages=2, lazy=True, fork=True).ok
    assert pc.check_variant("128x256", [2, 1], "clc", stages=2, epilogue_warps=2, lazy=True, variant_merge=1).ok


@pytest.mark.parametrize("tile,warps", [("128x256", None), ("256x256", 1)])
def test_lazy_wait_one_unit_late_is_caught(tile, warps):
    # waiting for the producer to begin the *next* unit deadlocks: that unit needs this request
    r = pc.check_variant(tile, [2, 1, 2], "clc", stages=2, epilogue_warps=warps, lazy=True,
                         mutate="lazy_wait_one_unit_late")
    assert not r.ok and "deadlock" in r.message


# ------------------------------------------------ the dependent-launch barrier (inputs_ready)
# The barrier is released as late as possible in these models (once every role that waits on it
# has reached its wait), so a role whose first unit needs the epilogue deadlocks.
@pytest.mark.parametrize("tile,sched,kw", [
    ("128x256", "static", {}),
    ("128x256", "clc", {}),
    ("128x256", "clc", {"lazy": True}),
    ("128x128", "static", {"fork": True}),
    ("256x256", "static", {"variant_merge": 1, "epilogue_warps": 1, "stages": 2}),
])
@pytest.mark.parametrize("units", [[2, 2, 2], [pc.SKIP, 0, 2, 1]])
def test_early_loads_protocol_verified(tile, sched, kw, units):
    r = pc.check_variant(tile, units, sched, early=True, **kw)
    assert r.ok, r.message


def test_early_loads_protocol_verified_cta_pair_clc():
    r = pc.check_variant("256x256", [pc.SKIP, 0, 2, 1], "clc", early=True, stages=2, epilogue_warps=1)
    assert r.ok, r.message


@pytest.mark.parametrize("mutation", pc.EARLY_MUTATIONS)
@pytest.mark.parametrize("tile,sched,kw", [("128x256", "clc", {"stages": 2}),
                                           ("128x256", "clc", {"stages": 2, "lazy": True}),
                                           ("256x256", "static", {"stages": 2, "epilogue_warps": 1})])
def test_early_loads_mistakes_are_caught(mutation, tile, sched, kw):
    if mutation == "scheduler_dep_wait_late" and sched == "static":
        pytest.skip("the static scheduler has no scheduler role")
    r = pc.check_variant(tile, [2, 2, 2, 2], sched, early=True, mutate=mutation, **kw)
    assert not r.ok and "deadlock" in r.message and "dependent_launch" in r.message, r.message


def test_early_mutations_need_early():
    with pytest.raises(ValueError):
        pc.check_variant("128x256", [2, 2, 2], "clc", mutate="mma_dep_wait_late")


@pytest.mark.parametrize("tile", ["128x128", "128x256", "256x256"])
@pytest.mark.parametrize("early", [False, True])
def test_nonpersistent_shape_protocol_verified(tile, early):
    # the non-persistent shape: one unit per CTA (pair), no queue -- the static model on one unit,
    # with and without inputs_ready
    r = pc.check_variant(tile, [3], "static", stages=2, early=early)
    assert r.ok, r.message
