"""Host-side checker of the GEMM kernel's barrier protocol.

The CUTLASS Task Scheduling pages check a captured schedule for deadlocks,
races and barrier initialisation before lowering it ("Introduction",
TaskManager.print_and_verify).  This kernel has no captured schedule: its role
loops are plain CUDA.  This module restates those loops -- TMA producer of each
CTA, the MMA issuer, the epilogue warps of each CTA and, under Cluster Launch
Control, the scheduler and every role's consumption of the responses -- as
small programs over mbarriers and buffers, with the arrival counts and
transaction bytes the kernel itself initialises its barriers with
(ts_gemm_protocol_info).  The native engine ts_protocol_check then explores
every interleaving of the roles and of the asynchronous units they drive (TMA
completions in any order, the in-order tcgen05 queue and its commits, CLC
responses) and reports

* a deadlock: no role can move and nothing is in flight, before every role
  has finished;
* a race: an MMA reads a ring stage (or, in the Merge layout, either half of
  it) that does not hold the k-block it expects
  (overwritten early or not yet landed) or accumulates onto the wrong partial
  sum, an epilogue reads an accumulator that is not the finished tile (or,
  for a unit with no k-blocks, one that a later unit already writes), or a
  CLC response slot is refilled before every role read it.

A model is one worker (a CTA, or a CTA pair) over a short sequence of work
units.  A unit has k-blocks (a whole tile or one K part of a split tile),
none (a group with K = 0 of a grouped GEMM: the MMA takes an accumulator and
commits it with no MMA issued, the epilogue reads and releases it), or is
skipped (TS "Schedules", Skippable Tiles: every role takes the unit from the
queue, but no load is issued and no accumulator is taken).  A second model,
build_split_program, covers the one protocol that crosses workers: the split
tiles' partials handed over through a per-slab counter in global memory.

Epilogue warps run identical, independent programs, so a model may keep fewer
of them than the kernel has; the barriers they arrive on then expect exactly
the removed warps' arrivals fewer, so a miscount in the kernel's constants
still shows.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field

import numpy as np

from . import _lib

OP_WAIT, OP_ARRIVE, OP_TMA, OP_MMA, OP_COMMIT, OP_TREAD, OP_CREQ, OP_CREAD, OP_GWRITE, OP_FENCE, OP_TICKET, \
    OP_TREADB = range(12)
SKIP = -1  # a skipped tile in a unit sequence
# mistakes that show only on units with no k-blocks (a skipped tile or a K = 0 group)
ZERO_K_MUTATIONS = ("mma_takes_skipped_accumulator", "epilogue_waits_skipped_tile", "zero_k_mma_no_commit",
                    "zero_k_epilogue_no_release")
MUTATIONS = ("tmem_empty_count_low", "tmem_empty_count_high", "clc_empty_count_low", "tx_bytes_one_cta",
             "producer_wait_parity", "epilogue_release_before_read", "mma_skip_stage_release",
             "fork_producer_ignores_second_consumer", "merge_mma_skips_b_wait") + ZERO_K_MUTATIONS
SPLIT_MUTATIONS = ("split_no_fence", "split_no_rearm", "split_last_early")
LAZY_MUTATIONS = ("lazy_wait_one_unit_late",)
# mistakes in where a role waits on the dependent-launch barrier (inputs_ready): after its third
# unit instead of its first
EARLY_MUTATIONS = ("mma_dep_wait_late", "producer_dep_wait_late", "scheduler_dep_wait_late")


def _tag(unit: int, kb: int) -> int:
    return unit * 1024 + kb


@dataclass
class Program:
    bars: list = field(default_factory=list)
    bar_names: list = field(default_factory=list)
    bufs: list = field(default_factory=list)
    roles: list = field(default_factory=list)  # (name, group or None, [op records])
    counters: list = field(default_factory=list)  # expected reductions of each global counter

    def bar(self, name: str, count: int) -> int:
        self.bars.append(int(count))
        self.bar_names.append(name)
        return len(self.bars) - 1

    def buf(self, name: str) -> int:
        self.bufs.append(name)
        return len(self.bufs) - 1

    def counter(self, reductions: int) -> int:
        self.counters.append(int(reductions))
        return len(self.counters) - 1


def build_program(proto: dict, units: list, sched: str = "static", epilogue_warps: int | None = None,
                  stages: int | None = None, mutate: str | None = None, fork: bool = False,
                  lazy: bool = False, lazy_lead: int = 1, early: bool = False) -> Program:
    """The kernel's role loops for one worker.

    proto           ts_gemm_protocol_info() of the variant.
    units           k-blocks of each work unit the worker processes, in order:
                    n > 0 k-blocks, 0 (a K = 0 group) or SKIP (a skipped tile).
    sched           "static", or "clc": after each unit every role consumes one
                    response; the first len(units) - 1 name a unit, the last fails.
    epilogue_warps  epilogue warps per CTA to model (default: the kernel's).
    stages          ring depth to model (default: the kernel's).
    mutate          plant one protocol mistake (MUTATIONS), for the checker's tests.
    fork            add the Fork pipeline group's second consumer of the ring (the
                    row-sum task): it reads every stage after the full barrier and
                    releases it on its own empty barrier; the producer refills a
                    stage only after both consumers released it (one-CTA tiles).
    lazy            lazy CLC requests (long K loops): the (A) producer of the even
                    CTA arrives on a barrier once per unit, when at most
                    `lazy_lead` of its k-blocks remain to be loaded (the kernel's
                    lead is 16; at once for a shorter or empty unit), and the
                    scheduler's request k waits for that point of unit k
                    (completion k + 1) before it is issued.
    early           inputs_ready: the dependent-launch barrier (the previous
                    kernel's completion; TS "Introduction", Core Terms: a PDL
                    barrier) gates the epilogue from its start, and every other
                    role waits on it after its first unit.  The model releases
                    the barrier as late as it can: a "previous kernel" role
                    arrives on it only once every other role has reached its
                    wait, so a role whose first unit needs the epilogue (a wait
                    that would last as long as the previous kernel, and could
                    run into its time limit) shows as a deadlock.

    A variant with proto["merge"] = 1 has the Merge layout of the "Pipeline
    Groups" page: two producers per CTA, one loading A onto full[s] and one
    loading B onto full_b[s], both waiting on the shared empty[s]; the MMA
    waits on both full barriers, and every producer consumes each CLC response.
    """
    merge = bool(proto.get("merge", 0))
    if fork and proto["cluster"] != 1:
        raise ValueError("the Fork consumer runs on one-CTA tiles only")
    if fork and merge:
        raise ValueError("the Merge layout has no Fork consumer")
    if mutate == "merge_mma_skips_b_wait" and not merge:
        raise ValueError("merge_mma_skips_b_wait needs a Merge variant")
    if mutate is not None and mutate not in MUTATIONS + LAZY_MUTATIONS + EARLY_MUTATIONS:
        raise ValueError(f"unknown mutation {mutate}")
    if mutate in LAZY_MUTATIONS and not lazy:
        raise ValueError(f"{mutate} needs lazy requests")
    if mutate in EARLY_MUTATIONS and not early:
        raise ValueError(f"{mutate} needs early (inputs_ready)")
    if any(nk != SKIP and nk < 0 for nk in units):
        raise ValueError("a unit has n >= 0 k-blocks or is SKIP")
    cg = proto["cluster"]
    S = stages or proto["stages"]
    E = proto["epilogue_warps"] if epilogue_warps is None else epilogue_warps
    dropped = (proto["epilogue_warps"] - E) * cg  # epilogue warps of the worker not modelled
    A, R = proto["accumulators"], proto["clc_slots"]
    P = Program()
    full = [[P.bar(f"full[{c}][{s}]", proto["full_arrivals"]) for s in range(S)] for c in range(cg)]
    full_b = [P.bar(f"full_b[{s}]", proto["full_arrivals"]) for s in range(S)] if merge else []
    empty = [[P.bar(f"empty[{c}][{s}]", proto["empty_arrivals"]) for s in range(S)] for c in range(cg)]
    tfull = [[P.bar(f"tmem_full[{c}][{a}]", proto["tmem_full_arrivals"]) for a in range(A)] for c in range(cg)]
    tempty_n = proto["tmem_empty_arrivals"] - dropped + {"tmem_empty_count_low": -1,
                                                          "tmem_empty_count_high": 1}.get(mutate, 0)
    tempty = [P.bar(f"tmem_empty[{a}]", tempty_n) for a in range(A)]
    clc_full = [[P.bar(f"clc_full[{c}][{r}]", proto["clc_full_arrivals"]) for r in range(R)] for c in range(cg)]
    clc_empty_n = proto["clc_empty_arrivals"] - dropped - (1 if mutate == "clc_empty_count_low" else 0) \
        + (1 if fork else 0)
    clc_empty = [P.bar(f"clc_empty[{r}]", clc_empty_n) for r in range(R)]
    aux_empty = [P.bar(f"aux_empty[{s}]", proto["aux_empty_arrivals"]) for s in range(S)] if fork else []
    clc = sched == "clc"
    began = P.bar("prod_began", 1) if (lazy and clc) else -1
    if early:
        n_prod = (2 if merge else 1) * cg
        gate = P.bar("roles_at_dependency_wait", n_prod + 1 + (1 if fork else 0) + (cg if clc else 0))
        pdl = P.bar("dependent_launch", 1)

    def dep_wait(ops, u, late):
        # a role's wait on the dependent-launch barrier after unit u (its first; the third under
        # the role's mutation)
        if early and u == (2 if late else 0):
            ops += [rec(OP_ARRIVE, gate, 0), rec(OP_WAIT, pdl, 0)]
    stage = [[P.buf(f"stage[{c}][{s}]") for s in range(S)] for c in range(cg)]  # A (and B unless Merge)
    stage_b = [[P.buf(f"stage_b[{c}][{s}]") for s in range(S)] for c in range(cg)] if merge else []
    accb = [P.buf(f"tmem[{a}]") for a in range(A)]
    slot = [[P.buf(f"clc_slot[{c}][{r}]") for r in range(R)] for c in range(cg)]
    a_bytes = proto["a_stage_bytes"] if merge else proto["stage_bytes"]  # per CTA, onto full[s]
    b_bytes = proto["stage_bytes"] - a_bytes  # per CTA, onto full_b[s] (Merge)
    tx = (proto["tx_bytes"] if not merge else a_bytes * cg) - (a_bytes if mutate == "tx_bytes_one_cta" else 0)

    def rec(*v):
        v = list(v) + [-1] * (8 - len(v))
        return v[:8]

    def consume(ops, c, k):
        r, ph = k % R, (k // R) & 1
        ops += [rec(OP_WAIT, clc_full[c][r], ph), rec(OP_CREAD, slot[c][r], k), rec(OP_ARRIVE, clc_empty[r], 0)]

    def adv(i, ph, n):
        return (0, ph ^ 1) if i + 1 == n else (i + 1, ph)

    # producers of each CTA: one (A and B onto full[s]), or with Merge one for A
    # onto full[s] and one for B onto full_b[s]
    lines = [("producer", full, stage, a_bytes, tx)]
    if merge:
        lines = [("producer_a", full, stage, a_bytes, tx), ("producer_b", [full_b], stage_b, b_bytes, b_bytes * cg)]
    for name, fbar, sbuf, nbytes, arm in lines:
        for c in range(cg):
            ops, s, ph, issued = [], 0, 0, 0
            signals = began >= 0 and c == 0 and name in ("producer", "producer_a")
            for u, nk in enumerate(units):
                near_end = nk - lazy_lead if nk > lazy_lead else 0
                if signals and nk <= 0:
                    ops.append(rec(OP_ARRIVE, began, 0))  # an empty unit counts as loaded at once
                for kb in range(max(nk, 0)):  # a skipped tile or a K = 0 group loads nothing
                    if signals and kb == near_end:
                        ops.append(rec(OP_ARRIVE, began, 0))  # unit u nearly loaded
                    ops.append(rec(OP_WAIT, empty[c][s], ph if mutate == "producer_wait_parity" else ph ^ 1))
                    if fork and mutate != "fork_producer_ignores_second_consumer":
                        ops.append(rec(OP_WAIT, aux_empty[s], ph ^ 1))
                    if c == 0:
                        ops.append(rec(OP_ARRIVE, fbar[0][s], arm))
                    ops.append(rec(OP_TMA, sbuf[c][s], _tag(u, kb), fbar[0][s], nbytes))
                    issued += 1
                    s, ph = adv(s, ph, S)
                dep_wait(ops, u, mutate == "producer_dep_wait_late")
                if clc:
                    consume(ops, c, u)
            if early and len(units) <= (2 if mutate == "producer_dep_wait_late" else 0):
                ops += [rec(OP_ARRIVE, gate, 0), rec(OP_WAIT, pdl, 0)]
            if c == 0:  # drain: the last issued loads landed
                for i in range(1, min(issued, S) + 1):
                    b = issued - i
                    ops.append(rec(OP_WAIT, fbar[0][b % S], (b // S) & 1))
            for _ in range(S):  # drain: the MMA (and the Fork consumer) released every stage
                ops.append(rec(OP_WAIT, empty[c][s], ph ^ 1))
                if fork:
                    ops.append(rec(OP_WAIT, aux_empty[s], ph ^ 1))
                s, ph = adv(s, ph, S)
            P.roles.append((f"{name}[{c}]", None, ops))

    ops, s, ph, a, aph = [], 0, 0, 0, 0  # MMA issuer of the even CTA
    mma_late = mutate == "mma_dep_wait_late"
    for u, nk in enumerate(units):
        if nk == SKIP and mutate != "mma_takes_skipped_accumulator":
            dep_wait(ops, u, mma_late)
            if clc:  # a skipped tile takes no accumulator; the queue still advances
                consume(ops, 0, u)
            continue
        ops.append(rec(OP_WAIT, tempty[a], aph ^ 1))
        for kb in range(max(nk, 0)):
            ops.append(rec(OP_WAIT, full[0][s], ph))
            if merge and mutate != "merge_mma_skips_b_wait":
                ops.append(rec(OP_WAIT, full_b[s], ph))
            sb = [stage_b[0][s], stage_b[1][s] if cg == 2 else -1] if merge else [-1, -1]
            ops.append(rec(OP_MMA, stage[0][s], stage[1][s] if cg == 2 else -1, accb[a], _tag(u, kb), *sb))
            if not (mutate == "mma_skip_stage_release" and u == 0 and kb == 0):
                ops.append(rec(OP_COMMIT, empty[0][s], empty[1][s] if cg == 2 else -1))
            s, ph = adv(s, ph, S)
        if not (mutate == "zero_k_mma_no_commit" and nk == 0):
            # with no k-block the commit completes at once: the epilogue finds an empty sum
            ops.append(rec(OP_COMMIT, tfull[0][a], tfull[1][a] if cg == 2 else -1))
        a, aph = adv(a, aph, A)
        dep_wait(ops, u, mma_late)
        if clc:
            consume(ops, 0, u)
    if early and len(units) <= (2 if mma_late else 0):
        ops += [rec(OP_ARRIVE, gate, 0), rec(OP_WAIT, pdl, 0)]
    P.roles.append(("mma", None, ops))

    for c in range(cg):  # epilogue warps of each CTA: one symmetry group per CTA
        for w in range(E):
            ops, a, aph = [], 0, 0
            if early:  # D is written only after the previous kernel completed
                ops.append(rec(OP_WAIT, pdl, 0))
            for u, nk in enumerate(units):
                if nk == SKIP and mutate != "epilogue_waits_skipped_tile":
                    if clc:  # a skipped tile stores nothing and takes no accumulator
                        consume(ops, c, u)
                    continue
                ops.append(rec(OP_WAIT, tfull[c][a], aph))
                if clc:  # the next response is taken as soon as the accumulator is held
                    consume(ops, c, u)
                if nk > 0:
                    read = rec(OP_TREAD, accb[a], _tag(u, nk - 1))
                else:
                    # K = 0 (or a skipped tile under the mutation): the accumulator's old
                    # contents are read and discarded (zeros are stored); only a later
                    # unit's MMA writing it during the read would be a race
                    read = rec(OP_TREADB, accb[a], _tag(u, 0))
                release = rec(OP_ARRIVE, tempty[a], 0)
                if mutate == "zero_k_epilogue_no_release" and nk == 0:
                    ops.append(read)
                else:
                    ops += [release, read] if mutate == "epilogue_release_before_read" else [read, release]
                a, aph = adv(a, aph, A)
            P.roles.append((f"epilogue[{c}][{w}]", f"epilogue[{c}]", ops))

    if fork:  # the Fork pipeline group's second consumer of the ring
        ops, s, ph = [], 0, 0
        for u, nk in enumerate(units):
            for kb in range(max(nk, 0)):
                ops += [rec(OP_WAIT, full[0][s], ph), rec(OP_TREAD, stage[0][s], _tag(u, kb)),
                        rec(OP_ARRIVE, aux_empty[s], 0)]
                s, ph = adv(s, ph, S)
            dep_wait(ops, u, False)  # before the unit's row-sum store
            if clc:
                consume(ops, 0, u)
        P.roles.append(("rowsum", None, ops))

    if clc:  # CLC scheduler of each CTA; the even CTA's request fills every CTA's slot
        for c in range(cg):
            ops = []
            for k in range(len(units)):
                r, ph2 = k % R, (k // R) & 1
                if c == 0:
                    ops.append(rec(OP_WAIT, clc_empty[r], ph2 ^ 1))
                    if began >= 0:  # request k waits until the producer began unit k
                        ops.append(rec(OP_WAIT, began, (k + (1 if mutate == "lazy_wait_one_unit_late" else 0)) & 1))
                    ops += [rec(OP_ARRIVE, clc_full[0][r], proto["clc_response_bytes"]),
                            rec(OP_CREQ, slot[0][r], slot[1][r] if cg == 2 else -1, k, clc_full[0][r],
                                clc_full[1][r] if cg == 2 else -1, proto["clc_response_bytes"])]
                else:
                    ops.append(rec(OP_ARRIVE, clc_full[c][r], proto["clc_response_bytes"]))
                consume(ops, c, k)
                dep_wait(ops, k, mutate == "scheduler_dep_wait_late")
            if early and len(units) <= (2 if mutate == "scheduler_dep_wait_late" else 0):
                ops += [rec(OP_ARRIVE, gate, 0), rec(OP_WAIT, pdl, 0)]
            P.roles.append((f"scheduler[{c}]", None, ops))
    if early:  # the previous kernel completes once every role that may has run ahead of it
        P.roles.append(("previous_kernel", None, [rec(OP_WAIT, gate, 0), rec(OP_ARRIVE, pdl, 0)]))
    return P


@dataclass
class Result:
    ok: bool
    status: int  # 0 verified, 1 violation, 2 state limit
    states: int
    message: str


def check(P: Program, max_states: int = 20_000_000) -> Result:
    """Explore every interleaving of the program with the native engine."""
    groups = {}
    role_group = [(-1 if g is None else groups.setdefault(g, len(groups))) for _, g, _ in P.roles]
    offsets = [0]
    flat = []
    for _, _, ops in P.roles:
        flat += ops
        offsets.append(len(flat))
    ops = np.ascontiguousarray(np.array(flat, dtype=np.int32).reshape(-1))
    bars = np.ascontiguousarray(np.array(P.bars, dtype=np.int32))
    grp = np.ascontiguousarray(np.array(role_group, dtype=np.int32))
    off = np.ascontiguousarray(np.array(offsets, dtype=np.int32))
    ctrs = np.ascontiguousarray(np.array(P.counters if P.counters else [0], dtype=np.int32))
    names = "\n".join([n for n, _, _ in P.roles] + P.bar_names + P.bufs).encode()
    msg = ctypes.create_string_buffer(512)
    states = ctypes.c_int64(0)
    rc = _lib.ts_protocol_check_ex(len(P.bars), bars.ctypes.data, len(P.bufs), len(P.roles), grp.ctypes.data,
                                   off.ctypes.data, ops.ctypes.data, len(P.counters), ctrs.ctypes.data, names,
                                   int(max_states), ctypes.byref(states), msg, len(msg))
    if rc < 0:
        raise ValueError("ts_protocol_check rejected the program")
    return Result(rc == 0, rc, int(states.value), msg.value.decode())


def check_variant(tile: str, units: list, sched: str = "static", out: int = 0, max_states: int = 20_000_000,
                  variant_epi_warps: int = 4, variant_merge: int = 0, **kw) -> Result:
    """Check the protocol of a compiled kernel variant (tile, output type,
    epilogue warp count and barrier layout) on a unit sequence."""
    from . import ts_gemm_protocol_info

    proto = ts_gemm_protocol_info(tile, out, variant_epi_warps, variant_merge)
    return check(build_program(proto, units, sched, **kw), max_states)


def build_split_program(parts: int, launches: int = 2, mutate: str | None = None) -> Program:
    """The split tiles' handoff of one 32-row slab, across the workers of its K parts.

    Part p (a different worker each) stores its fp32 partial of the slab, fences
    (__threadfence), and adds one to the slab's counter in global memory; the part
    that draws ticket parts - 1 re-arms the counter to 0 and sums the partials of
    every part (gemm_kernel.cuh, the split epilogue).  Nothing waits on another
    worker.  `launches` kernel launches run back to back on the same workspace
    (a barrier stands for the launch boundary), so a counter left armed shows as
    a launch with no reduction.  Checked: every reduction reads each part's
    partial of its own launch, and each launch reduces exactly once.

    mutate: "split_no_fence" (the ticket may overtake the partial's store),
    "split_no_rearm" (the counter is left at `parts`), "split_last_early" (the
    part that draws ticket parts - 2 reduces)."""
    if parts < 2:
        raise ValueError("a split tile has at least two parts")
    if mutate is not None and mutate not in SPLIT_MUTATIONS:
        raise ValueError(f"unknown mutation {mutate}")
    P = Program()
    ctr = P.counter(launches)
    partial = [P.buf(f"partial[{p}]") for p in range(parts)]
    boundary = P.bar("launch_boundary", parts)
    last = parts - (2 if mutate == "split_last_early" else 1)
    rearm = 0 if mutate == "split_no_rearm" else 1
    for p in range(parts):
        ops = []
        for L in range(launches):
            ops.append([OP_GWRITE, partial[p], L * 1024 + p, -1, -1, -1, -1, -1])
            if mutate != "split_no_fence":
                ops.append([OP_FENCE, -1, -1, -1, -1, -1, -1, -1])
            ops.append([OP_TICKET, ctr, last, partial[0], parts, L * 1024, rearm, -1])
            ops.append([OP_ARRIVE, boundary, 0, -1, -1, -1, -1, -1])
            ops.append([OP_WAIT, boundary, L & 1, -1, -1, -1, -1, -1])
        P.roles.append((f"part[{p}]", None, ops))
    return P


# ------------------------------------------------------------ protocol log
# The logging build of the kernel (ts_gemm_opts.protocol_log) records every role's barrier
# operations in program order.  These functions turn a model program and a kernel log into the
# same event vocabulary, so that each modelled role can be compared with what the kernel did.
PL_WAIT, PL_ARRIVE, PL_TMA, PL_MMA, PL_COMMIT, PL_CREQ, PL_PDL, PL_UNIT, PL_TLOAD, PL_CREAD, PL_SREAD = range(1, 12)
PF_FULL, PF_EMPTY, PF_TFULL, PF_TEMPTY, PF_CLC_FULL, PF_CLC_EMPTY, PF_AUX, PF_BEGAN, PF_MMA_DONE = range(9)
PF_NONE = 15
_FAMILY = {"full": PF_FULL, "empty": PF_EMPTY, "tmem_full": PF_TFULL, "tmem_empty": PF_TEMPTY,
           "clc_full": PF_CLC_FULL, "clc_empty": PF_CLC_EMPTY, "aux_empty": PF_AUX, "full_b": PF_AUX,
           "prod_began": PF_BEGAN}
_OP_NAME = {PL_WAIT: "wait", PL_ARRIVE: "arrive", PL_TMA: "tma", PL_MMA: "mma", PL_COMMIT: "commit",
            PL_CREQ: "clc_request", PL_PDL: "dependent_launch_wait", PL_TLOAD: "accumulator_read",
            PL_CREAD: "response_read", PL_SREAD: "stage_read"}
_FAM_NAME = {v: k for k, v in _FAMILY.items() if k != "full_b"}
_FAM_NAME.update({PF_MMA_DONE: "mma_done", PF_NONE: "-"})
LOG_ROLES = 20  # roles per CTA in the log: 0 producer, 1 MMA, 2 scheduler, 3 warp 3, 4 + j epilogue warp j


def encode_event(op: int, family: int = PF_NONE, index: int = 0, parity: int = 0) -> int:
    """The kernel's event word (PLog::put)."""
    return op | (family << 4) | (index << 8) | ((parity & 1) << 16)


def describe(ev) -> str:
    op, fam, idx, par = ev
    s = f"{_OP_NAME.get(op, op)} {_FAM_NAME.get(fam, fam)}[{idx}]"
    return s + (f" parity {par}" if op == PL_WAIT else "")


def decode_log(block) -> tuple[list, list]:
    """One role's log block (count, then events) -> (events, units).

    events: (op, family, index, parity) tuples in program order; units: the units the producer
    began, SKIP or their k-block counts.  Raises if the events overflowed the block."""
    block = np.asarray(block, dtype=np.int64)
    n = int(block[0])
    if n > block.size - 1:
        raise ValueError(f"the log holds {block.size - 1} events of {n}: give it more room")
    events, units = [], []
    for w in block[1:1 + n]:
        w = int(w)
        op = w & 0xF
        if op == PL_UNIT:
            units.append(SKIP if (w >> 4) & 1 else w >> 8)
            continue
        events.append((op, (w >> 4) & 0xF, (w >> 8) & 0xFF, (w >> 16) & 1 if op == PL_WAIT else 0))
    return events, units


def _bar(name: str):
    """Model barrier name -> (family, index); None for the model's own gate barrier."""
    base = name.split("[")[0]
    if base == "roles_at_dependency_wait":
        return None
    if base == "dependent_launch":
        return "pdl"
    idx = int(name.rstrip("]").split("[")[-1]) if "[" in name else 0
    return _FAMILY[base], idx


def _buf_index(name: str) -> int:
    return int(name.rstrip("]").split("[")[-1])


def model_events(P: Program, role: str) -> list:
    """The modelled role's operations in the log's vocabulary: barrier operations, and the reads
    of accumulators, CLC responses and (by the Fork task) ring stages.  The gate on which the model
    holds back the previous kernel is the model's own."""
    ops = next(o for n, _, o in P.roles if n == role)
    out = []
    for o in ops:
        kind = o[0]
        if kind == OP_WAIT:
            b = _bar(P.bar_names[o[1]])
            if b == "pdl":
                out.append((PL_PDL, PF_NONE, 0, 0))
            elif b is not None:
                out.append((PL_WAIT, b[0], b[1], o[2] & 1))
        elif kind == OP_ARRIVE:
            b = _bar(P.bar_names[o[1]])
            if b is not None and b != "pdl":
                out.append((PL_ARRIVE, b[0], b[1], 0))
        elif kind == OP_TMA:
            b = _bar(P.bar_names[o[3]])
            out.append((PL_TMA, b[0], b[1], 0))
        elif kind == OP_MMA:
            out.append((PL_MMA, PF_FULL, _buf_index(P.bufs[o[1]]), 0))
        elif kind == OP_COMMIT:
            b = _bar(P.bar_names[o[1]])
            out.append((PL_COMMIT, b[0], b[1], 0))
        elif kind == OP_CREQ:
            b = _bar(P.bar_names[o[4]])
            out.append((PL_CREQ, b[0], b[1], 0))
        elif kind in (OP_TREAD, OP_TREADB):
            name = P.bufs[o[1]]
            if name.startswith("tmem"):
                out.append((PL_TLOAD, PF_TFULL, _buf_index(name), 0))
            elif name.startswith("stage"):
                out.append((PL_SREAD, PF_FULL, _buf_index(name), 0))
        elif kind == OP_CREAD:
            out.append((PL_CREAD, PF_CLC_FULL, _buf_index(P.bufs[o[1]]), 0))
    return out


def kernel_events(events: list, lazy_signals: bool) -> list:
    """A role's logged events as the model states them: the MMA issuer's final commit and wait on
    its own completion barrier (before TMEM is freed) are not modelled, and the producers' arrivals
    on prod_began are modelled only where the scheduler waits on them (lazy CLC requests, the
    even CTA's producer); the kernel makes them on every unit."""
    return [e for e in events if e[1] != PF_MMA_DONE and not (e[1] == PF_BEGAN and e[0] == PL_ARRIVE and
                                                              not lazy_signals)]


def log_role(model_role: str) -> tuple[int, int]:
    """Model role name -> (CTA within the worker, log role)."""
    base = model_role.split("[")[0]
    idx = [int(x) for x in model_role.replace("]", "").split("[")[1:]]
    if base in ("producer", "producer_a"):
        return idx[0], 0
    if base == "producer_b":
        return idx[0], 3
    if base == "mma":
        return 0, 1
    if base == "scheduler":
        return idx[0], 2
    if base == "rowsum":
        return 0, 3
    if base == "epilogue":
        return idx[0], 4 + idx[1]
    raise ValueError(f"no log role for {model_role}")


def compare_with_log(P: Program, log_blocks, worker_ctas: list, lazy: bool) -> list:
    """Compare every modelled role with the kernel's log of one worker.

    log_blocks[c][r]: the log block of CTA worker_ctas[c] and role r.  Returns a list of
    mismatch descriptions (empty when every role did exactly what the model says)."""
    problems = []
    for name, _, _ in P.roles:
        if name == "previous_kernel":
            continue
        c, r = log_role(name)
        got, _ = decode_log(log_blocks[worker_ctas[c]][r])
        got = kernel_events(got, lazy and c == 0 and r == 0)
        want = model_events(P, name)
        if got != want:
            k = next((i for i, (g, w) in enumerate(zip(got, want)) if g != w), min(len(got), len(want)))
            problems.append(f"{name} (CTA {worker_ctas[c]}, log role {r}): event {k}: kernel "
                            f"{describe(got[k]) if k < len(got) else 'ends'}, model "
                            f"{describe(want[k]) if k < len(want) else 'ends'} ({len(got)} / {len(want)} events)")
    return problems
