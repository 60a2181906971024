"""The protocol log's host side (no GPU): event words, decoding and the model comparison."""
import numpy as np
import pytest

import tile_scheduling_gb300.protocol as pc


def _fake_log(P, ctas, units, lazy, drop_role=None, swap=None):
    """A log as the kernel would write it if it did exactly what the model says."""
    cap = 512
    log = np.zeros((ctas, pc.LOG_ROLES, cap + 1), dtype=np.int32)
    for name, _, _ in P.roles:
        if name == "previous_kernel" or name == drop_role:
            continue
        c, r = pc.log_role(name)
        words = []
        evs = pc.model_events(P, name)
        if swap is not None and swap[0] == name:
            i = swap[1]
            evs[i], evs[i + 1] = evs[i + 1], evs[i]
        words += [pc.encode_event(*e) for e in evs]
        if (c, r) == (0, 0):  # the even CTA's producer also records the units it begins
            words = [pc.PL_UNIT | ((1 if u == pc.SKIP else 0) << 4) | (max(u, 0) << 8) for u in units] + words
        log[c, r, 0] = len(words)
        log[c, r, 1:1 + len(words)] = words
    return log


@pytest.mark.parametrize("tile,sched,kw", [("128x128", "static", {}), ("128x128", "clc", {}),
                                           ("256x256", "clc", {}), ("128x128", "clc", {"early": True}),
                                           ("128x128", "clc", {"lazy": True, "lazy_lead": 16}),
                                           ("128x128", "clc", {"fork": True})])
def test_a_log_that_follows_the_model_matches(ts, tile, sched, kw):
    units = [3, pc.SKIP, 0, 2]
    proto = ts.ts_gemm_protocol_info(tile, ts.TS_OUT_F32, 4, 0)
    P = pc.build_program(proto, units, sched, **kw)
    cg = proto["cluster"]
    log = _fake_log(P, cg, units, kw.get("lazy", False))
    events, got_units = pc.decode_log(log[0, 0])
    assert got_units == units
    assert pc.compare_with_log(P, log, list(range(cg)), kw.get("lazy", False)) == []


def test_a_reordered_or_missing_role_is_reported(ts):
    units = [3, 2]
    proto = ts.ts_gemm_protocol_info("128x128", ts.TS_OUT_F32, 4, 0)
    P = pc.build_program(proto, units, "clc")
    swapped = _fake_log(P, 1, units, False, swap=("mma", 1))
    problems = pc.compare_with_log(P, swapped, [0], False)
    assert len(problems) == 1 and problems[0].startswith("mma") and "event 1" in problems[0]
    missing = _fake_log(P, 1, units, False, drop_role="epilogue[0][2]")
    problems = pc.compare_with_log(P, missing, [0], False)
    assert len(problems) == 1 and "epilogue[0][2]" in problems[0] and "kernel ends" in problems[0]


def test_a_planted_model_mistake_does_not_match_the_correct_log(ts):
    # the log of the correct protocol against a model with a wrong producer wait parity
    units = [3, 2]
    proto = ts.ts_gemm_protocol_info("128x128", ts.TS_OUT_F32, 4, 0)
    good = pc.build_program(proto, units, "static")
    log = _fake_log(good, 1, units, False)
    bad = pc.build_program(proto, units, "static", mutate="producer_wait_parity")
    problems = pc.compare_with_log(bad, log, [0], False)
    assert len(problems) == 1 and problems[0].startswith("producer[0]")


def test_event_words_round_trip():
    for ev in [(pc.PL_WAIT, pc.PF_EMPTY, 5, 1), (pc.PL_COMMIT, pc.PF_TFULL, 1, 0), (pc.PL_PDL, pc.PF_NONE, 0, 0),
               (pc.PL_CREQ, pc.PF_CLC_FULL, 1, 0)]:
        block = np.array([1, pc.encode_event(*ev)], dtype=np.int32)
        assert pc.decode_log(block) == ([ev], [])
    with pytest.raises(ValueError):
        pc.decode_log(np.array([3, 1, 1], dtype=np.int32))  # three events recorded, room for two


def test_kernel_only_events_are_dropped():
    evs = [(pc.PL_ARRIVE, pc.PF_BEGAN, 0, 0), (pc.PL_WAIT, pc.PF_EMPTY, 0, 1), (pc.PL_COMMIT, pc.PF_MMA_DONE, 0, 0),
           (pc.PL_WAIT, pc.PF_MMA_DONE, 0, 0)]
    assert pc.kernel_events(evs, lazy_signals=False) == [(pc.PL_WAIT, pc.PF_EMPTY, 0, 1)]
    assert pc.kernel_events(evs, lazy_signals=True) == evs[:2]
