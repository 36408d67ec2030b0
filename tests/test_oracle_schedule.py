"""Pins of the refresh schedule (oracle) against hand-worked sequences, and
the library's native ps_schedule_step against the oracle on random runs
(host code: no GPU needed)."""
import ctypes
import os
import random

import pytest

from oracle.schedule import FULL, REFRESH, REINIT, SLIDE, ScheduleState, schedule_step


def _run(tau, full, blk, steps):
    st = ScheduleState()
    return [schedule_step(tau, full, blk, st, c, done) for c, done in steps], st


def test_every_step_when_tau_is_zero():
    acts, _ = _run(0, 0, 32, [(0, False)] * 4)
    assert acts == [REFRESH] * 4


def test_tau_counts_committed_tokens():
    # tau 3: 1 + 1 -> no; + 1 = 3 -> refresh; 0 -> no; 2 -> no; 5 -> refresh (7 >= 3)
    acts, st = _run(3, 0, 32, [(1, False), (1, False), (1, False), (0, False), (2, False),
                               (5, False)])
    assert acts == [0, 0, REFRESH, 0, 0, REFRESH] and st.since == 0


def test_every_second_refresh_is_full():
    acts, st = _run(1, 2, 32, [(1, False)] * 5)
    assert acts == [REFRESH, REFRESH | FULL, REFRESH, REFRESH | FULL, REFRESH]
    assert st.refreshes == 5


def test_block_done_slides_and_restarts():
    acts, st = _run(2, 2, 16, [(3, False), (4, True), (1, False), (1, False)])
    assert acts[0] == REFRESH
    assert acts[1] == REFRESH | FULL | SLIDE | REINIT and st.block_start == 16
    assert acts[2] == 0 and acts[3] == REFRESH            # counts restarted at the slide
    assert st.refreshes == 1


def test_native_schedule_matches_the_oracle():
    from drift_aware_kv_spherical_gb300 import _build
    from drift_aware_kv_spherical_gb300 import polestar as ps
    if not os.path.exists(ps.LIB_PATH):
        _build.build()
    rng = random.Random(7)
    for trial in range(200):
        tau, full, blk = rng.randint(0, 6), rng.randint(0, 4), rng.choice([8, 16, 32])
        nat, o = ps.Schedule(tau, full, blk), ScheduleState()
        for _ in range(40):
            c, done = rng.randint(0, 5), rng.random() < 0.1
            assert nat.step(c, done) == schedule_step(tau, full, blk, o, c, done)
            s = nat.state
            assert (s.since, s.refreshes, s.block_start) == (o.since, o.refreshes, o.block_start)
    assert (ps.SCHED_REFRESH, ps.SCHED_FULL, ps.SCHED_SLIDE, ps.SCHED_REINIT) == \
        (REFRESH, FULL, SLIDE, REINIT)


def test_native_schedule_rejects_bad_arguments():
    from drift_aware_kv_spherical_gb300 import _build
    from drift_aware_kv_spherical_gb300 import polestar as ps
    if not os.path.exists(ps.LIB_PATH):
        _build.build()
    f = ps.Library.load().cdll.ps_schedule_step
    st = ps.ScheduleState(3, 1, 0)
    assert f(None, ctypes.byref(st), 0, 0) == -ps.PS_ERR_ARG
    for bad in (ps.ScheduleParams(-1, 0, 8), ps.ScheduleParams(1, -1, 8),
                ps.ScheduleParams(1, 0, 0)):
        assert f(ctypes.byref(bad), ctypes.byref(st), 0, 0) == -ps.PS_ERR_ARG
    good = ps.ScheduleParams(2, 0, 8)
    assert f(ctypes.byref(good), ctypes.byref(st), -1, 0) == -ps.PS_ERR_ARG
    assert (st.since, st.refreshes, st.block_start) == (3, 1, 0)      # unchanged
    big = ps.ScheduleState(2 ** 31 - 2, 0, 0)
    assert f(ctypes.byref(ps.ScheduleParams(2 ** 31 - 1, 0, 8)), ctypes.byref(big), 5, 0) == \
        ps.SCHED_REFRESH                                               # saturates, then fires


def _expected_refresh_steps(tau, counts):
    """Steps (0-based, the step whose outcome triggers it) after which a
    refresh is scheduled: the running token count reaches tau, then restarts."""
    out, run = [], 0
    for t, c in enumerate(counts):
        run += c
        if run >= tau:
            out.append(t)
            run = 0
    return out


@pytest.mark.parametrize("impl", ["oracle", "native"])
def test_refreshes_follow_the_running_count(impl):
    rng = random.Random(11)
    if impl == "native":
        from drift_aware_kv_spherical_gb300 import _build
        from drift_aware_kv_spherical_gb300 import polestar as ps
        if not os.path.exists(ps.LIB_PATH):
            _build.build()
    for _ in range(100):
        tau, full = rng.randint(0, 9), rng.randint(0, 5)
        counts = [rng.randint(0, 4) for _ in range(60)]
        if impl == "oracle":
            st = ScheduleState()
            acts = [schedule_step(tau, full, 32, st, c, False) for c in counts]
        else:
            nat = ps.Schedule(tau, full, 32)
            acts = [nat.step(c, False) for c in counts]
        got = [t for t, a in enumerate(acts) if a & REFRESH]
        assert got == _expected_refresh_steps(tau, counts)
        fulls = [t for t, a in enumerate(acts) if a & FULL]
        assert fulls == (got[full - 1::full] if full > 0 else [])
        assert not any(a & (SLIDE | REINIT) for a in acts)


def test_block_progress_hand_worked():
    from oracle.schedule import block_progress
    role = [0, 0, 1, 2]
    # sequence 0 commits two tokens (one of them suffix), sequence 1 one
    commit = [[1, 0, 1, 0], [0, 1, 0, 0]]
    undecided = [[0, 1, 0, 1], [0, 0, 1, 1]]       # seq 0 still has current token 1 open
    assert block_progress(commit, undecided, role) == (2, False)
    undecided = [[0, 0, 1, 1], [0, 0, 0, 1]]       # only suffix / inactive left: decided
    assert block_progress(commit, undecided, role) == (2, True)
    assert block_progress([[0] * 4], [[0] * 4], role) == (0, True)
