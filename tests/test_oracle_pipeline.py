"""Pins for the oracle's pipeline cursor, mbarrier model and CTA simulator.

Pinned against the lessons' printed tables (``tests/golden/``), the closed
form of the cursor, the barrier rules stated on the pages, and the deadlock
scenarios the pages describe.
"""
import itertools

import pytest

from oracle.mbarrier import MBarrier, ProtocolError
from oracle.pipeline_state import (PipelineState, closed_form, consumer_start,
                                   producer_start, sequence)
from oracle.simulator import lockstep_timeline, simulate, two_stage_parity_table
from conftest import read_golden


# -- cursor -------------------------------------------------------------------

def test_three_stage_step_table():
    rows = [tuple(map(int, r)) for r in read_golden("pipeline_state_3stage.txt")]
    st = PipelineState(3)
    got = [st.as_tuple()]
    for _ in range(len(rows) - 1):
        got.append(st.step().as_tuple())
    assert got == rows


def test_start_states_and_role_sequences():
    rows = read_golden("lesson12_roles.txt")
    assert producer_start(3).as_tuple() == (0, 1, 0)
    assert consumer_start(3).as_tuple() == (0, 0, 0)
    prod = [(int(r[2]), int(r[3])) for r in rows if r[0] == "producer"]
    cons = [(int(r[2]), int(r[3])) for r in rows if r[0] == "consumer"]
    assert sequence(3, 1, len(prod)) == prod
    assert sequence(3, 0, len(cons)) == cons


@pytest.mark.parametrize("S", range(1, 9))
def test_advance_equals_repeated_step(S):
    for index, phase, n in itertools.product(range(S), (0, 1), range(65)):
        a = PipelineState(S, index, phase, 5).advance(n)
        b = PipelineState(S, index, phase, 5)
        for _ in range(n):
            b.step()
        assert a.as_tuple() == b.as_tuple(), (S, index, phase, n)


@pytest.mark.parametrize("S", range(1, 9))
def test_closed_form(S):
    for p0 in (0, 1):
        st = PipelineState(S, 0, p0, 0)
        for t in range(5 * S + 3):
            assert st.as_tuple() == closed_form(S, p0, t)
            st.step()


def test_phase_flips_once_per_pass():
    # a one-stage ring flips on every step; an S-stage ring every S steps
    assert [s for _, s in sequence(1, 0, 4)] == [0, 1, 0, 1]
    assert [s for _, s in sequence(4, 1, 9)] == [1, 1, 1, 1, 0, 0, 0, 0, 1]


# -- mbarrier -----------------------------------------------------------------

def test_init_state():
    b = MBarrier(96)
    assert (b.phase, b.pending, b.tx, b.parity) == (0, 96, 0, 0)


def test_phase_completes_iff_arrivals_and_tx_reach_zero():
    for count, nbytes in itertools.product((1, 2, 3), (16, 16384)):
        b = MBarrier(count)
        for _ in range(count - 1):
            assert not b.arrive()
        # last arrival registers bytes: arrivals reach 0 but tx does not
        assert not b.arrive_expect_tx(nbytes)
        assert b.phase == 0 and b.pending == 0 and b.tx == nbytes
        assert not b.complete_tx(nbytes - 1)
        assert b.phase == 0
        assert b.complete_tx(1)
        assert b.phase == 1 and b.pending == count and b.tx == 0
    # no bytes at all: the last plain arrival completes the phase
    b = MBarrier(2)
    assert not b.arrive() and b.arrive() and b.phase == 1
    # bytes delivered but an arrival still owed: no completion
    b = MBarrier(2)
    b.arrive_expect_tx(64)
    b.complete_tx(64)
    assert b.phase == 0 and b.pending == 1
    assert b.arrive() and b.phase == 1


def test_two_partial_copies_complete_one_phase():
    """Figure of "异步协作：mbarrier": two 2048-byte copies under one
    arrive.expect_tx complete exactly one phase, on the last byte."""
    b = MBarrier(1)
    b.arrive_expect_tx(4096)
    assert b.parity == 0
    b.complete_tx(2048)
    assert b.parity == 0
    b.complete_tx(2048)
    assert b.parity == 1 and b.phase == 1


def test_bytes_delivered_before_expect_are_accounted():
    b = MBarrier(1)
    b.complete_tx(100)            # transiently negative tx
    assert b.phase == 0
    b.arrive_expect_tx(100)
    assert b.phase == 1


def test_wait_semantics_is_parity_difference():
    b = MBarrier(1)
    assert not b.test_wait_parity(0) and b.test_wait_parity(1)
    b.arrive()
    assert b.test_wait_parity(0) and not b.test_wait_parity(1)
    b.arrive()
    assert not b.test_wait_parity(0)   # two completions: parity 0 again


def test_over_arrival_is_an_error():
    b = MBarrier(2)
    b.arrive()
    with pytest.raises(ProtocolError):
        b.arrive(2)


# -- lesson tables --------------------------------------------------------------

def test_three_stage_eight_tile_timeline():
    want = [tuple(map(int, r)) for r in read_golden("timeline_3stage_8tiles.txt")]
    got = []
    for row in lockstep_timeline(3, 8, consumers=96):
        assert not row["producer_blocks"]
        assert row["consumer_passes"]
        got.append((row["tile"], *row["write"], row["empty_parity_at_wait"],
                    *row["full_flip"], row["full_parity_at_wait"],
                    *row["empty_flip"], *row["read"]))
    assert got == want


def test_two_stage_parity_table():
    want = [tuple(map(int, r)) for r in read_golden("parity_2stage.txt")]
    assert two_stage_parity_table(4) == want


# -- simulator: safety under random schedules ------------------------------------

@pytest.mark.parametrize("S", [1, 2, 3, 4, 6])
@pytest.mark.parametrize("consumers", [1, 3, 7])
def test_protocol_is_safe_under_random_schedules(S, consumers):
    for seed in range(12):
        tiles = (seed * 5) % 23
        r = simulate(S, tiles, consumers, seed=seed)
        assert r.status == "done", r.violations
        assert r.violations == []
        assert r.max_lead <= S
        assert [(i, p) for _, i, p in r.producer_log] == sequence(S, 1, tiles)
        for log in r.consumer_logs:
            assert [(i, p) for _, i, p in log] == sequence(S, 0, tiles)
        # each barrier completed once per use of its stage
        for s in range(S):
            uses = len(range(s, tiles, S))
            assert r.full_phases[s] == uses
            # empty: once per use, plus nothing else (the tail only waits)
            assert r.empty_phases[s] == uses


def test_per_thread_release_counts_also_safe():
    """96 consumer threads each arriving (the lesson's count) is as safe as
    one arrival per consumer warp."""
    r = simulate(3, 8, 96, seed=1)
    assert r.status == "done" and not r.violations


# -- simulator: the deadlocks the lesson describes --------------------------------

def test_producer_starting_at_phase_zero_deadlocks():
    r = simulate(3, 8, 3, producer_start_phase=0, seed=0)
    assert r.status == "deadlock"
    assert r.producer_log == []


def test_full_barrier_expecting_a_whole_warp_deadlocks():
    # full barrier initialised with 32 arrivals, but only the elected lane arrives
    r = simulate(3, 8, 3, full_count=32, seed=0)
    assert r.status == "deadlock"
    assert all(len(log) == 0 for log in r.consumer_logs)


def test_consumer_that_never_releases_deadlocks():
    r = simulate(3, 8, 3, releasing=2, seed=0)
    assert r.status == "deadlock"
    assert len(r.producer_log) == 3          # the ring fills, then stalls


def test_missing_release_with_fewer_tiles_than_stages_finishes_but_tail_blocks():
    # With tiles <= S the ring never wraps, so only the tail notices.
    r = simulate(3, 2, 3, releasing=2, seed=0)
    assert r.status == "deadlock"
    r2 = simulate(3, 2, 3, releasing=2, seed=0, tail=False)
    assert r2.status == "done"


def test_checker_flags_a_planted_overwrite():
    """The checker itself must catch a broken protocol: when the empty barrier
    counts only one of three consumers, some schedule lets the producer
    overwrite a stage the other two are still reading."""
    found = any(simulate(1, 6, 3, empty_count=1, releasing=1, seed=seed).violations
                for seed in range(40))
    assert found
