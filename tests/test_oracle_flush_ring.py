"""The flush ring of the row and column sums (consumer warps hand each finished
band or strip to a flush warp through a few shared-memory slots with the
full/empty mbarrier protocol of the tile ring, run the other way round),
checked on the oracle's discrete-event model under random interleavings:
every record arrives in order and intact, for the row sum's 2 slots, the
column sum's 1 and other depths.  Planted mistakes -- the writers starting at the readers' parity, a
full barrier expecting one arrival instead of one per writer warp, the
reader starting at the writers' parity -- are each caught."""
import pytest

from oracle.simulator import simulate_flush_ring


@pytest.mark.parametrize("slots", [1, 2, 3, 4])
@pytest.mark.parametrize("writers", [1, 4, 8])
def test_every_record_arrives_in_order_and_intact(slots, writers):
    for seed in range(40):
        r = simulate_flush_ring(slots, 13, writers, seed=seed)
        assert r.status == "done", (seed, r.status)
        assert r.violations == [], (seed, r.violations[:3])
        assert r.taken == list(range(13))


def test_writers_starting_at_the_readers_parity_deadlock():
    # The writers' first empty wait then waits for a release that needs their
    # own first record: nothing can move.
    r = simulate_flush_ring(2, 6, 4, seed=1, writer_start_parity=0)
    assert r.status == "deadlock"


def test_full_barrier_counting_one_writer_loses_shares():
    # One arrival completes the slot while other warps are still writing.
    bad = 0
    for seed in range(40):
        r = simulate_flush_ring(2, 8, 4, seed=seed, full_count=1)
        bad += bool(r.violations) or r.status != "done"
    assert bad > 0


def test_reader_starting_at_the_writers_parity_reads_too_early():
    bad = 0
    for seed in range(40):
        r = simulate_flush_ring(2, 8, 4, seed=seed, reader_start_parity=1)
        bad += bool(r.violations) or r.status != "done"
    assert bad > 0
