"""The row slots of the 1-D row sum's long rows, checked on a discrete-event
model under random interleavings.

A row that does not fit one window is loaded in P pieces, one window each,
through the tile ring of S stages (full barrier: the producer's arrival;
empty barrier: one arrival per consumer warp).  At a row's last piece every
consumer warp releases the stage, writes its partial of the row into slot
(row mod R) and arrives on that slot's barrier (expected count: the number of
warps); warp 0 alone then waits on the slot (parity (row div R) mod 2) and
reads every warp's partial.  The other warps go straight on.  A slot is safe
to reuse once warp 0 has read it, and the kernel relies on the ring alone for
that: another warp can be at most S windows past the window warp 0 released
last, so it reaches the slot of row + K only if K P <= S.  With R = 16 slots
that holds for S <= 15 stages at any P >= 1 (the kernel allows at most 8).

The barriers follow the mbarrier model of the oracle ("异步协作：mbarrier",
"cute(12) async_pipeline" §6).  Checked: warp 0 finds every warp's partial of
row k tagged k, for every row, in order, and nothing deadlocks.  Planted
mistakes -- too few slots for the stages, a slot barrier that expects one
arrival, as many stages as slots -- are each caught: the fast warps move a
slot's barrier whole phases on before warp 0 waits on it, so warp 0 either
reads a later row's partials or waits on a parity that has come round again
(a deadlock here, a timed-out wait on the GPU)."""
import random

import pytest

from oracle.mbarrier import MBarrier, ProtocolError


def simulate_row_slots(stages, pieces, warps, rows, slots=16, *, seed=0, slot_count=None,
                       slow_warp0=0.05, max_steps=None):
    """Returns (status, violations, rows read by warp 0 in order)."""
    rng = random.Random(seed)
    windows = rows * pieces
    full = [MBarrier(1) for _ in range(stages)]
    empty = [MBarrier(warps) for _ in range(stages)]
    row_bar = [MBarrier(warps if slot_count is None else slot_count) for _ in range(slots)]
    red = [[None] * warps for _ in range(slots)]
    pj = 0                                  # producer: next window to load
    wj = [0] * warps                        # each warp's window
    ws = ["wait"] * warps                   # wait -> release -> (deposit -> [row_wait -> read])
    read, violations = [], []
    budget = max_steps or 50 * windows * (warps + 1)
    for _ in range(budget):
        acts = []
        if pj < windows and empty[pj % stages].test_wait_parity(((pj // stages) & 1) ^ 1):
            acts.append(-1)
        for w in range(warps):
            j = wj[w]
            if j >= windows:
                continue
            st = ws[w]
            if st == "wait" and not full[j % stages].test_wait_parity((j // stages) & 1):
                continue
            lr = j // pieces
            if st == "row_wait" and not row_bar[lr % slots].test_wait_parity((lr // slots) & 1):
                continue
            acts.append(w)
        if not acts:
            done = pj >= windows and all(j >= windows for j in wj)
            return ("done" if done else "deadlock"), violations, read
        # warp 0 runs slowly, so the other warps get as far ahead as the ring lets them
        others = [a for a in acts if a != 0]
        who = 0 if (0 in acts and (not others or rng.random() < slow_warp0)) else \
            rng.choice(others)
        try:
            if who == -1:
                full[pj % stages].arrive()          # the window has landed
                pj += 1
                continue
            j = wj[who]
            lr = j // pieces
            st = ws[who]
            last = j % pieces == pieces - 1
            if st == "wait":
                ws[who] = "release"
            elif st == "release":
                empty[j % stages].arrive()
                if last:
                    ws[who] = "deposit"
                else:
                    ws[who], wj[who] = "wait", j + 1
            elif st == "deposit":
                red[lr % slots][who] = lr
                row_bar[lr % slots].arrive()
                if who == 0:
                    ws[who] = "row_wait"
                else:
                    ws[who], wj[who] = "wait", j + 1
            elif st == "row_wait":
                ws[who] = "read"
            else:                                    # warp 0 reads the row's partials
                got = list(red[lr % slots])
                if got != [lr] * warps:
                    violations.append((lr, got))
                read.append(lr)
                ws[who], wj[who] = "wait", j + 1
        except ProtocolError as e:
            violations.append(("protocol", str(e)))
            return "error", violations, read
    return "budget", violations, read


@pytest.mark.parametrize("stages", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("pieces", [1, 2, 3, 5])
@pytest.mark.parametrize("warps", [4, 8])
def test_every_row_is_read_whole_and_in_order(stages, pieces, warps):
    rows = 40
    for seed in range(12):
        status, violations, read = simulate_row_slots(stages, pieces, warps, rows, seed=seed)
        assert status == "done", (seed, status)
        assert violations == [], (seed, violations[:3])
        assert read == list(range(rows))


def test_sixteen_slots_hold_up_to_fifteen_stages():
    for seed in range(20):
        status, violations, _ = simulate_row_slots(15, 1, 4, 60, seed=seed, slow_warp0=0.01)
        assert status == "done" and violations == [], seed


def test_too_few_slots_for_the_stages_are_caught():
    # 2 slots with 8 one-piece stages: the fast warps complete slot 0's
    # barrier four times before warp 0 waits for its first phase
    bad = 0
    for seed in range(20):
        status, violations, _ = simulate_row_slots(8, 1, 4, 40, slots=2, seed=seed,
                                                   slow_warp0=0.01)
        bad += bool(violations) or status != "done"
    assert bad > 0


def test_as_many_stages_as_slots_is_caught():
    # 16 one-piece stages: a fast warp writes row 16's partial into row 0's
    # slot before warp 0 reads it
    bad = 0
    for seed in range(30):
        status, violations, _ = simulate_row_slots(16, 1, 4, 80, seed=seed, slow_warp0=0.005)
        bad += bool(violations) or status != "done"
    assert bad > 0


def test_slot_barrier_expecting_one_arrival_is_caught():
    bad = 0
    for seed in range(20):
        status, violations, _ = simulate_row_slots(4, 2, 4, 30, seed=seed, slot_count=1)
        bad += bool(violations) or status != "done"
    assert bad > 0
