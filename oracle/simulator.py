"""Discrete-event model of one warp-specialised CTA running the tile pipeline.

Test infrastructure (see ``oracle/__init__.py``).

Agents and their programs follow "cute(12) async_pipeline" §3 (producer and
consumer loops), §6.6-6.9 (producer_acquire, consumer_wait, consumer_release,
producer_tail) and the mbarrier rules of "异步协作：mbarrier":

* producer (one elected thread), per tile t with cursor (s, p):
  wait empty[s] with parity p; arrive.expect_tx(full[s], tile bytes); hand the
  copy to the copy engine; step the cursor.  After the last tile it waits on
  every stage's empty barrier once more (the tail), stepping in between.
* copy engine: delivers each issued tile in one or two parts, in any order
  across tiles; every part lands in the stage buffer and then subtracts its
  bytes from full[s]'s tx-count.
* consumers (``consumers`` agents: one per thread or one per warp, depending on
  how the empty barrier is counted), per tile t with cursor (s, p): wait
  full[s] with parity p; read the stage; arrive on empty[s]; step.

The scheduler picks, at every step, one runnable action uniformly at random
(seeded).  A wait is runnable only when its parity test passes.  When nothing
is runnable and some agent has not finished, the run is a deadlock.

Checked at every step:
  (i)   a consumer reads stage s for tile t only when the buffer holds all the
        bytes of tile t;
  (ii)  the producer hands tile t to the copy engine only after every consumer
        has released tile t - S from the same stage;
  (iii) the producer is never more than S tiles ahead of the slowest consumer
        ("cute(12) async_pipeline" §1.2);
  (iv)  the (index, phase) each role used for each tile is recorded, so tests
        can compare it with the cursor's closed form.
"""
from __future__ import annotations

import random
from dataclasses import dataclass, field

from .mbarrier import MBarrier, ProtocolError
from .pipeline_state import PipelineState


@dataclass
class SimResult:
    status: str                      # "done" | "deadlock" | "budget" | "error"
    steps: int
    producer_log: list = field(default_factory=list)   # (t, index, phase)
    consumer_logs: list = field(default_factory=list)  # per consumer
    max_lead: int = 0
    violations: list = field(default_factory=list)
    full_phases: list = field(default_factory=list)
    empty_phases: list = field(default_factory=list)


def simulate(stages: int, tiles: int, consumers: int, *, seed: int = 0,
             tile_bytes: int = 16384, producer_start_phase: int = 1,
             consumer_start_phase: int = 0, full_count: int = 1,
             empty_count: int | None = None, releasing: int | None = None,
             split_parts: bool = True, max_steps: int | None = None,
             tail: bool = True) -> SimResult:
    """Run one CTA's pipeline under a random interleaving.

    ``full_count`` / ``empty_count`` are the expected arrival counts of the
    barriers; ``releasing`` is how many consumers actually arrive on empty
    (default: all of them).  The defaults are the correct protocol; the
    deadlock scenarios of the lesson are obtained by changing one of them.
    """
    rng = random.Random(seed)
    empty_count = consumers if empty_count is None else empty_count
    releasing = consumers if releasing is None else releasing
    if max_steps is None:
        max_steps = 50 * (tiles + stages + 2) * (consumers + 4)

    full = [MBarrier(full_count) for _ in range(stages)]
    empty = [MBarrier(empty_count) for _ in range(stages)]
    buf_tile = [-1] * stages           # tile whose bytes the buffer holds
    buf_bytes = [0] * stages           # bytes of that tile already landed
    released = [set() for _ in range(stages)]  # consumers done with buf tile
    issued_tile = [-1] * stages        # last tile handed to the copy engine
    reading = [set() for _ in range(stages)]

    res = SimResult(status="done", steps=0,
                    consumer_logs=[[] for _ in range(consumers)])

    # producer program counter
    prod = {"t": 0, "op": "wait", "st": PipelineState(stages, 0, producer_start_phase, 0),
            "tail_left": stages if tail else 0}
    cons = [{"t": 0, "op": "wait", "st": PipelineState(stages, 0, consumer_start_phase, 0)}
            for _ in range(consumers)]
    done_count = [0] * consumers        # tiles fully released per consumer
    engine: list[tuple[int, int, int]] = []   # (stage, tile, bytes)

    def producer_actions():
        if prod["op"] == "done":
            return []
        st = prod["st"]
        if prod["op"] in ("wait", "tail"):
            if empty[st.index].test_wait_parity(st.phase):
                return [("prod_" + prod["op"],)]
            return []
        return [("prod_" + prod["op"],)]

    def consumer_actions(c):
        cs = cons[c]
        if cs["op"] == "done":
            return []
        st = cs["st"]
        if cs["op"] == "wait":
            if full[st.index].test_wait_parity(st.phase):
                return [("cons_wait", c)]
            return []
        return [("cons_" + cs["op"], c)]

    def all_done():
        return prod["op"] == "done" and all(c["op"] == "done" for c in cons)

    # initial transitions for zero-tile runs
    if tiles == 0:
        prod["op"] = "tail" if prod["tail_left"] else "done"
        for c in cons:
            c["op"] = "done"

    try:
        while not all_done():
            if res.steps >= max_steps:
                res.status = "budget"
                break
            acts = producer_actions()
            for c in range(consumers):
                acts += consumer_actions(c)
            acts += [("engine", i) for i in range(len(engine))]
            if not acts:
                res.status = "deadlock"
                break
            act = rng.choice(acts)
            res.steps += 1
            kind = act[0]
            if kind == "prod_wait":
                prod["op"] = "arrive"
            elif kind == "prod_arrive":
                st = prod["st"]
                full[st.index].arrive_expect_tx(tile_bytes)
                prod["op"] = "issue"
            elif kind == "prod_issue":
                st = prod["st"]
                t, s = prod["t"], st.index
                # (ii): the previous tile of this stage is released by all
                prev = issued_tile[s]
                if prev >= 0 and (len(released[s]) < consumers or reading[s]):
                    res.violations.append(f"overwrite of stage {s} (tile {prev}) by tile {t}")
                # (iii)
                lead = (t + 1) - min(done_count)
                res.max_lead = max(res.max_lead, lead)
                if lead > stages:
                    res.violations.append(f"producer leads by {lead} at tile {t}")
                res.producer_log.append((t, st.index, st.phase))
                issued_tile[s] = t
                released[s] = set()
                buf_tile[s] = t
                buf_bytes[s] = 0
                if split_parts and tile_bytes >= 2 and rng.random() < 0.5:
                    first = rng.randrange(1, tile_bytes)
                    engine.append((s, t, first))
                    engine.append((s, t, tile_bytes - first))
                else:
                    engine.append((s, t, tile_bytes))
                st.step()
                prod["t"] += 1
                if prod["t"] == tiles:
                    prod["op"] = "tail" if prod["tail_left"] else "done"
                else:
                    prod["op"] = "wait"
            elif kind == "prod_tail":
                prod["st"].step()
                prod["tail_left"] -= 1
                if prod["tail_left"] == 0:
                    prod["op"] = "done"
            elif kind == "engine":
                s, t, nbytes = engine.pop(act[1])
                if buf_tile[s] == t:
                    buf_bytes[s] += nbytes
                full[s].complete_tx(nbytes)
            elif kind == "cons_wait":
                c = act[1]
                cs = cons[c]
                st = cs["st"]
                s, t = st.index, cs["t"]
                # (i)
                if buf_tile[s] != t or buf_bytes[s] != tile_bytes:
                    res.violations.append(
                        f"consumer {c} read stage {s} for tile {t} holding tile "
                        f"{buf_tile[s]} with {buf_bytes[s]} bytes")
                res.consumer_logs[c].append((t, st.index, st.phase))
                reading[s].add(c)
                cs["op"] = "release"
            elif kind == "cons_release":
                c = act[1]
                cs = cons[c]
                st = cs["st"]
                s = st.index
                reading[s].discard(c)
                released[s].add(c)
                if c < releasing:
                    empty[s].arrive()
                done_count[c] += 1
                st.step()
                cs["t"] += 1
                cs["op"] = "done" if cs["t"] == tiles else "wait"
    except ProtocolError as exc:
        res.status = "error"
        res.violations.append(str(exc))

    res.full_phases = [b.phase for b in full]
    res.empty_phases = [b.phase for b in empty]
    return res


def lockstep_timeline(stages: int, tiles: int, consumers: int = 96,
                      tile_bytes: int = 16384) -> list[dict]:
    """Run producer, copy engine and consumers strictly one tile after another
    and record, per tile, what each barrier showed -- the quantities of the
    8-tile barrier timeline in "cute(12) async_pipeline" §7.6."""
    full = [MBarrier(1) for _ in range(stages)]
    empty = [MBarrier(consumers) for _ in range(stages)]
    pw = PipelineState(stages, 0, 1, 0)
    pr = PipelineState(stages, 0, 0, 0)
    rows = []
    for t in range(tiles):
        s = pw.index
        row = {"tile": t, "write": (pw.index, pw.phase)}
        row["empty_parity_at_wait"] = empty[s].parity
        row["producer_blocks"] = not empty[s].test_wait_parity(pw.phase)
        full_before = full[s].parity
        full[s].arrive_expect_tx(tile_bytes)
        assert full[s].parity == full_before, "expect_tx alone must not complete"
        full[s].complete_tx(tile_bytes)
        row["full_flip"] = (full_before, full[s].parity)
        pw.step()
        cs = pr.index
        row["read"] = (pr.index, pr.phase)
        row["full_parity_at_wait"] = full[cs].parity
        row["consumer_passes"] = full[cs].test_wait_parity(pr.phase)
        empty_before = empty[cs].parity
        for _ in range(consumers):
            empty[cs].arrive()
        row["empty_flip"] = (empty_before, empty[cs].parity)
        pr.step()
        rows.append(row)
    return rows


def two_stage_parity_table(iterations: int = 4) -> list[tuple[int, int, int, int, int]]:
    """Reproduce the 2-stage parity walk of "异步协作：mbarrier" (section on
    how phases tell rounds apart): one full barrier per stage, both starting in
    phase 0, a consumer cursor that flips its parity after each pass over the
    two stages.  Rows: (iteration, stage, parity waited on, barrier parity
    after its phase completes, cursor parity at the end of the iteration)."""
    bars = [MBarrier(1), MBarrier(1)]
    cur = PipelineState(2, 0, 0, 0)
    rows = []
    for it in range(iterations):
        s, waited = cur.index, cur.phase
        bars[s].arrive_expect_tx(2048)
        bars[s].complete_tx(2048)
        assert bars[s].test_wait_parity(waited)
        cur.step()
        rows.append((it, s, waited, bars[s].parity, cur.phase))
    return rows


@dataclass
class RingResult:
    status: str                      # "done" | "deadlock" | "budget"
    steps: int
    taken: list = field(default_factory=list)        # keys in the order the reader took them
    violations: list = field(default_factory=list)


def simulate_flush_ring(slots: int, records: int, writers: int, *, seed: int = 0,
                        writer_start_parity: int = 1, reader_start_parity: int = 0,
                        full_count: int | None = None, max_steps: int | None = None
                        ) -> RingResult:
    """Discrete-event model of the sums' flush ring: ``writers`` consumer
    warps hand ``records`` records to one flush warp through ``slots``
    shared-memory slots, with the full/empty mbarrier protocol of the tile
    ring ("cute(12) async_pipeline" §3, §6) run the other way round.

    * writer w, record k (slot k mod slots, parity (k div slots) mod 2 XOR
      writer_start_parity): wait empty[slot]; write its share of the slot
      (tagged with k); arrive on full[slot].
    * reader, record k (same slot, parity (k div slots) mod 2 XOR
      reader_start_parity): wait full[slot]; read every writer's share; arrive
      on empty[slot] (expected count 1).

    full[slot] expects ``full_count`` arrivals (default: one per writer).
    Checked: the reader takes records in order and finds every share of
    record k tagged k (no share overwritten by record k + slots before it was
    read, none missing)."""
    rng = random.Random(seed)
    fc = writers if full_count is None else full_count
    full = [MBarrier(fc) for _ in range(slots)]
    empty = [MBarrier(1) for _ in range(slots)]
    share = [[None] * writers for _ in range(slots)]
    wk = [0] * writers          # next record of each writer
    wstate = ["wait"] * writers  # "wait" (empty) then "arrive" (full)
    rk = 0
    rstate = "wait"
    res = RingResult(status="done", steps=0)
    budget = max_steps or 100 * (records + 1) * (writers + 2) * slots
    for step in range(budget):
        acts = []
        for w in range(writers):
            if wk[w] >= records:
                continue
            s, par = wk[w] % slots, ((wk[w] // slots) & 1) ^ writer_start_parity
            if wstate[w] == "wait":
                if empty[s].test_wait_parity(par):
                    acts.append(("w", w))
            else:
                acts.append(("w", w))
        if rk < records:
            s, par = rk % slots, ((rk // slots) & 1) ^ reader_start_parity
            if rstate == "wait":
                if full[s].test_wait_parity(par):
                    acts.append(("r", 0))
            else:
                acts.append(("r", 0))
        if not acts:
            res.steps = step
            if rk < records or any(k < records for k in wk):
                res.status = "deadlock"
            return res
        who, i = rng.choice(acts)
        try:
            if who == "w":
                s = wk[i] % slots
                if wstate[i] == "wait":       # passed the empty wait: write the share
                    share[s][i] = wk[i]
                    wstate[i] = "arrive"
                else:
                    full[s].arrive()
                    wstate[i] = "wait"
                    wk[i] += 1
            else:
                s = rk % slots
                if rstate == "wait":          # passed the full wait: read every share
                    got = list(share[s])
                    if got != [rk] * writers:
                        res.violations.append((rk, got))
                    res.taken.append(rk)
                    rstate = "arrive"
                else:
                    empty[s].arrive()
                    rstate = "wait"
                    rk += 1
        except ProtocolError as e:
            res.violations.append(("protocol", str(e)))
            res.status = "error"
            res.steps = step
            return res
    res.status = "budget"
    res.steps = budget
    return res
