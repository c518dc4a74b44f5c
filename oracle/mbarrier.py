"""Behavioural model of one mbarrier object.

Test infrastructure (see ``oracle/__init__.py``).

Sources:
* "异步协作：mbarrier" (Async coordination: mbarrier), section "mbarrier": the
  barrier keeps a count of arrivals still owed in the current phase, a phase
  number, and (for bulk copies) a tx-count of bytes still in flight; init sets
  phase 0 and the owed count to the expected count; ``arrive.expect_tx`` both
  arrives once and registers bytes; the copy engine subtracts delivered bytes,
  possibly in several parts; the phase completes only when the owed arrivals
  and the tx-count are both zero, after which the next phase starts with the
  expected count again.
* "cute(12) async_pipeline", §6.2 (init / wait / arrive) and §6.3
  (arrive_and_expect_tx, complete_tx): ``wait(parity)`` returns once the
  barrier's current phase parity differs from the argument.

Readings (also listed with the design notes):
* ``arrive_expect_tx`` applies both of its effects before the completion test,
  so a single arrive that registers bytes cannot complete the phase by itself.
* The tx-count may go transiently negative when delivered bytes are counted
  before the matching expect; completion is tested only on (owed == 0 and
  tx == 0).
* More arrivals than the expected count in one phase is a protocol error.
"""
from __future__ import annotations


class ProtocolError(RuntimeError):
    pass


class MBarrier:
    def __init__(self, expected: int) -> None:
        if expected < 1:
            raise ValueError("an mbarrier expects at least one arrival")
        self.expected = expected
        self.pending = expected
        self.tx = 0
        self.phase = 0          # unbounded phase number
        self.completions = 0    # == phase; kept for readability in traces

    # -- state -------------------------------------------------------------
    @property
    def parity(self) -> int:
        return self.phase & 1

    def _settle(self) -> bool:
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.completions += 1
            self.pending = self.expected
            return True
        return False

    # -- operations --------------------------------------------------------
    def arrive(self, count: int = 1) -> bool:
        """Arrive ``count`` times; returns True if this completed the phase."""
        if count < 1 or count > self.pending:
            raise ProtocolError("more arrivals than the phase expects")
        self.pending -= count
        return self._settle()

    def arrive_expect_tx(self, nbytes: int) -> bool:
        if self.pending < 1:
            raise ProtocolError("more arrivals than the phase expects")
        self.tx += nbytes
        self.pending -= 1
        return self._settle()

    def expect_tx(self, nbytes: int) -> bool:
        self.tx += nbytes
        return self._settle()

    def complete_tx(self, nbytes: int) -> bool:
        self.tx -= nbytes
        return self._settle()

    def test_wait_parity(self, parity: int) -> bool:
        """True once the phase with this parity has completed, i.e. the
        current phase parity is no longer ``parity``."""
        return self.parity != (parity & 1)
