"""Ring cursor of a multi-stage pipeline: (index, phase, count).

Test infrastructure (see ``oracle/__init__.py``).

Source: "cute(12) async_pipeline" -- §2.1 (the triple), §2.2 (the step rule and
its 3-stage table), §2.3 and §6.1 (start states and the batched advance).

The cursor names the stage a role works on next and the parity it waits with.
Stepping moves to the next stage; passing the last stage wraps to stage 0 and
inverts the phase bit, in step with the mbarrier, whose phase also advances
once per completed round.  The producer starts with phase 1 because every
buffer is free at the start, the consumer with phase 0.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass
class PipelineState:
    stages: int
    index: int = 0
    phase: int = 0
    count: int = 0

    def __post_init__(self) -> None:
        if self.stages < 1:
            raise ValueError("a pipeline has at least one stage")
        if not 0 <= self.index < self.stages:
            raise ValueError("index out of range")
        if self.phase not in (0, 1):
            raise ValueError("phase is a single bit")

    def step(self) -> "PipelineState":
        """The ``++`` of §2.2: next stage; wrapping past the last stage flips
        the phase bit.  The count is the number of steps taken so far."""
        self.index += 1
        self.count += 1
        if self.index == self.stages:
            self.index = 0
            self.phase ^= 1
        return self

    def advance(self, n: int) -> "PipelineState":
        """Take ``n`` steps at once (§6.1).  The phase flips once per wrap of
        the ring, so it flips iff the number of wraps, (index + n) // stages,
        is odd."""
        if n < 0:
            raise ValueError("a cursor only moves forward")
        wraps = (self.index + n) // self.stages
        self.phase ^= wraps & 1
        self.index = (self.index + n) % self.stages
        self.count += n
        return self

    def copy(self) -> "PipelineState":
        return PipelineState(self.stages, self.index, self.phase, self.count)

    def as_tuple(self) -> tuple[int, int, int]:
        return (self.index, self.phase, self.count)


def producer_start(stages: int) -> PipelineState:
    """§2.3: the producer starts at stage 0 with the *opposite* phase (1),
    because all buffers are free before anything has been written."""
    return PipelineState(stages, 0, 1, 0)


def consumer_start(stages: int) -> PipelineState:
    """§3.2: the consumer starts from the default cursor (0, 0, 0)."""
    return PipelineState(stages, 0, 0, 0)


def closed_form(stages: int, start_phase: int, t: int) -> tuple[int, int, int]:
    """State after ``t`` steps from (0, start_phase, 0): stage t mod S, phase
    flipped once per completed pass over the ring."""
    return (t % stages, start_phase ^ ((t // stages) & 1), t)


def sequence(stages: int, start_phase: int, n: int) -> list[tuple[int, int]]:
    """The (index, phase) a role uses for its first ``n`` tiles, by stepping."""
    st = PipelineState(stages, 0, start_phase, 0)
    out = []
    for _ in range(n):
        out.append((st.index, st.phase))
        st.step()
    return out
