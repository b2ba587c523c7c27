"""Oracle of Target-priority Draft admission: host-side decision rules.

TEST INFRASTRUCTURE: only the tests may import this module.

Source: "Resource-Efficient Speculative Decoding for Long-Context LLM
Serving", section 4.3 "Target-Priority Intra-GPU Co-Execution", paragraphs
"Target-priority scheduling" and the two that follow it.

Rules, as the page states them:
  * A Draft step may start under the selected allocation n0 only if the
    estimated Target latency increase is within budget, dT_hat <= eps_T, and
    the estimated Draft single-step time plus a margin fits the remaining
    window, t_D_hat + delta <= S_hat.
  * One Draft step (one token) is admitted at a time; at most one unfinished
    step per request.
  * The instruction carries (request, round, sequence number, allocation,
    latest start time), t_latest = t0 + S_hat - t_D_hat - delta.  Before
    starting, the Draft checks that the instruction still matches the current
    request and round and that t_latest has not passed; otherwise the
    instruction is not executed.
  * An ACK carrying the sequence number closes the step; only then may the
    Target schedule another one for that request.
  * Execution results update the estimates.  If the observed Target latency
    increase exceeds the budget, no new concurrent step is submitted until
    the Target's state allows it again.

Readings where the page leaves a step open (each is listed in the design
notes): the estimates are exponential moving averages with weight `ema` on
the newest observation, x <- x + ema * (obs - x); an expired or mismatched
instruction also releases the request's slot; a pause set by an over-budget
observation lasts until the next round whose estimate is back within budget.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional


@dataclasses.dataclass
class Instruction:
    req: int
    round: int
    seq: int
    alloc: int
    t_latest: float


@dataclasses.dataclass
class Scheduler:
    eps_T: float
    delta: float
    ema: float
    t_D: float   # Draft single-step time under the allocation (offline record, then updated)
    dT: float    # Target latency increase under the allocation (offline record, then updated)
    alloc: int   # the selected allocation n0
    paused: bool = False
    in_flight: Dict[int, int] = dataclasses.field(default_factory=dict)  # req -> seq
    seq: Dict[int, int] = dataclasses.field(default_factory=dict)

    def new_round(self):
        """A new verification round: a pause ends once the estimate is back within budget."""
        if self.paused and self.dT <= self.eps_T:
            self.paused = False

    def try_admit(self, req: int, rnd: int, now: float, S_hat: float) -> Optional[Instruction]:
        if self.paused or req in self.in_flight:
            return None
        if not (self.dT <= self.eps_T and self.t_D + self.delta <= S_hat):
            return None
        s = self.seq.get(req, 0) + 1
        self.seq[req] = s
        self.in_flight[req] = s
        return Instruction(req, rnd, s, self.alloc, now + S_hat - self.t_D - self.delta)

    def check_start(self, ins: Instruction, cur_req: int, cur_round: int, now: float) -> bool:
        """Draft side, before starting: run only a current, unexpired instruction."""
        ok = ins.req == cur_req and ins.round == cur_round and now <= ins.t_latest
        if not ok and self.in_flight.get(ins.req) == ins.seq:
            del self.in_flight[ins.req]
        return ok

    def ack(self, req: int, seq: int, t_obs: float) -> bool:
        """Completion of one Draft step; stale or unknown ACKs change nothing."""
        if self.in_flight.get(req) != seq:
            return False
        del self.in_flight[req]
        self.t_D = self.t_D + self.ema * (t_obs - self.t_D)
        return True

    def observe_target(self, T_co: float, T_alone: float):
        d = (T_co - T_alone) / T_alone
        self.dT = self.dT + self.ema * (d - self.dT)
        if d > self.eps_T:
            self.paused = True
