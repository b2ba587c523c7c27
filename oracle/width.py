"""Oracle of the I/O-aware dynamic verification width controller.

TEST INFRASTRUCTURE: only the tests may import this module.

Source: "Resource-Efficient Speculative Decoding for Long-Context LLM
Serving", section 4.2, paragraph "I/O-aware dynamic verification widths"
(and Eq. 3 for the transfer amortisation it follows).

The controller picks the width for the next round as
    q* = argmin_{q in Q} T_round_hat(q) / U_hat(q),
the estimated round time over the estimated number of committed tokens.
Statistics are updated at the end of each round; widths without records are
first tried in a limited initial sampling phase; the width changes only when
the estimated benefit exceeds the switching threshold.

Readings where the page leaves the formulas open (listed in the design notes):
  * the round time is Draft generation + max(history transfer, attention) +
    rejection correction, so transfer and the attention it overlaps are not
    counted twice (section 4.2: "without counting overlapped time twice");
  * each component and the committed count are exponential moving averages
    with weight `ema` on the newest record (the page: "recent" costs);
  * initial sampling tries each width n_init times, in the order given;
  * "benefit exceeds the threshold": switch from the current width q_c to q*
    only if cost(q*) < (1 - threshold) * cost(q_c);
  * ties in the argmin go to the earlier width in Q.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional


@dataclasses.dataclass
class WidthStats:
    n: int = 0
    t_draft: float = 0.0
    t_h2d: float = 0.0
    t_attn: float = 0.0
    t_correct: float = 0.0
    committed: float = 0.0


class WidthController:
    def __init__(self, widths: List[int], ema: float, threshold: float, n_init: int):
        if not widths or not (0.0 < ema <= 1.0) or threshold < 0.0 or n_init < 1:
            raise ValueError("bad controller configuration")
        self.widths = list(widths)
        self.ema, self.threshold, self.n_init = ema, threshold, n_init
        self.stats: Dict[int, WidthStats] = {q: WidthStats() for q in self.widths}
        self.current = self.widths[0]

    def _upd(self, old: float, new: float, first: bool) -> float:
        return new if first else old + self.ema * (new - old)

    def record(self, q: int, t_draft: float, t_h2d: float, t_attn: float, t_correct: float, committed: float):
        """End-of-round statistics of a round verified at width q."""
        s = self.stats[q]
        first = s.n == 0
        s.t_draft = self._upd(s.t_draft, t_draft, first)
        s.t_h2d = self._upd(s.t_h2d, t_h2d, first)
        s.t_attn = self._upd(s.t_attn, t_attn, first)
        s.t_correct = self._upd(s.t_correct, t_correct, first)
        s.committed = self._upd(s.committed, committed, first)
        s.n += 1

    def cost(self, q: int) -> Optional[float]:
        """T_round_hat(q) / U_hat(q), or None without records (or no committed tokens yet)."""
        s = self.stats[q]
        if s.n == 0 or s.committed <= 0.0:
            return None
        return (s.t_draft + max(s.t_h2d, s.t_attn) + s.t_correct) / s.committed

    def next_width(self) -> int:
        for q in self.widths:  # limited initial sampling
            if self.stats[q].n < self.n_init:
                self.current = q
                return q
        best, best_cost = None, None
        for q in self.widths:
            c = self.cost(q)
            if c is not None and (best_cost is None or c < best_cost):
                best, best_cost = q, c
        cur_cost = self.cost(self.current)
        if best is not None and (cur_cost is None or best_cost < (1.0 - self.threshold) * cur_cost):
            self.current = best
        return self.current
