"""Oracle of commit-aware KV tiering: integer bookkeeping, exact.

TEST INFRASTRUCTURE: only the tests may import this module; the product path
never does.

Source: "Resource-Efficient Speculative Decoding for Long-Context LLM
Serving", section 4.1 "Commit-Aware Rollback-Free KV Tiering", Eqs. (4)-(5).

Each request's Target KV is split into three regions (Eq. 4):
Sealed History [0, H) on the CPU, Active Tail [H, C_r) and Speculative
Frontier [C_r, L_r) on the GPU, with 0 <= H <= C_r <= L_r.  The migration
endpoint is E = max{H, g * floor(max(0, C_r - T) / g)} (Eq. 5): when E > H the
interval [H, E) is copied to the CPU asynchronously, and H advances to E only
once that copy has completed.  At the end of a round the committed prefix
becomes C'_r with C_r <= C'_r <= L_r, and the rejected suffix [C'_r, L_r) is
released on the GPU; it never meets [0, H).

Readings: "H already aligned to g" is taken as a precondition (H is a multiple
of g, which holds when H starts at 0 and only ever advances to an E);
T >= 0 and g >= 1.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Tuple


def migration_endpoint(H: int, C: int, T: int, g: int) -> int:
    """Eq. (5): E = max{H, g * floor(max(0, C - T) / g)}."""
    if g < 1 or T < 0 or H < 0 or C < H or H % g:
        raise ValueError("need g >= 1, T >= 0, 0 <= H <= C and H a multiple of g")
    return max(H, g * (max(0, C - T) // g))


def migration_interval(H: int, C: int, T: int, g: int) -> Optional[Tuple[int, int]]:
    """[H, E) when E > H, else None (the state is left unchanged)."""
    E = migration_endpoint(H, C, T, g)
    return (H, E) if E > H else None


@dataclasses.dataclass
class TierState:
    """One request's region boundaries; `pending` is the endpoint of a migration in flight."""

    H: int = 0
    C: int = 0
    L: int = 0
    pending: Optional[int] = None

    def check(self):
        if not (0 <= self.H <= self.C <= self.L):
            raise ValueError("regions must satisfy 0 <= H <= C_r <= L_r")

    def round(self, C: int, L: int):
        """A new round: the committed prefix and the logical length including candidates."""
        if C < self.C or L < C:
            raise ValueError("the committed prefix never shrinks and L_r >= C_r")
        self.C, self.L = C, L
        self.check()

    def plan(self, T: int, g: int) -> Optional[Tuple[int, int]]:
        """Start a migration if Eq. (5) asks for one and none is in flight."""
        if self.pending is not None:
            return None
        iv = migration_interval(self.H, self.C, T, g)
        if iv is not None:
            self.pending = iv[1]
        return iv

    def copy_completed(self):
        """H advances only after the copy has completed (section 4.1)."""
        if self.pending is not None:
            self.H, self.pending = self.pending, None

    def commit(self, C_new: int) -> Tuple[int, int]:
        """End of round: keep [0, C_new), release [C_new, L_r); returns the released interval."""
        if not (self.C <= C_new <= self.L):
            raise ValueError("the retained prefix C'_r lies in [C_r, L_r]")
        released = (C_new, self.L)
        if released[0] < self.H:  # cannot happen while H <= C_r <= C'_r
            raise AssertionError("rollback would touch CPU history")
        self.C = self.L = C_new
        return released
