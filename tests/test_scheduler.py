"""Target-priority Draft admission ("Resource-Efficient Speculative Decoding for Long-Context LLM
Serving", section 4.3): the oracle pinned on hand-checked scenarios of the page's rules, and the
library's decisions equal to the oracle's on random event sequences (host-only, no GPU)."""
import os

import numpy as np
import pytest

from oracle.scheduler import Scheduler

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_rules_by_hand():
    s = Scheduler(eps_T=0.05, delta=0.1, ema=0.5, t_D=1.0, dT=0.02, alloc=34)
    # window too short: 1.0 + 0.1 > 1.05
    assert s.try_admit(0, 7, now=10.0, S_hat=1.05) is None
    ins = s.try_admit(0, 7, now=10.0, S_hat=2.0)
    assert (ins.req, ins.round, ins.seq, ins.alloc) == (0, 7, 1, 34)
    assert ins.t_latest == 10.0 + 2.0 - 1.0 - 0.1
    # one unfinished step per request; another request is independent
    assert s.try_admit(0, 7, 10.0, 5.0) is None
    assert s.try_admit(1, 7, 10.0, 5.0).seq == 1
    # a stale ACK changes nothing; the right one closes the step and updates t_D
    assert not s.ack(0, 99, 3.0)
    assert s.ack(0, 1, 2.0) and s.t_D == 1.5
    # expiry and mismatch are refused at start and release the request
    ins = s.try_admit(0, 7, now=20.0, S_hat=2.0)  # t_latest = 20 + 2 - 1.5 - 0.1 = 20.4
    assert ins.t_latest == pytest.approx(20.4)
    assert not s.check_start(ins, 0, 7, now=20.5)
    assert s.try_admit(0, 7, 21.0, 3.0) is not None
    other = s.try_admit(2, 7, now=0.0, S_hat=10.0)
    assert not s.check_start(other, 2, 8, now=0.0)  # the round has moved on
    assert s.try_admit(2, 8, 0.0, 10.0) is not None
    # an over-budget Target observation pauses submission until a later round within budget
    s.observe_target(1.2, 1.0)  # +20% > 5%
    assert s.paused and s.dT == pytest.approx(0.02 + 0.5 * (0.2 - 0.02))
    assert s.try_admit(5, 8, 0.0, 100.0) is None
    s.new_round()
    assert s.paused  # estimate 0.11 still above 0.05
    s.observe_target(1.0, 1.0)
    s.observe_target(1.0, 1.0)  # dT -> 0.0275
    s.new_round()
    assert not s.paused and s.try_admit(5, 9, 0.0, 100.0) is not None


def test_library_matches_oracle_on_random_sequences():
    from speculative_decoding_verification_chunked_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from speculative_decoding_verification_chunked_gb300 import svx
    rng = np.random.default_rng(7)
    for trial in range(60):
        cfg = dict(eps_T=float(rng.uniform(0, 0.2)), delta=float(rng.uniform(0, 0.5)), ema=float(rng.uniform(0.1, 1)),
                   t_D=float(rng.uniform(0.2, 2)), dT=float(rng.uniform(0, 0.2)), alloc=int(rng.integers(1, 60)))
        o = Scheduler(**cfg)
        lib = svx.Scheduler(cfg["eps_T"], cfg["delta"], cfg["ema"], cfg["t_D"], cfg["dT"], cfg["alloc"])
        issued = []
        now, rnd = 0.0, 0
        for _ in range(400):
            ev = rng.integers(0, 5)
            now += float(rng.uniform(0, 0.5))
            if ev == 0:
                req, S = int(rng.integers(0, 4)), float(rng.uniform(0, 3))
                a, b = o.try_admit(req, rnd, now, S), lib.try_admit(req, rnd, now, S)
                assert (a is None) == (b is None)
                if a is not None:
                    assert (a.req, a.round, a.seq, a.alloc) == (b.req, b.round, b.seq, b.alloc)
                    assert a.t_latest == b.t_latest
                    issued.append((a, b))
            elif ev == 1 and issued:
                a, b = issued[int(rng.integers(0, len(issued)))]
                cur_req, cur_round = (a.req, rnd) if rng.random() < 0.8 else (a.req + 1, rnd)
                t = now + float(rng.uniform(-1, 1))
                assert o.check_start(a, cur_req, cur_round, t) == lib.check_start(b, cur_req, cur_round, t)
            elif ev == 2 and issued:
                a, _ = issued[int(rng.integers(0, len(issued)))]
                seq = a.seq if rng.random() < 0.8 else a.seq + 1
                t = float(rng.uniform(0.1, 3))
                assert o.ack(a.req, seq, t) == lib.ack(a.req, seq, t)
            elif ev == 3:
                ta = float(rng.uniform(1, 2))
                tc = ta * float(rng.uniform(0.95, 1.3))
                o.observe_target(tc, ta)
                lib.observe_target(tc, ta)
            else:
                rnd += 1
                o.new_round()
                lib.new_round()
            t_D, dT, paused = lib.estimates()
            assert (t_D, dT, paused) == (o.t_D, o.dT, o.paused)
