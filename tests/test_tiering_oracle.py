"""Pins of the tiering oracle ("Resource-Efficient Speculative Decoding for Long-Context LLM
Serving", section 4.1, Eqs. 4-5): hand-worked endpoints, the closed-form tail bound that
follows from Eq. 5, and the region invariants over random rounds."""
import numpy as np
import pytest

from oracle.tiering import TierState, migration_endpoint, migration_interval


@pytest.mark.parametrize("H,C,T,g,E", [
    (0, 1000, 512, 128, 384),    # 488 // 128 = 3 -> 384
    (384, 1000, 512, 128, 384),  # nothing new to migrate
    (384, 1200, 512, 128, 640),  # 688 // 128 = 5 -> 640
    (0, 300, 512, 128, 0),       # committed prefix shorter than the tail target
    (0, 512, 512, 128, 0),
    (0, 640, 512, 128, 128),
    (0, 7, 0, 1, 7),             # g = 1, T = 0: everything committed moves
    (64, 64, 0, 64, 64),
])
def test_endpoint_hand_examples(H, C, T, g, E):
    assert migration_endpoint(H, C, T, g) == E
    iv = migration_interval(H, C, T, g)
    assert iv == ((H, E) if E > H else None)


def test_endpoint_tail_bound_and_alignment():
    rng = np.random.default_rng(0)
    for _ in range(5000):
        g = int(rng.choice([1, 16, 64, 128, 256]))
        T = int(rng.integers(0, 2048))
        H = g * int(rng.integers(0, 100))
        C = H + int(rng.integers(0, 5000))
        E = migration_endpoint(H, C, T, g)
        assert E >= H and E % g == 0 and E <= C
        if E > H:  # the GPU keeps between T and T + g - 1 committed tokens
            assert T <= C - E < T + g
        else:
            assert g * (max(0, C - T) // g) <= H


def test_bad_arguments():
    for args in [(0, 10, 5, 0), (3, 10, 5, 2), (5, 4, 0, 1), (0, 10, -1, 1)]:
        with pytest.raises(ValueError):
            migration_endpoint(*args)


def test_regions_over_random_rounds():
    rng = np.random.default_rng(1)
    for trial in range(200):
        T, g = 512, int(rng.choice([64, 128]))
        s = TierState()
        for _ in range(60):
            k = int(rng.integers(1, 9))
            s.round(s.C, s.C + k)  # k candidates appended after the committed prefix
            iv = s.plan(T, g)
            if iv is not None:
                assert iv[0] == s.H and s.pending == iv[1]
                assert s.H <= s.C  # until the copy completes H does not move
            if rng.random() < 0.7:
                s.copy_completed()
            accepted = int(rng.integers(0, k + 1))
            rel = s.commit(s.C + accepted)
            assert rel[0] >= s.H and rel[0] == s.C  # rollback never reaches CPU history
            s.check()
        s.copy_completed()
        assert s.H % g == 0 and s.C - s.H >= 0


def test_state_rejects_impossible_transitions():
    s = TierState()
    s.round(10, 15)
    with pytest.raises(ValueError):
        s.round(9, 15)  # committed prefix cannot shrink
    with pytest.raises(ValueError):
        s.commit(16)    # beyond the logical length
    with pytest.raises(ValueError):
        s.commit(9)     # below the committed prefix
