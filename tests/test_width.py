"""Dynamic verification width ("Resource-Efficient Speculative Decoding for Long-Context LLM
Serving", section 4.2): the oracle pinned on a noise-free synthetic round model whose optimum is
known in closed form, and the library's choices equal to the oracle's (host-only, no GPU)."""
import os

import numpy as np
import pytest

from oracle.width import WidthController

WIDTHS = [2, 4, 6, 8]


def expected_committed(q, a):
    """Tokens committed by a round of width q when each draft token is accepted independently with
    probability a: the accepted prefix plus the Target's own token, sum_{i=0..q} a^i."""
    return (1 - a ** (q + 1)) / (1 - a)


def round_terms(q, a, t_h2d=5.0, c_draft=0.3, attn0=0.2, attn_q=0.05, corr=0.1):
    return q * c_draft, t_h2d, attn0 + attn_q * q, corr, expected_committed(q, a)


@pytest.mark.parametrize("a", [0.3, 0.6, 0.8, 0.95])
def test_noise_free_model_converges_to_the_closed_form_optimum(a):
    c = WidthController(WIDTHS, ema=0.5, threshold=0.0, n_init=1)
    for _ in range(12):
        q = c.next_width()
        c.record(q, *round_terms(q, a))
    costs = {q: (lambda d, h, at, co, u: (d + max(h, at) + co) / u)(*round_terms(q, a)) for q in WIDTHS}
    assert c.next_width() == min(WIDTHS, key=lambda q: costs[q])
    for q in WIDTHS:
        assert c.cost(q) == pytest.approx(costs[q], rel=1e-12)


def test_initial_sampling_order_and_threshold():
    c = WidthController(WIDTHS, ema=1.0, threshold=0.2, n_init=2)
    seen = []
    for _ in range(8):
        q = c.next_width()
        seen.append(q)
        c.record(q, 1.0, 4.0, 0.5, 0.0, {2: 2.0, 4: 2.5, 6: 2.6, 8: 2.7}[q])
    assert seen == [2, 2, 4, 4, 6, 6, 8, 8]
    # cost: 5/2=2.5, 5/2.5=2.0, 5/2.6, 5/2.7; current 8 (1.85) - the best, stays
    assert c.next_width() == 8
    # width 4 becomes 10% cheaper than 8: below the 20% threshold, no switch
    c.record(4, 1.0, 4.0, 0.5, 0.0, 3.0)  # cost 5/3 = 1.67 vs 5/2.7 = 1.85
    assert c.next_width() == 8
    c.record(4, 1.0, 4.0, 0.5, 0.0, 5.0)  # now clearly better (cost 1.0)
    assert c.next_width() == 4


def test_bad_configuration():
    for args in [([], 0.5, 0.1, 1), ([2], 0.0, 0.1, 1), ([2], 0.5, -1, 1), ([2], 0.5, 0.1, 0)]:
        with pytest.raises(ValueError):
            WidthController(*args)


def test_library_matches_oracle():
    from speculative_decoding_verification_chunked_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from speculative_decoding_verification_chunked_gb300 import svx
    rng = np.random.default_rng(3)
    for trial in range(40):
        ema, thr, n_init = float(rng.uniform(0.05, 1)), float(rng.uniform(0, 0.3)), int(rng.integers(1, 4))
        o = WidthController(WIDTHS, ema, thr, n_init)
        lib = svx.WidthController(WIDTHS, ema, thr, n_init)
        a = float(rng.uniform(0.2, 0.95))
        for _ in range(100):
            q = o.next_width()
            assert lib.next_width() == q
            terms = [x * float(rng.uniform(0.8, 1.25)) for x in round_terms(q, a)]
            terms[4] = float(rng.integers(0, q + 2))  # committed tokens of one round, sometimes 0
            o.record(q, *terms)
            lib.record(q, *terms)
            for w in WIDTHS:
                assert lib.cost(w) == o.cost(w)
    with pytest.raises(svx.SvxError):
        svx.WidthController(WIDTHS, 0.5, 0.1, 1).record(3, 1, 1, 1, 1, 1)
