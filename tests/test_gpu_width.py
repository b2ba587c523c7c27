"""The dynamic verification width driven by measured round costs.

"Resource-Efficient Speculative Decoding for Long-Context LLM Serving", section 4.2,
"I/O-aware dynamic verification widths": verification costs are estimated from the
history's transfer and the chunk computation, and the next round's width is the
one with the least estimated round time per committed token.  Here every round is
a real streamed verification round at the width the controller chose (q drafts,
q + 1 queries), its transfer and attention times come from the library's own
timing (svx_round_stats), the Draft's cost and the accepted drafts come from a
seeded synthetic model, and the library's controller must choose exactly what
the oracle's controller chooses on the same records.
"""
import numpy as np
import pytest

import workloads as W
from helpers import check_parity, oracle_out, pinned_alloc, sample_rows, bf16_tensor
from oracle.width import WidthController as OracleWidth

pytestmark = pytest.mark.gpu

WIDTHS = [2, 4, 6, 8]


@pytest.fixture(scope="module")
def svx():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_chunked_gb300 import svx as mod
    return mod


def test_width_controller_follows_measured_round_costs(svx):
    import torch
    base = W.Workload("width", 4, 32, 8, 128, (16384, 16384, 12000, 16384), 2048, 9, seed=91)
    hist = W.layer_inputs(base, hist_alloc=pinned_alloc)  # one history for every width
    kh = [bf16_tensor(k) for k in hist.k_hist]
    vh = [bf16_tensor(v) for v in hist.v_hist]
    per_width = {}
    for q in WIDTHS:  # q drafts -> q + 1 verification queries and candidates
        wq = base.with_(n_query=q + 1)
        xq = W.layer_inputs(wq, requests=[])
        xq = W.LayerInputs(xq.q, hist.k_hist, hist.v_hist, xq.k_cand, xq.v_cand, xq.parent)
        per_width[q] = (wq, xq, bf16_tensor(xq.q, "cuda"), bf16_tensor(xq.k_cand, "cuda"),
                        bf16_tensor(xq.v_cand, "cuda"))
    rng = np.random.default_rng(92)
    accept, draft_ms_per_token, correct_ms = 0.7, 0.25, 0.1
    lib = svx.WidthController(WIDTHS, ema=0.5, threshold=0.05, n_init=2)
    ora = OracleWidth(WIDTHS, ema=0.5, threshold=0.05, n_init=2)
    chosen = []
    last_out = {}
    with svx.Verifier(base.n_req, base.n_q_heads, base.n_kv_heads, base.head_dim, 9, base.chunk_tokens, n_slots=3,
                      timing=True) as v:
        for r in range(24):
            q = lib.next_width()
            assert ora.next_width() == q
            chosen.append(q)
            wq, xq, qd, kc, vc = per_width[q]
            o = torch.empty((wq.n_req, wq.n_q_heads, q + 1, wq.head_dim), dtype=torch.bfloat16, device="cuda")
            lse = torch.empty((wq.n_req, wq.n_q_heads, q + 1), dtype=torch.float32, device="cuda")
            v.run_round(qd, wq.hist_len, kh, vh, wq.chunk_tokens, o, lse, cand_k=kc, cand_v=vc, timeout_ms=60000)
            st = v.stats()
            # the synthetic Draft: q tokens at a fixed cost, each accepted with probability `accept` until the
            # first rejection; the round commits the accepted prefix plus the Target's own token
            accepted = 0
            while accepted < q and rng.random() < accept:
                accepted += 1
            terms = (q * draft_ms_per_token, st["copy_busy_ms"], st["chunk_kernel_ms"] + st["finish_kernel_ms"],
                     correct_ms, float(accepted + 1))
            assert terms[1] > 0 and terms[2] > 0
            lib.record(q, *terms)
            ora.record(q, *terms)
            for w_ in WIDTHS:
                assert lib.cost(w_) == ora.cost(w_)
            torch.cuda.synchronize()
            last_out[q] = (o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64))
    # initial sampling visited every width twice, in order; afterwards the controller kept a width
    assert chosen[:8] == [2, 2, 4, 4, 6, 6, 8, 8]
    assert set(chosen[8:]) <= set(WIDTHS)
    # every width's last round is correct
    for q, (o, l) in last_out.items():
        wq, xq = per_width[q][:2]
        rows = sample_rows(wq, 24, seed=q)
        check_parity(o, l, *oracle_out(wq, xq, rows=rows), rows=rows)
