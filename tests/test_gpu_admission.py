"""Target-priority admission driving real Draft steps beside verification rounds.

"Resource-Efficient Speculative Decoding for Long-Context LLM Serving", section 4.3,
"Target-priority scheduling" and the two paragraphs after it: a Draft step starts
only when the scheduler admits it (estimated Target slow-down within budget, the
step fits the round's remaining window), the Draft checks the instruction's latest
start time right before starting, and an ACK closes the step.  Here the Draft step
is one bf16 GEMM on a low-priority stream, admitted through the library's
scheduler (svx_sched_*), while the Target streams verification rounds; the
measured round times are fed back to the scheduler.
"""
import os
import sys
import types

import numpy as np
import pytest

import workloads as W
from helpers import check_parity, gpu_inputs, oracle_out, sample_rows

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def svx():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_chunked_gb300 import svx as mod
    return mod


@pytest.mark.parametrize("mode", ["zero_copy_8_ctas", "adaptive_copy_engine"])
def test_admitted_draft_steps_keep_their_deadlines_and_rounds_stay_correct(svx, mode):
    import torch

    import bench
    w = W.Workload("admission", 4, 32, 8, 128, (24000, 9000, 16385, 3), 2048, 5, seed=81)
    x, t = gpu_inputs(w)
    cs = torch.cuda.Stream(priority=-1)
    kw = {"zero_copy_8_ctas": {"zero_copy": True, "zero_copy_ctas": 8},
          "adaptive_copy_engine": {"adaptive": True, "zero_copy_ctas": 32}}[mode]
    outs = []
    o = torch.empty((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=3,
                      compute_stream=cs, **kw) as v:
        def step():
            v.run_round(t["q"], w.hist_len, t["kh"], t["vh"], w.chunk_tokens, o, lse, cand_k=t["kc"],
                        cand_v=t["vc"], parent=x.parent)
            cs.synchronize()
            outs.append((o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)))

        for _ in range(3):
            step()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cs)
        for _ in range(4):
            step()
        e1.record(cs)
        e1.synchronize()
        ms_alone = e0.elapsed_time(e1) / 4
        o_alone, l_alone = outs[-1]
        outs.clear()
        draft = bench.AdmittedDraft(torch.device("cuda", torch.cuda.current_device()), w.n_req, eps_target=0.05,
                                    delta_ms=0.1)
        R = types.SimpleNamespace(torch=torch, cs=cs)
        # the adaptive context explores its other engine on whole rounds (round 10 here), which reads as an
        # over-budget round and pauses admission for a few rounds: it gets more rounds
        n_co = 12 if mode != "adaptive_copy_engine" else 24
        _ms, rec = bench.run_admitted(R, step, n_co, ms_alone, draft)
        # a checked round: no kernel of the context gave up a bounded wait in any round above
        v.run_round(t["q"], w.hist_len, t["kh"], t["vh"], w.chunk_tokens, o, lse, cand_k=t["kc"], cand_v=t["vc"],
                    parent=x.parent, timeout_ms=60000)
    # the protocol: Draft steps ran, each started no later than its instruction's latest start time
    if mode != "adaptive_copy_engine":
        assert rec["draft_steps"] > 0, (rec, ms_alone)
    else:  # Draft steps ran, or the scheduler paused them after an over-budget round (an engine switch)
        assert rec["draft_steps"] > 0 or rec["paused_rounds"] > 0, (rec, ms_alone)
    assert rec["instructions"] >= rec["draft_steps"]
    assert rec["started_after_t_latest"] == 0
    assert all(t_launch <= t_latest for t_launch, t_latest in draft.log)
    # the scheduler saw every round's measured time
    t_d, d_t, _paused = draft.sched.estimates()
    assert t_d > 0.0 and np.isfinite(d_t)
    # verification is unchanged by the co-running Draft.  A fixed engine's rounds are bit-identical to the
    # rounds run alone (the work plan does not depend on timing); the adaptive context may change engines
    # between rounds, and with them the launch's CTA budget and reduction order, so its rounds are held to
    # the parity bar instead.  The oracle checks every round.
    assert len(outs) == n_co
    rows = sample_rows(w, 48, seed=8)
    ref = oracle_out(w, x, rows=rows)
    for o_r, l_r in outs:
        if mode != "adaptive_copy_engine":
            assert np.array_equal(o_r, o_alone) and np.array_equal(l_r, l_alone)
        check_parity(o_r, l_r, *ref, rows=rows)


def test_an_over_budget_round_pauses_admission(svx):
    """A round observed over the budget pauses new Draft instructions until a round's estimate is back
    within it (the scheduler's pause, driven by measured round times)."""
    import torch

    import bench
    draft = bench.AdmittedDraft(torch.device("cuda", torch.cuda.current_device()), 2, eps_target=0.05, ema=1.0)
    draft.begin_round(0, 50.0)
    assert draft.sched.try_admit(0, 0, draft.now_ms(), 40.0) is not None
    draft.end_round(100.0, 50.0)  # the Target took twice as long beside the Draft
    draft.begin_round(1, 50.0)
    assert draft.sched.estimates()[2] and draft.paused_rounds == 1
    assert draft.sched.try_admit(1, 1, draft.now_ms(), 40.0) is None
    draft.end_round(50.0, 50.0)  # alone again: the estimate is back within budget
    draft.begin_round(2, 50.0)
    assert not draft.sched.estimates()[2]
    assert draft.sched.try_admit(1, 2, draft.now_ms(), 40.0) is not None
