"""svx_verify_static, the round that allocates nothing, against the context round.

Some callers cannot call cudaMalloc while they run (an engine whose memory
manager owns all device memory after start-up, or a decode loop that cannot
afford an allocation's cost or implicit synchronisation).  For them the library
keeps its round state in a static device array; this checks that two calls in a
row through that entry point give the same O and LSE as the ordinary
context-based entry points, within the parity tolerance of the other tests.
Collected last on purpose: a failure here leaves every other test already run.
"""
import numpy as np
import pytest

import workloads as W
from helpers import check_parity, gpu_inputs, oracle_out, run_gpu

pytestmark = pytest.mark.gpu

CASES = [
    W.Workload("static_qwen", 4, 32, 8, 128, (3000, 1, 4096, 777), 1024, 5, seed=41),
    W.Workload("static_tree", 3, 16, 4, 128, (513, 0, 2048), 512, 16, tree=True, seed=42),
]


@pytest.fixture(scope="module")
def svx():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_chunked_gb300 import svx as mod
    return mod


def static_round(svx, w, t, x):
    import torch
    o = torch.empty((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
    svx.verify_static(t["q"], w.hist_len, t["kh"], t["vh"], o, lse, cand_k=t["kc"], cand_v=t["vc"],
                      parent=x.parent, n_kv_heads=w.n_kv_heads)
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def test_static_round_matches_context_round_twice(svx):
    for w in CASES:  # two calls in a row, different shapes: nothing of the first leaks into the second
        x, t = gpu_inputs(w, resident=True)
        o_s, l_s = static_round(svx, w, t, x)
        with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens) as v:
            o_c, l_c = run_gpu(v, w, t, x)
        check_parity(o_s, l_s, o_c, l_c)
        check_parity(o_s, l_s, *oracle_out(w, x))
    # no kernel of the static rounds gave up a bounded wait; the check clears what it reads
    assert svx.static_check() is False
    assert svx.static_check() is False


def run_static_case(svx, w, with_candidates=True):
    """One static call, checked against the oracle."""
    import torch
    x, t = gpu_inputs(w, resident=True)
    o = torch.empty((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
    kc, vc = (t["kc"], t["vc"]) if with_candidates else (None, None)
    svx.verify_static(t["q"], w.hist_len, t["kh"], t["vh"], o, lse, cand_k=kc, cand_v=vc,
                      parent=x.parent if with_candidates else None, n_kv_heads=w.n_kv_heads)
    torch.cuda.synchronize()
    o_s, l_s = o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)
    check_parity(o_s, l_s, *oracle_out(w, x, with_candidates=with_candidates))
    return o_s, l_s


# rows = n_req * n_q_heads * n_query against the scratch limit of 8 * (16 + 4 d) bytes per row after a
# 256-byte header: 7,943 rows at d = 128, 15,420 at d = 64
UNDER_128 = W.Workload("static_under_128", 32, 8, 8, 128, tuple(range(40, 40 + 32 * 7, 7)), 64, 31, seed=44)
OVER_128 = UNDER_128.with_(name="static_over_128", n_req=33, hist_len=(16,) * 33)
UNDER_64 = W.Workload("static_under_64", 62, 8, 2, 64, tuple(range(5, 5 + 62 * 3, 3)), 64, 31, seed=45)
OVER_64 = UNDER_64.with_(name="static_over_64", n_req=63, hist_len=(16,) * 63)


def test_static_round_covers_no_candidates_head_dim_64_and_many_requests(svx):
    # no candidate region: the finish kernel runs without candidate k/v
    run_static_case(svx, W.Workload("static_nocand", 3, 16, 4, 128, (700, 3, 129), 256, 4, seed=46),
                    with_candidates=False)
    # head dimension 64, with a token tree
    run_static_case(svx, W.Workload("static_d64", 3, 8, 2, 64, (1000, 3, 300), 256, 8, tree=True, seed=47))
    # more than 64 requests with history: several chunk launches that share state slot 0
    run_static_case(svx, W.Workload("static_many", 70, 8, 2, 128, tuple(50 + 13 * b for b in range(70)), 256, 4,
                                    seed=48))
    assert svx.static_check() is False


@pytest.mark.parametrize("under,over", [(UNDER_128, OVER_128), (UNDER_64, OVER_64)], ids=["d128", "d64"])
def test_static_round_size_limit_is_exact(svx, under, over):
    import torch
    assert under.n_req * under.n_q_heads * under.n_query <= (svx.STATIC_SCRATCH_BYTES - 256) // (
        8 * (16 + 4 * under.head_dim)) < over.n_req * over.n_q_heads * over.n_query
    run_static_case(svx, under)  # the largest shape of this form that fits runs and is correct
    w = over
    q = torch.zeros((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
    k = torch.zeros((16, w.n_kv_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(svx.SvxError) as e:
        svx.verify_static(q, w.hist_len, [k] * w.n_req, [k] * w.n_req, o, lse, n_kv_heads=w.n_kv_heads)
    assert e.value.status == svx.ERR_INVALID_ARG and "static scratch" in e.value.message
    assert svx.static_check() is False


def test_static_binding_checks_parents_and_head_count(svx):
    import torch
    q = torch.zeros((2, 4, 3, 128), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((2, 4, 3), dtype=torch.float32, device="cuda")
    kc = torch.zeros((2, 3, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(svx.SvxError) as e:  # 3 parents for 2 requests x 3 nodes: refused before the C call
        svx.verify_static(q, [0, 0], [None, None], [None, None], o, lse, cand_k=kc, cand_v=kc, parent=[-1, 0, 1])
    assert e.value.status == svx.ERR_INVALID_ARG
    with pytest.raises(svx.SvxError) as e:  # nothing to infer the KV head count from
        svx.verify_static(q, [0, 0], [None, None], [None, None], o, lse)
    assert e.value.status == svx.ERR_INVALID_ARG and "n_kv_heads" in e.value.message


def test_static_round_rejects_rounds_beyond_its_scratch(svx):
    import torch
    w = W.Workload("too_big", 256, 32, 8, 128, (1,) * 256, 64, 32, seed=43)  # 262144 query rows
    q = torch.zeros((w.n_req, w.n_q_heads, w.n_query, 128), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
    k = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(svx.SvxError) as e:
        svx.verify_static(q, w.hist_len, [k] * 256, [k] * 256, o, lse, n_kv_heads=8)
    assert e.value.status == svx.ERR_INVALID_ARG and "static scratch" in e.value.message
