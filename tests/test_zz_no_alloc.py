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
