"""Every query row of one full-size layer against the oracle (no sampling).

The qwen3-shaped layer (8 requests, 32 query / 8 KV heads, d = 128, 32768 history
tokens each, 5 verification queries, causal candidate chain) streamed from pinned
host memory in the benchmark's chunks of 2048 tokens: all 1,280 rows of O and LSE
are compared with the float64 oracle, which runs one (request, KV head) pair per
process.
"""
import numpy as np
import pytest

import workloads as W
from helpers import check_parity, gpu_inputs, oracle_all_rows_parallel, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def svx():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_chunked_gb300 import svx as mod
    return mod


def test_every_row_of_a_full_qwen3_layer(svx):
    w = W.named("qwen3")
    x, t = gpu_inputs(w)
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=3) as v:
        o, l = run_gpu(v, w, t, x)
    o_ref, l_ref = oracle_all_rows_parallel(w, x)
    assert not np.isnan(o_ref).any() and not np.isnan(l_ref).any()
    check_parity(o, l, o_ref, l_ref)
