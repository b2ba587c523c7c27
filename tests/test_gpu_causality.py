"""The candidate-region mask as the GPU applies it, pinned bit-exactly.

The finish kernel derives each query's visible candidates on the device (a causal
chain: candidates 0..j; a token tree: j and its ancestors), independently of the
host's mask words.  A candidate that query j must not see may not change O_j or
LSE_j in any bit ("Resource-Efficient Speculative Decoding for Long-Context LLM
Serving", section 4.2: a candidate is masked by absolute position, so later
candidates are invisible; token trees restrict it to the ancestors).  Each test
perturbs the K and V of chosen candidates and checks, row by row, that exactly the
rows the oracle's visibility table marks as seeing a perturbed candidate change,
and that every other row is bit-identical.  This checks the device-side mask bit
for bit against the oracle's, without reading it out.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from helpers import check_parity, gpu_inputs, oracle_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def svx():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_chunked_gb300 import svx as mod
    return mod


CASES = [
    W.Workload("chain5", 3, 8, 2, 128, (300, 0, 77), 128, 5, seed=61),
    W.Workload("tree16", 3, 16, 4, 128, (200, 513, 1), 256, 16, tree=True, seed=62),
    W.Workload("tree32_deep", 2, 8, 8, 64, (40, 0), 64, 32, tree=True, tree_max_depth=31, seed=63),
    W.Workload("chain32_d64", 2, 4, 1, 64, (129, 5), 64, 32, seed=64),
]


def _round(svx, w, t, x, kc, vc, tc=True):
    import torch
    o = torch.empty((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens,
                      tensor_cores=tc) as v:
        v.run_round(t["q"], w.hist_len, t["kh"], t["vh"], w.chunk_tokens, o, lse, cand_k=kc, cand_v=vc,
                    parent=x.parent, timeout_ms=60000)
    torch.cuda.synchronize()
    # bit patterns: equality of the raw bits, not of the values
    return (o.view(torch.int16).cpu().numpy().copy(), lse.view(torch.int32).cpu().numpy().copy(),
            o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64))


def _perturbations(w, seed):
    """Sets of (request, candidate) pairs to perturb: every single candidate of request 0, and a few
    random subsets over all requests."""
    rng = np.random.default_rng(seed)
    sets = [[(0, i)] for i in range(w.n_query)]
    for _ in range(3):
        k = int(rng.integers(1, max(2, w.n_query // 2)))
        sets.append([(int(rng.integers(0, w.n_req)), int(i)) for i in rng.choice(w.n_query, size=k, replace=False)])
    return sets


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_invisible_candidates_leave_rows_bit_identical(svx, w):
    import torch
    x, t = gpu_inputs(w, resident=True)
    ob, lb, o0, l0 = _round(svx, w, t, x, t["kc"], t["vc"])
    check_parity(o0, l0, *oracle_out(w, x))
    vis = O.visibility_table(w.n_req, w.n_query, x.parent)  # the oracle's words, not the library's
    gen = torch.Generator(device="cuda").manual_seed(1000 + w.seed)
    for pert in _perturbations(w, w.seed):
        kc, vc = t["kc"].clone(), t["vc"].clone()
        for b, i in pert:
            kc[b, i] = (torch.randn(kc[b, i].shape, generator=gen, device="cuda") * 3).to(kc.dtype)
            vc[b, i] = (torch.randn(vc[b, i].shape, generator=gen, device="cuda") * 3).to(vc.dtype)
        ob2, lb2, _, _ = _round(svx, w, t, x, kc, vc)
        for b in range(w.n_req):
            for j in range(w.n_query):
                sees = any(pb == b and (int(vis[b][j]) >> i) & 1 for pb, i in pert)
                same_o = np.array_equal(ob[b, :, j], ob2[b, :, j])
                same_l = np.array_equal(lb[b, :, j], lb2[b, :, j])
                if sees:
                    assert not (same_o and same_l), f"{w.name}: row (b={b}, j={j}) sees {pert} but did not change"
                else:
                    assert same_o and same_l, f"{w.name}: row (b={b}, j={j}) cannot see {pert} but changed"


def test_fma_and_tensor_core_paths_share_the_mask(svx):
    """The same check with the FP32-FMA chunk kernel: the mask lives in the finish kernel, which both
    chunk kernels feed, and history must never be masked."""
    w = CASES[1]
    x, t = gpu_inputs(w, resident=True)
    ob, lb, o0, l0 = _round(svx, w, t, x, t["kc"], t["vc"], tc=False)
    check_parity(o0, l0, *oracle_out(w, x))
    vis = O.visibility_table(w.n_req, w.n_query, x.parent)
    kc, vc = t["kc"].clone(), t["vc"].clone()
    i = w.n_query - 1  # the last node: only itself sees it (no node has a higher index)
    kc[1, i] = -kc[1, i]
    vc[1, i] = vc[1, i] * 2
    ob2, lb2, _, _ = _round(svx, w, t, x, kc, vc, tc=False)
    for b in range(w.n_req):
        for j in range(w.n_query):
            sees = b == 1 and (int(vis[b][j]) >> i) & 1
            same = np.array_equal(ob[b, :, j], ob2[b, :, j]) and np.array_equal(lb[b, :, j], lb2[b, :, j])
            assert same != bool(sees), (b, j)
