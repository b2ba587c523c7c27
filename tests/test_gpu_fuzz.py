"""Seeded random configurations against the oracle: batch size, head grouping, query count (up to
32, several row passes), head dimension, ragged and empty histories, chunk size, causal chain or
token tree, and history resident in HBM, streamed through the copy engine (as separate and as
batched host tensors) or read in place (zero-copy).  Every draw is fixed by its index."""
import numpy as np
import pytest

from helpers import check_parity, gpu_inputs, oracle_out, run_gpu, sample_rows
from workloads import synth as W

pytestmark = pytest.mark.gpu

N_CASES = 24


@pytest.fixture(scope="module")
def svx():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_chunked_gb300 import svx as mod
    return mod


def draw_case(i):
    rng = np.random.default_rng([7, i])
    B = int(rng.integers(1, 7))
    hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8]))
    nq = int(rng.integers(1, 33))
    while G * nq * hkv > 1024:  # keep the oracle quick
        nq = max(1, nq // 2)
    d = int(rng.choice([64, 128], p=[0.25, 0.75]))
    lens = tuple(int(x) if rng.random() > 0.15 else 0 for x in rng.integers(1, 2500, size=B))
    if max(lens) == 0:
        lens = (1,) + lens[1:]
    chunk = int(rng.choice([64, 128, 256, 1000]))
    tree = bool(rng.random() < 0.35)
    mode = str(rng.choice(["resident", "streamed", "batched", "zero_copy"]))
    w = W.Workload(f"fuzz{i}", B, hkv * G, hkv, d, lens, chunk, nq, tree=tree, tree_max_depth=int(rng.integers(1, 8)),
                   seed=1000 + i)
    return w, mode


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_configuration(svx, i):
    import torch
    w, mode = draw_case(i)
    x, t = gpu_inputs(w, resident=(mode == "resident"))
    if mode == "batched":  # all requests' history as rows of one pinned tensor (2D chunk copies)
        cmax = max(w.hist_len)
        kb = torch.zeros((w.n_req, cmax, w.n_kv_heads, w.head_dim), dtype=torch.bfloat16).pin_memory()
        vb = torch.zeros_like(kb).pin_memory()
        for b, C in enumerate(w.hist_len):
            if C:
                kb[b, :C].copy_(t["kh"][b])
                vb[b, :C].copy_(t["vh"][b])
        t["kh"] = [kb[b, :C] if C else None for b, C in enumerate(w.hist_len)]
        t["vh"] = [vb[b, :C] if C else None for b, C in enumerate(w.hist_len)]
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=2,
                      zero_copy=(mode == "zero_copy"), zero_copy_ctas=8 if i % 2 else 0) as v:
        o, l = run_gpu(v, w, t, x)
    check_parity(o, l, *oracle_out(w, x))


N_LARGE = 8


def draw_large_case(i):
    """Long ragged histories (up to 60k tokens per request, up to 8 requests): many tiles per CTA
    group, parts spread over several CTAs (and grids shrunk to the state-slot limit), several pushes."""
    rng = np.random.default_rng([8, i])
    B = int(rng.integers(1, 9))
    hkv = int(rng.choice([2, 4, 8]))
    G = int(rng.choice([1, 4, 8]))
    nq = int(rng.integers(1, 17))
    lens = tuple(int(x) for x in rng.integers(1, 60000, size=B))
    chunk = int(rng.choice([2048, 8192, 65536]))
    tree = bool(rng.random() < 0.4)
    mode = ("resident", "streamed", "batched", "zero_copy")[i % 4]
    w = W.Workload(f"large{i}", B, hkv * G, hkv, 128, lens, chunk, nq, tree=tree, seed=2000 + i)
    return w, mode


@pytest.mark.parametrize("i", range(N_LARGE))
def test_random_large_configuration_sampled(svx, i):
    import torch
    w, mode = draw_large_case(i)
    x, t = gpu_inputs(w, resident=(mode == "resident"))
    if mode == "batched":
        cmax = max(w.hist_len)
        kb = torch.zeros((w.n_req, cmax, w.n_kv_heads, w.head_dim), dtype=torch.bfloat16).pin_memory()
        vb = torch.zeros_like(kb).pin_memory()
        for b, C in enumerate(w.hist_len):
            kb[b, :C].copy_(t["kh"][b])
            vb[b, :C].copy_(t["vh"][b])
        t["kh"] = [kb[b, :C] for b, C in enumerate(w.hist_len)]
        t["vh"] = [vb[b, :C] for b, C in enumerate(w.hist_len)]
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=3,
                      zero_copy=(mode == "zero_copy"), zero_copy_ctas=8 if i % 2 else 0) as v:
        o, l = run_gpu(v, w, t, x)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    rows = sample_rows(w, 32)
    check_parity(o, l, *oracle_out(w, x, rows=rows), rows=rows)
