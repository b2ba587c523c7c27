"""Stream-ordering cases of the round API, checked against the oracle.

A round whose parts are all device-resident (or zero-copy) enqueues work on the compute stream
only, so it can be captured into a CUDA graph once and replayed: the host cost of the API calls
(validation, planning, launches) is paid at capture time.  Replays reuse the captured round's epoch;
the finish kernel marks the state slots it consumed as unwritten, so one replay never merges
another's state.

The library's kernels are launched so that they may start while the kernel before them in the
stream still runs, and wait before touching global memory; a caller's kernel that writes a round's
inputs right before the library's launch must still be seen."""
import numpy as np
import pytest

from helpers import check_parity, gpu_inputs, oracle_out
from workloads import synth as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def svx():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_chunked_gb300 import svx as mod
    return mod


def _copy_inputs(dst, src):
    dst["q"].copy_(src["q"])
    dst["kc"].copy_(src["kc"])
    dst["vc"].copy_(src["vc"])
    for a, b in zip(dst["kh"] + dst["vh"], src["kh"] + src["vh"]):
        if a is not None:
            a.copy_(b)


@pytest.mark.parametrize("zero_copy", [False, True], ids=["device_history", "zero_copy_history"])
@pytest.mark.parametrize("chunk", [512, 4096], ids=["several_pushes", "one_push"])
def test_round_replays_from_a_cuda_graph(svx, chunk, zero_copy):
    import torch
    w = W.Workload("graph", 3, 16, 4, 128, (700, 1500, 129), chunk, 5, seed=41)
    x0, t0 = gpu_inputs(w, layer=0, resident=not zero_copy)
    x1, t1 = gpu_inputs(w, layer=1, resident=not zero_copy)
    keep = {k: (v.clone() if not isinstance(v, list) else [None if e is None else e.clone() for e in v])
            for k, v in t0.items()}  # (host history is copied to pageable memory: only a source here)
    B, Hq, nq, d = w.n_req, w.n_q_heads, w.n_query, w.head_dim
    o = torch.empty((B, Hq, nq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, nq), dtype=torch.float32, device="cuda")
    cs = torch.cuda.Stream()

    def round_(v):
        v.run_round(t0["q"], w.hist_len, t0["kh"], t0["vh"], w.chunk_tokens, o, lse, cand_k=t0["kc"],
                    cand_v=t0["vc"], parent=x0.parent)

    def out():
        torch.cuda.synchronize()
        return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)

    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=2,
                      compute_stream=cs, zero_copy=zero_copy) as v:
        round_(v)  # eager round first: kernels configured, reference for the replays
        check_parity(*out(), *oracle_out(w, x0))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            round_(v)
        _copy_inputs(t0, t1)  # new inputs in the captured buffers
        g.replay()
        check_parity(*out(), *oracle_out(w, x1))
        _copy_inputs(t0, keep)  # and back: a replay must not see the previous replay's state
        g.replay()
        g.replay()
        check_parity(*out(), *oracle_out(w, x0))


def test_inputs_written_by_kernels_right_before_the_launches(svx):
    import torch
    w = W.Workload("order", 3, 16, 4, 128, (900, 1700, 300), 4096, 5, seed=42)
    x0, t0 = gpu_inputs(w, layer=0, resident=True)
    x1, t1 = gpu_inputs(w, layer=1, resident=True)
    B, Hq, nq, d = w.n_req, w.n_q_heads, w.n_query, w.head_dim
    o = torch.empty((B, Hq, nq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, nq), dtype=torch.float32, device="cuda")
    cs = torch.cuda.Stream()
    q_new, kc_new = t1["q"].clone(), t1["kc"].clone()
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=2,
                      compute_stream=cs) as v:
        # the history of layer 1 in layer 0's buffers, outside the stream order of the round
        for a, b in zip(t0["kh"] + t0["vh"], t1["kh"] + t1["vh"]):
            a.copy_(b)
        t0["vc"].copy_(t1["vc"])
        torch.cuda.synchronize()
        for _ in range(3):  # back-to-back rounds, each with its inputs written by kernels on the stream
            with torch.cuda.stream(cs):
                torch.cuda._sleep(200000)               # keep the stream busy so launches queue up
                torch.add(q_new, 0, out=t0["q"])        # a kernel writing Q right before the push
            v.round_begin(t0["q"], w.hist_len)
            v.candidate_attn(t0["kc"], t0["vc"], x0.parent)
            v.push_chunk([(b, 0, t0["kh"][b], t0["vh"][b]) for b in range(B) if w.hist_len[b]])
            with torch.cuda.stream(cs):
                torch.add(kc_new, 0, out=t0["kc"])      # a kernel writing candidate K right before finish
            v.round_finish(o, lse)
            with torch.cuda.stream(cs):                 # and one overwriting them right after
                t0["q"].zero_()
                t0["kc"].zero_()
        torch.cuda.synchronize()
        check_parity(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                     *oracle_out(w, x1))
