"""A round whose parts are all device-resident (or zero-copy) enqueues work on the compute stream
only, so it can be captured into a CUDA graph once and replayed: the host cost of the API calls
(validation, planning, launches) is paid at capture time.  Replays reuse the captured round's epoch;
the finish kernel marks the state slots it consumed as unwritten, so one replay never merges
another's state.  The oracle checks every replay."""
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
