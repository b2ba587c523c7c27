"""Copy/compute overlap through the library's own events, staged-launch CTA budgets, and a round
run beside a co-running Draft load.

"Resource-Efficient Speculative Decoding for Long-Context LLM Serving", section 4.2
("Pipelined KV transfers and prefetching"): chunk i + 1 transfers while chunk i is
computed, and the next layer's chunks are prefetched while the current layer
finishes.  Section 4.3 ("Target-priority scheduling"): the Target's verification
runs beside the Draft, and co-running work shares the SMs, the L2 and HBM.
"""
import threading

import numpy as np
import pytest

import workloads as W
from helpers import check_parity, gpu_inputs, oracle_out, run_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def svx():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_chunked_gb300 import svx as mod
    return mod


def _multi_layer(w, n_layers):
    """n_layers layers of streamed inputs (pinned host history) and their outputs."""
    import torch
    layers = []
    for layer in range(n_layers):
        x, t = gpu_inputs(w, layer=layer)
        o = torch.empty((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
        layers.append((x, t, o, lse))
    return layers


def test_window_covers_a_multi_layer_step(svx):
    """Three layer rounds enqueued back to back form one timing window: its counts equal the plan's,
    the copy intervals are disjoint and in issue order, each chunk kernel starts after its own copies,
    and the exposed kernel time is a part of the kernel time.  Each layer is checked against the
    oracle, and a reset opens a window with the next rounds only."""
    import torch
    w = W.Workload("win", 3, 16, 4, 128, (3000, 1100, 2600), 512, 5, seed=71)
    layers = _multi_layer(w, 3)
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=3,
                      timing=True) as v:
        for x, t, o, lse in layers:
            v.run_round(t["q"], w.hist_len, t["kh"], t["vh"], w.chunk_tokens, o, lse, cand_k=t["kc"],
                        cand_v=t["vc"])
        ws = v.window_stats()
        iv = v.window_intervals()
        last = v.stats()
        n_chunks = max(-(-C // w.chunk_tokens) for C in w.hist_len)
        assert ws["n_rounds"] == 3 and ws["n_pushes"] == 3 * n_chunks == iv.shape[0]
        assert ws["h2d_bytes"] == 3 * w.hist_bytes and ws["device_bytes"] == 0
        assert np.all(np.isfinite(iv)) and np.all(iv[:, 1] > iv[:, 0])
        assert np.all(iv[1:, 0] >= iv[:-1, 1] - 1e-3)  # one copy stream: disjoint, in issue order
        assert np.all(iv[:, 2] >= iv[:, 1] - 1e-3) and np.all(iv[:, 3] > iv[:, 2])
        assert abs(ws["copy_busy_ms"] - float(np.sum(iv[:, 1] - iv[:, 0]))) < 1e-3
        assert abs(ws["chunk_kernel_ms"] - float(np.sum(iv[:, 3] - iv[:, 2]))) < 1e-3
        assert 0.0 <= ws["chunk_kernel_exposed_ms"] <= ws["chunk_kernel_ms"] + 1e-6
        assert ws["window_ms"] >= ws["copy_busy_ms"] + ws["copy_gap_ms"] - 1e-3
        assert ws["window_ms"] >= iv[-1, 3] - min(0.0, iv[0, 0]) - 1e-3
        # the last round's statistics are the window's last n_chunks pushes
        assert abs(last["copy_busy_ms"] - float(np.sum(iv[-n_chunks:, 1] - iv[-n_chunks:, 0]))) < 1e-3
        torch.cuda.synchronize()
        for x, t, o, lse in layers:
            check_parity(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                         *oracle_out(w, x))
        v.window_reset()
        x, t, o, lse = layers[0]
        v.run_round(t["q"], w.hist_len, t["kh"], t["vh"], w.chunk_tokens, o, lse, cand_k=t["kc"], cand_v=t["vc"],
                    timeout_ms=60000)
        ws2 = v.window_stats()
        assert ws2["n_rounds"] == 1 and ws2["n_pushes"] == n_chunks and ws2["h2d_bytes"] == w.hist_bytes


def test_window_calls_outside_their_state_are_refused(svx):
    import torch
    w = W.Workload("win_err", 1, 4, 1, 64, (100,), 64, 2, seed=72)
    x, t = gpu_inputs(w)
    with svx.Verifier(1, 4, 1, 64, 2, 128) as v:  # no timing flag
        with pytest.raises(svx.SvxError) as e:
            v.window_stats()
        assert e.value.status == svx.ERR_BAD_STATE
    with svx.Verifier(1, 4, 1, 64, 2, 128, timing=True) as v:
        with pytest.raises(svx.SvxError) as e:  # nothing finished yet
            v.window_stats()
        assert e.value.status == svx.ERR_BAD_STATE
        v.round_begin(t["q"], w.hist_len)
        with pytest.raises(svx.SvxError) as e:  # inside a round
            v.window_reset()
        assert e.value.status == svx.ERR_BAD_STATE
        o = torch.empty((1, 4, 2, 64), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((1, 4, 2), dtype=torch.float32, device="cuda")
        v.push_chunk([(0, 0, t["kh"][0], t["vh"][0])])
        v.round_finish(o, lse, timeout_ms=60000)
        assert v.window_stats()["n_rounds"] == 1


@pytest.mark.parametrize("staged_ctas", [1, 8, 16])
def test_staged_launch_cta_budget(svx, staged_ctas):
    """Chunk launches over staged parts on a few SMs give the same result (the work plan changes, the
    arithmetic does not), including a 64-row two-warpgroup pass and ragged parts."""
    w = W.Workload("staged", 4, 32, 8, 128, (5000, 1, 2049, 777), 1024, 8, seed=73)
    x, t = gpu_inputs(w)
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=3,
                      staged_ctas=staged_ctas) as v:
        o, l = run_gpu(v, w, t, x)
    check_parity(o, l, *oracle_out(w, x))


class _GemmLoad:
    """A stand-in Draft: bf16 4096^3 GEMMs on a lowest-priority stream from a host thread."""

    def __init__(self, n=4096):
        import torch
        lo, _hi = torch.cuda.Stream.priority_range()
        self.torch = torch
        self.stream = torch.cuda.Stream(priority=lo)
        self.a = torch.randn((n, n), device="cuda", dtype=torch.bfloat16)
        self.b = torch.randn((n, n), device="cuda", dtype=torch.bfloat16)
        self.c = torch.empty((n, n), device="cuda", dtype=torch.bfloat16)
        self.stop = False
        self.count = 0
        self.device = torch.cuda.current_device()

    def _run(self):
        torch = self.torch
        torch.cuda.set_device(self.device)  # a new host thread has no current device of its own
        ev = torch.cuda.Event()
        while not self.stop:
            with torch.cuda.stream(self.stream):
                for _ in range(4):
                    torch.matmul(self.a, self.b, out=self.c)
                ev.record(self.stream)
            ev.synchronize()
            self.count += 4

    def __enter__(self):
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()
        return self

    def __exit__(self, *exc):
        self.stop = True
        self.thread.join()
        self.torch.cuda.synchronize()


@pytest.mark.parametrize("mode", ["copy_engine", "copy_engine_16_ctas", "zero_copy_8_ctas"])
def test_round_beside_a_draft_gemm_load(svx, mode):
    """Streamed rounds while a low-priority bf16 GEMM loop runs on the same GPU: the outputs are
    bit-identical to the same rounds run alone (the work plan does not depend on timing) and match
    the oracle on sampled rows."""
    import torch
    w = W.Workload("coexec", 4, 32, 8, 128, (24000, 9000, 16385, 3), 2048, 5, seed=74)
    x, t = gpu_inputs(w)
    kw = {"copy_engine": {}, "copy_engine_16_ctas": {"staged_ctas": 16},
          "zero_copy_8_ctas": {"zero_copy": True, "zero_copy_ctas": 8}}[mode]
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=3,
                      **kw) as v:
        o_alone, l_alone = run_gpu(v, w, t, x)
        with _GemmLoad() as load:
            outs = [run_gpu(v, w, t, x) for _ in range(3)]
        assert load.count > 0
    for o, l in outs:
        assert np.array_equal(o, o_alone) and np.array_equal(l, l_alone)
    rows = sample_rows(w, 48, seed=7)
    check_parity(outs[-1][0], outs[-1][1], *oracle_out(w, x, rows=rows), rows=rows)
    del torch


# ---------------------------------------------------------------- host-side failures and the adaptive path


def _pushes(svx, w, t, row_bytes):
    """The plan's cohort chunks as raw part lists (request, start, n, k address, v address)."""
    chunks = {}
    for j, _s, b, t0, n in svx.plan_chunks(w.hist_len, w.chunk_tokens, 3):
        chunks.setdefault(j, []).append((b, t0, n))
    return [[(b, t0, n, t["kh"][b].data_ptr() + t0 * row_bytes, t["vh"][b].data_ptr() + t0 * row_bytes)
             for b, t0, n in chunks[j]] for j in sorted(chunks)]


@pytest.mark.parametrize("nth", [1, 2, 5])
def test_a_refused_copy_leaves_the_round_open_and_the_context_usable(svx, nth):
    """A copy submission refused on the host (the test hook stands in for a failing cudaMemcpyAsync)
    fails its push with SVX_ERR_CUDA; pushing the same chunk again completes the round, which matches
    the oracle, and the next round runs normally."""
    import torch
    w = W.Workload("refuse", 3, 16, 4, 128, (1500, 700, 1100), 256, 5, seed=75)
    x, t = gpu_inputs(w)
    row_bytes = w.n_kv_heads * w.head_dim * 2
    o = torch.empty((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=3,
                      timing=True) as v:
        v.round_begin(t["q"], w.hist_len)
        v.candidate_attn(t["kc"], t["vc"])
        v.debug_fail_copy(nth)
        refused = 0
        for p in _pushes(svx, w, t, row_bytes):
            try:
                v.push_raw(p)
            except svx.SvxError as e:
                assert e.status == svx.ERR_CUDA and "not processed" in e.message
                refused += 1
                v.push_raw(p)  # the same chunk again
        assert refused == 1
        v.round_finish(o, lse, timeout_ms=60000)
        torch.cuda.synchronize()
        st = v.stats()
        assert st["h2d_bytes"] == w.hist_bytes  # the refused push's partial copies are not counted
        check_parity(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                     *oracle_out(w, x))
        o2, l2 = run_gpu(v, w, t, x)
    check_parity(o2, l2, *oracle_out(w, x))


def test_a_delayed_copy_shows_as_a_copy_gap_and_exposed_compute(svx):
    """The host sleeps before one push's copies, so the copy stream runs dry: the window shows the gap,
    the previous push's chunk kernel runs inside it with no transfer to hide it, and the round is still
    correct."""
    import torch
    w = W.Workload("delay", 2, 32, 8, 128, (6000, 6000), 1024, 5, seed=76)
    x, t = gpu_inputs(w)
    row_bytes = w.n_kv_heads * w.head_dim * 2
    pushes = _pushes(svx, w, t, row_bytes)
    k = 3  # the delayed push
    o = torch.empty((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=3,
                      timing=True) as v:
        v.window_reset()
        v.round_begin(t["q"], w.hist_len)
        v.candidate_attn(t["kc"], t["vc"])
        for i, p in enumerate(pushes):
            if i == k:
                v.debug_delay_copy(1, 80)  # the next copy submission, the first of push k
            v.push_raw(p)
        v.round_finish(o, lse, timeout_ms=60000)
        ws = v.window_stats()
        iv = v.window_intervals()
    # push k's copy interval starts when its first copy is submitted, after the pause
    gap = iv[k, 0] - iv[k - 1, 1]
    assert gap >= 70.0 and ws["copy_gap_ms"] >= 70.0
    # the previous push's chunk kernel ran in the gap, outside every copy interval
    kern = iv[k - 1, 3] - iv[k - 1, 2]
    assert iv[k - 1, 2] >= iv[k - 1, 1] - 1e-3 and iv[k - 1, 3] <= iv[k, 0] + 1e-3
    assert ws["chunk_kernel_exposed_ms"] >= 0.9 * kern
    torch.cuda.synchronize()
    check_parity(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                 *oracle_out(w, x))


def test_adaptive_streaming_moves_to_in_place_reads_when_copies_are_slow(svx):
    """The adaptive context measures both engines on whole rounds: round 0 is staged, round 1 read in
    place.  A host-side pause inside one of round 0's copies (which the copy-time events see as a very
    slow copy) makes the copy engine's figure slow, so round 2 and later read in place too.  Every round
    matches the oracle."""
    import torch
    w = W.Workload("adaptive", 2, 16, 4, 128, (4096, 3000), 1024, 5, seed=77)
    x, t = gpu_inputs(w)
    row_bytes = w.n_kv_heads * w.head_dim * 2
    pushes = _pushes(svx, w, t, row_bytes)
    assert len(pushes) == 4
    o = torch.empty((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
    ref = oracle_out(w, x)
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=3,
                      timing=True, adaptive=True, zero_copy_ctas=16) as v:
        stats = []
        for rnd in range(3):
            v.round_begin(t["q"], w.hist_len)
            v.candidate_attn(t["kc"], t["vc"])
            for i, p in enumerate(pushes):
                if rnd == 0 and i == 2:
                    # a pause between push 2's first and second copy submissions: its copy interval
                    # (first submission to last copy done) reads as a very slow copy
                    v.debug_delay_copy(2, 100)
                v.push_raw(p)
            v.round_finish(o, lse, timeout_ms=60000)
            stats.append(v.stats())
            torch.cuda.synchronize()
            check_parity(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), *ref)
    assert stats[0]["n_zero_copy_pushes"] == 0  # staged: the copy engine's first measurement
    assert stats[0]["n_chunk_launches"] == 4
    # read in place: the other engine's first measurement.  The round's four pushes launch together when it
    # finishes, each request's chunks merged into one part (they are consecutive rows of one buffer)
    assert stats[1]["n_zero_copy_pushes"] == 1 and stats[1]["n_chunk_launches"] == 1
    assert stats[2]["n_zero_copy_pushes"] == 1  # the copy engine was measured slow
    # bytes read in place count as host bytes, and the in-place kernels count as transfer time
    assert stats[1]["h2d_bytes"] == w.hist_bytes and stats[1]["copy_busy_ms"] == 0.0
    assert stats[1]["transfer_busy_ms"] > 0.0


def test_a_window_past_its_round_limit_starts_again(svx):
    """A timing window holds at most 4096 rounds: the round after the limit opens a new window, whose
    figures cover only its own rounds; the round statistics stay available and each round is correct."""
    import torch
    w = W.Workload("wrap", 1, 4, 1, 64, (300,), 300, 2, seed=78)
    x, t = gpu_inputs(w, resident=True)
    o = torch.empty((1, 4, 2, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 4, 2), dtype=torch.float32, device="cuda")
    parts = [(0, 0, 300, t["kh"][0].data_ptr(), t["vh"][0].data_ptr())]
    with svx.Verifier(1, 4, 1, 64, 2, 300, timing=True) as v:
        v.window_reset()
        for r in range(4096 + 5):
            v.round_begin(t["q"], w.hist_len)
            v.candidate_attn(t["kc"], t["vc"])
            v.push_raw(parts)
            v.round_finish(o, lse, timeout_ms=60000 if r == 4096 + 4 else 0)
            if r == 4095:
                ws = v.window_stats()
                assert ws["n_rounds"] == 4096 and ws["n_pushes"] == 4096
        ws = v.window_stats()
        assert ws["n_rounds"] == 5 and ws["n_pushes"] == 5 and ws["device_bytes"] == 5 * w.hist_bytes
        assert v.window_intervals().shape == (5, 4) and v.window_rounds().shape == (5, 3)
        st = v.stats()
        assert st["chunk_kernel_ms"] > 0 and st["n_chunk_launches"] == 1
    torch.cuda.synchronize()
    check_parity(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), *oracle_out(w, x))


@pytest.mark.parametrize("order", ["reversed", "split_buffers"])
def test_an_adaptive_in_place_round_merges_only_what_continues(svx, order):
    """An adaptive round read in place launches its parts when it finishes.  A chunk merges into its
    request's part only when it continues it (next tokens, next rows of the same buffer); otherwise it goes
    to a later launch of the round, so no launch holds two parts of one request.  Pushed in reverse order,
    or from a separate buffer per chunk, the round needs several launches and still matches the oracle."""
    import torch
    w = W.Workload("defer", 2, 16, 4, 128, (4096, 3000), 1024, 5, seed=79)
    x, t = gpu_inputs(w)
    row_bytes = w.n_kv_heads * w.head_dim * 2
    pushes = _pushes(svx, w, t, row_bytes)
    keep = []
    if order == "reversed":
        pushes = pushes[::-1]
    else:  # every chunk copied into its own pinned buffer, one spare row after it, so that no chunk's rows
        # can end where the next chunk's buffer starts
        new = []
        for ps in pushes:
            row = []
            for b, t0, n, _k, _v in ps:
                kb = torch.empty((n + 1,) + tuple(t["kh"][b].shape[1:]), dtype=torch.bfloat16).pin_memory()
                vb = torch.empty((n + 1,) + tuple(t["vh"][b].shape[1:]), dtype=torch.bfloat16).pin_memory()
                kb[:n].copy_(t["kh"][b][t0:t0 + n])
                vb[:n].copy_(t["vh"][b][t0:t0 + n])
                keep += [kb, vb]
                row.append((b, t0, n, kb.data_ptr(), vb.data_ptr()))
            new.append(row)
        pushes = new
    o = torch.empty((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
    ref = oracle_out(w, x)
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=3,
                      timing=True, adaptive=True, zero_copy_ctas=16) as v:
        for rnd in range(2):  # round 0 staged, round 1 read in place
            v.round_begin(t["q"], w.hist_len)
            v.candidate_attn(t["kc"], t["vc"])
            for p in pushes:
                v.push_raw(p)
            v.round_finish(o, lse, timeout_ms=60000)
            st = v.stats()
            torch.cuda.synchronize()
            check_parity(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), *ref)
        assert st["n_zero_copy_pushes"] == 1 and st["copy_busy_ms"] == 0.0
        # request 0 has 4 chunks, request 1 has 3: none merges, so one launch per chunk rank
        assert st["n_chunk_launches"] == 4, st["n_chunk_launches"]
        assert st["h2d_bytes"] == w.hist_bytes


@pytest.mark.parametrize("order", ["forward", "reversed"])
def test_a_zero_copy_round_launches_once_when_its_chunks_continue(svx, order):
    """SVX_FLAG_ZERO_COPY: a round's pushes launch together when it finishes.  Chunks pushed in plan
    order continue one another (consecutive rows of each request's buffer) and merge into one part per
    request, one launch; pushed in reverse they cannot merge and need one launch per chunk rank.  Both
    match the oracle."""
    import torch
    w = W.Workload("zcmerge", 3, 16, 4, 128, (4096, 3000, 130), 1024, 5, seed=80)
    x, t = gpu_inputs(w)
    row_bytes = w.n_kv_heads * w.head_dim * 2
    pushes = _pushes(svx, w, t, row_bytes)
    if order == "reversed":
        pushes = pushes[::-1]
    o = torch.empty((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
    with svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens, n_slots=3,
                      timing=True, zero_copy=True, zero_copy_ctas=32) as v:
        v.round_begin(t["q"], w.hist_len)
        v.candidate_attn(t["kc"], t["vc"])
        for p in pushes:
            v.push_raw(p)
        v.round_finish(o, lse, timeout_ms=60000)
        st = v.stats()
    torch.cuda.synchronize()
    check_parity(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                 *oracle_out(w, x))
    assert st["n_copies"] == 0 and st["h2d_bytes"] == w.hist_bytes and st["n_zero_copy_pushes"] == 1
    assert st["n_chunk_launches"] == (1 if order == "forward" else len(pushes))
