"""GPU parity: the CUDA path through the C ABI against the float64 oracle on the
same seeded inputs.  Bar (tests/helpers.py): O max abs <= 1e-2, mean abs <= 1e-3;
LSE relative <= 1e-4.

Small cases span several 32-token tiles, ragged tails, empty histories, several
query-row blocks and both masks; full-size cases use the named workloads'
shapes in the launch configuration the benchmark times and check sampled rows.
"""
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


def make_verifier(svx, w, n_slots=2, chunk=None, **kw):
    return svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, chunk or w.chunk_tokens,
                        n_slots=n_slots, **kw)


SMALL = [
    W.named("tiny"),
    W.Workload("ragged", 5, 8, 2, 128, (0, 1, 33, 700, 1031), 256, 7, seed=11),
    W.Workload("k0", 3, 8, 2, 128, (300, 64, 97), 64, 1, seed=12),
    W.Workload("tree64", 3, 16, 4, 128, (200, 513, 1), 128, 16, tree=True, seed=13),
    W.Workload("g8", 2, 16, 2, 128, (450, 333), 100, 4, seed=14),
    W.Workload("g1", 2, 4, 4, 64, (129, 70), 32, 3, seed=15),
    W.Workload("q32", 2, 8, 4, 128, (90, 257), 64, 32, seed=16),
    W.Workload("tree32", 2, 8, 8, 64, (40, 77), 16, 32, tree=True, tree_max_depth=40, seed=17),
    W.Workload("kscale", 4, 32, 8, 128, (777, 2048, 5, 4000), 512, 7, k_head_scale=True, seed=18),
    W.Workload("r48", 2, 16, 2, 128, (700, 1300), 256, 6, seed=22),   # 48 rows: row split, 16 idle
    W.Workload("r96", 2, 16, 4, 128, (500, 901), 128, 24, seed=23),   # 96 rows: two passes, last half empty
    W.Workload("r12", 2, 8, 4, 128, (600, 1025), 256, 6, seed=24),    # 12 rows: two 8-row column blocks
    W.Workload("r16", 3, 16, 8, 128, (129, 2000, 64), 512, 8, seed=25),  # 16 rows, exactly two blocks
    W.Workload("g1d128", 2, 8, 8, 128, (300, 129), 128, 3, seed=28),    # one query head per KV head
    # head dimension 64 with an even KV-head count and <= 32 rows per head: two heads per tile row
    W.Workload("pair_r32", 3, 64, 2, 64, (1000, 1, 300), 256, 1, seed=26),   # 32 rows per head, one pair
    W.Workload("pair_h6", 2, 12, 6, 64, (777, 129), 128, 5, seed=27),        # 10 rows per head, three pairs
    # head dimension 64 without head pairs: 16 KiB ring slots, the PV product's upper half not kept
    W.Workload("tree_d64", 3, 16, 4, 64, (200, 1300, 1), 128, 16, tree=True, seed=29),  # 64 rows: row split
    W.Workload("odd_d64", 2, 6, 3, 64, (700, 1031), 256, 5, seed=30),  # odd KV-head count: one head per tile
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
@pytest.mark.parametrize("resident", [False, True], ids=["streamed", "resident"])
@pytest.mark.parametrize("tc", [True, False], ids=["tc", "fma"])
def test_small_parity(svx, w, resident, tc):
    x, t = gpu_inputs(w, resident=resident)
    with make_verifier(svx, w, tensor_cores=tc) as v:
        o, l = run_gpu(v, w, t, x)
    check_parity(o, l, *oracle_out(w, x))


@pytest.mark.parametrize("hist", [(1,), (127,), (128,), (129,), (4095, 1, 300), (20000, 7000)])
def test_tile_edges_tensor_core_path(svx, hist):
    """Token counts around the 128-token tile and a stream-K split of unequal parts."""
    w = W.Workload("edge", len(hist), 32, 8, 128, hist, 4096, 5, seed=30 + len(hist))
    x, t = gpu_inputs(w, resident=True)
    with make_verifier(svx, w) as v:
        o, l = run_gpu(v, w, t, x)
    check_parity(o, l, *oracle_out(w, x))


# Tile-split corner cases of the tensor-core kernel: more (KV head, row pass) CTA groups than SMs
# (160 groups of one CTA, two waves), and one long request that would spread over more state slots
# than there are (the grid shrinks until it spans at most 8).
SPLIT_EDGES = [
    W.Workload("groups160", 1, 320, 40, 128, (300,), 128, 32, seed=26),
    W.Workload("long1", 1, 32, 8, 128, (60000,), 8192, 5, seed=27),
    # 70 requests: a push of more than 64 parts is split into several launches
    W.Workload("req70", 70, 8, 2, 128, tuple(17 + 13 * i for i in range(70)), 256, 3, seed=29),
    # the API's limits: 256 requests (a full staging slot, four launches per chunk), 32-node trees of any
    # depth (a full parent block in the finish launch), empty and ragged histories, 64 rows per KV head
    W.Workload("max256", 256, 4, 2, 128, tuple((37 * i) % 301 for i in range(256)), 64, 32, tree=True,
               tree_max_depth=31, seed=33),
]


@pytest.mark.parametrize("w", SPLIT_EDGES, ids=[w.name for w in SPLIT_EDGES])
@pytest.mark.parametrize("resident", [False, True], ids=["streamed", "resident"])
def test_tile_split_edges(svx, w, resident):
    x, t = gpu_inputs(w, resident=resident)
    with make_verifier(svx, w) as v:
        o, l = run_gpu(v, w, t, x)
    check_parity(o, l, *oracle_out(w, x))


@pytest.mark.parametrize("ragged", [False, True], ids=["equal", "ragged"])
def test_batched_host_history_is_copied_in_2d(svx, ragged):
    """History of all requests in one pinned [B][C][Hkv][d] tensor: the parts of a chunk are equally
    strided, so each chunk is staged with one 2D copy for K and one for V (ragged lengths: the
    chunks where every request still has a full chunk)."""
    import torch
    hist = (700, 300, 520, 129) if ragged else (700, 700, 700, 700)
    w = W.Workload("batched", 4, 16, 4, 128, hist, 128, 5, seed=31)
    x, t = gpu_inputs(w)
    cmax = max(hist)
    kb = torch.zeros((w.n_req, cmax, w.n_kv_heads, w.head_dim), dtype=torch.bfloat16).pin_memory()
    vb = torch.zeros_like(kb).pin_memory()
    for b in range(w.n_req):
        kb[b, :hist[b]].copy_(t["kh"][b])
        vb[b, :hist[b]].copy_(t["vh"][b])
    t["kh"] = [kb[b, :hist[b]] for b in range(w.n_req)]
    t["vh"] = [vb[b, :hist[b]] for b in range(w.n_req)]
    with make_verifier(svx, w, timing=True) as v:
        o, l = run_gpu(v, w, t, x)
        st = v.stats()
    check_parity(o, l, *oracle_out(w, x))
    chunks = {}
    for C in hist:
        for j in range(-(-C // w.chunk_tokens)):
            chunks.setdefault(j, []).append(min(w.chunk_tokens, C - j * w.chunk_tokens))
    expect = sum(2 if (len(n) > 1 and len(set(n)) == 1) else 2 * len(n) for n in chunks.values())
    assert st["n_copies"] == expect and st["h2d_bytes"] == w.hist_bytes


def test_chunk_order_does_not_matter(svx):
    w = SMALL[1]
    x, t = gpu_inputs(w)
    ref = oracle_out(w, x)
    n_chunks = max(-(-C // w.chunk_tokens) for C in w.hist_len)
    rng = np.random.default_rng(0)
    with make_verifier(svx, w, n_slots=3) as v:
        for order in (list(range(n_chunks))[::-1], list(rng.permutation(n_chunks))):
            o, l = run_gpu(v, w, t, x, chunk_order=order)
            check_parity(o, l, *ref)


def test_back_to_back_rounds_and_no_candidates(svx):
    w = SMALL[0].with_(n_req=2, hist_len=(512, 300))
    with make_verifier(svx, w) as v:
        for layer in range(3):
            x, t = gpu_inputs(w, layer=layer)
            o, l = run_gpu(v, w, t, x, with_candidates=(layer != 1), timeout_ms=60000)
            check_parity(o, l, *oracle_out(w, x, with_candidates=(layer != 1)))


def test_query_with_nothing_visible(svx):
    import torch
    w = W.Workload("empty", 2, 4, 2, 64, (0, 40), 16, 2, seed=19)
    x, t = gpu_inputs(w)
    with make_verifier(svx, w) as v:
        o, l = run_gpu(v, w, t, x, with_candidates=False)
    assert np.all(o[0] == 0) and np.all(np.isneginf(l[0]))
    ref = oracle_out(w, x, rows=[(1, h, j) for h in range(4) for j in range(2)], with_candidates=False)
    check_parity(o[1:], l[1:], ref[0][1:], ref[1][1:])
    del torch


def test_mixed_host_and_device_parts_in_one_push(svx):
    import torch
    w = W.Workload("mixed", 4, 8, 2, 128, (300, 260, 0, 511), 128, 5, seed=20)
    x, t = gpu_inputs(w)
    # requests 1 and 3 keep their history on the device, 0 stays pinned host memory
    for b in (1, 3):
        t["kh"][b] = t["kh"][b].cuda()
        t["vh"][b] = t["vh"][b].cuda()
    with make_verifier(svx, w) as v:
        o, l = run_gpu(v, w, t, x)
    check_parity(o, l, *oracle_out(w, x))
    del torch


def test_user_streams_and_timing_stats(svx):
    import torch
    w = SMALL[1]
    x, t = gpu_inputs(w)
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    with make_verifier(svx, w, compute_stream=cs, copy_stream=xs, timing=True) as v:
        o, l = run_gpu(v, w, t, x)
        st = v.stats()
    check_parity(o, l, *oracle_out(w, x))
    assert st["h2d_bytes"] == w.hist_bytes and st["device_bytes"] == 0
    n_parts = sum(-(-C // w.chunk_tokens) for C in w.hist_len)
    n_chunks = max(-(-C // w.chunk_tokens) for C in w.hist_len)
    assert 2 * n_chunks <= st["n_copies"] <= 2 * n_parts  # equally strided parts of a chunk share 2D copies
    assert st["round_ms"] > 0 and st["chunk_kernel_ms"] > 0 and st["copy_busy_ms"] > 0


@pytest.mark.parametrize("tc", [True, False], ids=["tc", "fma"])
def test_part_past_32_bit_element_offsets(svx, tc):
    """One resident part of 2,131,480 tokens (8 KV heads, d = 128: element offsets up to 2.18e9, past
    2^31).  Its history is a 4099-token block repeated 520 times and no candidate region is attended,
    so every key's weight is the block key's, counted 520 times: O equals the block's O and LSE the
    block's LSE + ln 520 (Eq. 9's normaliser).  The oracle computes the block alone."""
    import torch
    n, m = 4099, 520
    w = W.Workload("block", 1, 32, 8, 128, (n,), n, 5, seed=34)
    x, t = gpu_inputs(w, resident=True)
    kb = t["kh"][0].repeat(m, 1, 1)
    vb = t["vh"][0].repeat(m, 1, 1)
    assert kb.shape[0] * w.n_kv_heads * w.head_dim > 2 ** 31
    o = torch.empty((1, 32, 5, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 32, 5), dtype=torch.float32, device="cuda")
    with svx.Verifier(1, 32, 8, 128, 5, 64, n_slots=2, tensor_cores=tc) as v:
        v.run_round(t["q"], (n * m,), [kb], [vb], n * m, o, lse, timeout_ms=60000)
        torch.cuda.synchronize()
    og, lg = o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)
    del kb, vb, t
    torch.cuda.empty_cache()
    o_ref, l_ref = oracle_out(w, x, with_candidates=False)
    check_parity(og, lg, o_ref, l_ref + np.log(m))


# ---------------------------------------------------------------- errors


def test_state_machine_and_argument_errors(svx):
    import torch
    w = W.Workload("err", 2, 8, 2, 128, (100, 50), 64, 3, seed=21)
    x, t = gpu_inputs(w)
    o = torch.empty((2, 8, 3, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 8, 3), dtype=torch.float32, device="cuda")
    with make_verifier(svx, w) as v:
        def status(fn, *a, **k):
            try:
                fn(*a, **k)
                return svx.OK
            except svx.SvxError as e:
                return e.status

        kh, vh = t["kh"], t["vh"]
        assert status(v.push_chunk, [(0, 0, kh[0][:64], vh[0][:64])]) == svx.ERR_BAD_STATE
        assert status(v.round_finish, o, lse) == svx.ERR_BAD_STATE
        v.round_begin(t["q"], w.hist_len)
        assert status(v.round_begin, t["q"], w.hist_len) == svx.ERR_BAD_STATE
        # part past the end of the history, duplicate request, too many tokens for a slot
        assert status(v.push_chunk, [(1, 40, kh[1][:20], vh[1][:20])]) == svx.ERR_INVALID_ARG
        assert status(v.push_chunk, [(0, 0, kh[0][:10], vh[0][:10]), (0, 10, kh[0][10:20], vh[0][10:20])]) \
            == svx.ERR_INVALID_ARG
        assert status(v.push_chunk, [(0, 0, kh[0][:100], vh[0][:100])]) == svx.ERR_INVALID_ARG
        # pageable host memory cannot be streamed
        pk = torch.zeros((10, 2, 128), dtype=torch.bfloat16)
        assert status(v.push_chunk, [(0, 0, pk, pk)]) == svx.ERR_INVALID_ARG
        # wrong candidate count, bad tree
        assert status(v.candidate_attn, t["kc"][:, :2].contiguous(), t["vc"][:, :2].contiguous(), None, 2) \
            == svx.ERR_INVALID_ARG
        # tensors whose layout is not the C layout are refused before the call
        assert status(v.candidate_attn, t["kc"].transpose(2, 3), t["vc"], None) == svx.ERR_INVALID_ARG
        assert status(v.push_chunk, [(0, 0, kh[0][:64].float(), vh[0][:64])]) == svx.ERR_INVALID_ARG
        assert status(v.candidate_attn, t["kc"], t["vc"], np.array([[0, 0, 1], [-1, 0, 1]])) == svx.ERR_INVALID_ARG
        # a missing chunk fails the coverage check at finish and closes the round
        v.push_chunk([(0, 0, kh[0][:64], vh[0][:64]), (1, 0, kh[1][:50], vh[1][:50])])
        assert status(v.round_finish, o, lse) == svx.ERR_INVALID_ARG
        assert "coverage" in svx.lib.svx_last_error(v._h).decode()
        # duplicate coverage is rejected too
        v.round_begin(t["q"], w.hist_len)
        v.push_chunk([(0, 0, kh[0][:64], vh[0][:64]), (1, 0, kh[1][:50], vh[1][:50])])
        v.push_chunk([(0, 64, kh[0][64:], vh[0][64:])])
        v.push_chunk([(0, 64, kh[0][64:], vh[0][64:])])
        assert status(v.round_finish, o, lse) == svx.ERR_INVALID_ARG
        # and the context still computes a correct round afterwards
        o2, l2 = run_gpu(v, w, t, x, timeout_ms=60000)
    check_parity(o2, l2, *oracle_out(w, x))


# ---------------------------------------------------------------- full size, sampled rows


@pytest.mark.parametrize("name", ["qwen3", "internlm", "tree", "fulldepth"])
def test_full_size_sampled(svx, name):
    w = W.named(name)
    if name == "fulldepth":
        w = w.with_(n_layers=1)  # one layer of the 36-layer stack: same shapes per layer
    x, t = gpu_inputs(w)
    with make_verifier(svx, w, n_slots=3) as v:
        o, l = run_gpu(v, w, t, x)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    rows = sample_rows(w, 24)
    ref = oracle_out(w, x, rows=rows)
    check_parity(o, l, *ref, rows=rows)


@pytest.mark.parametrize("name", ["qwen3", "tree"])
def test_head_dim_64_at_full_size_sampled(svx, name):
    """The qwen3 and tree shapes with d = 64 (the tiny workload's head dimension) at full size, history
    resident in HBM and pushed as one part per request, as the benchmark's resident round does."""
    w0 = W.named(name)
    w = w0.with_(name=name + "_d64", head_dim=64, chunk_tokens=max(w0.hist_len))
    x, t = gpu_inputs(w, resident=True)
    with make_verifier(svx, w, n_slots=3, chunk=w0.chunk_tokens) as v:
        o, l = run_gpu(v, w, t, x)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    rows = sample_rows(w, 24)
    ref = oracle_out(w, x, rows=rows)
    check_parity(o, l, *ref, rows=rows)


def test_full_depth_rounds_back_to_back_with_prefetch(svx):
    """36 layer rounds enqueued without any host wait (finish with timeout 0), so each layer's
    chunk copies queue behind the previous layer's: cross-layer prefetch through the slot events.
    Inputs come from the device-side generator and are read back from pinned host memory for the
    oracle.  Sampled rows of the first, a middle and the last layer are checked."""
    import torch
    w = W.named("fulldepth").with_(hist_len=(4096, 3000), chunk_tokens=1024)
    bf = torch.bfloat16
    layers = []
    for l in range(w.n_layers):
        kh = [torch.empty((C, w.n_kv_heads, w.head_dim), dtype=bf, pin_memory=True) for C in w.hist_len]
        vh = [torch.empty((C, w.n_kv_heads, w.head_dim), dtype=bf, pin_memory=True) for C in w.hist_len]
        q, _, _, kc, vc, parent = W.layer_inputs_device(w, l, "cuda", hist_out_k=kh, hist_out_v=vh)
        o = torch.empty((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=bf, device="cuda")
        lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
        layers.append((q, kh, vh, kc, vc, o, lse))
    torch.cuda.synchronize()
    with make_verifier(svx, w, n_slots=3) as v:
        for q, kh, vh, kc, vc, o, lse in layers:
            v.run_round(q, w.hist_len, kh, vh, w.chunk_tokens, o, lse, cand_k=kc, cand_v=vc)
        torch.cuda.synchronize()
    u16 = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)  # noqa: E731
    for l in (0, 17, 35):
        q, kh, vh, kc, vc, o, lse = layers[l]
        x = W.LayerInputs(u16(q), [u16(k) for k in kh], [u16(v_) for v_ in vh], u16(kc), u16(vc), None)
        rows = sample_rows(w, 12, seed=l)
        o_gpu = o.float().cpu().numpy().astype(np.float64)
        l_gpu = lse.cpu().numpy().astype(np.float64)
        check_parity(o_gpu, l_gpu, *oracle_out(w, x, rows=rows), rows=rows)


ZC = [SMALL[0], SMALL[1], SMALL[3], SMALL[8], SMALL[14], SMALL[15], SMALL[16], SMALL[17]]  # tiny, ragged, tree64,
# kscale, head pairs, d = 64 with one head per tile


@pytest.mark.parametrize("w", ZC, ids=[w.name for w in ZC])
@pytest.mark.parametrize("cap", [0, 8])
def test_zero_copy_reads_host_history_in_place(svx, w, cap):
    """SVX_FLAG_ZERO_COPY: pinned host parts go to the chunk kernel without a staging copy, on at
    most `cap` CTAs (0 = all SMs); whole-history parts exceed max_chunk_tokens on purpose."""
    x, t = gpu_inputs(w)
    with make_verifier(svx, w, zero_copy=True, zero_copy_ctas=cap, timing=True) as v:
        o, l = run_gpu(v, w, t, x, chunk_order=None)
        st = v.stats()
        assert st["n_copies"] == 0 and st["h2d_bytes"] == w.hist_bytes
        # whole histories in one push each
        import torch
        o2 = torch.empty((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=torch.bfloat16, device="cuda")
        l2 = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
        v.round_begin(t["q"], w.hist_len)
        v.candidate_attn(t["kc"], t["vc"], x.parent)
        v.push_chunk([(b, 0, t["kh"][b], t["vh"][b]) for b in range(w.n_req) if w.hist_len[b]])
        v.round_finish(o2, l2, timeout_ms=60000)
    ref = oracle_out(w, x)
    check_parity(o, l, *ref)
    check_parity(o2.float().cpu().numpy().astype(np.float64), l2.cpu().numpy().astype(np.float64), *ref)


def test_tiering_migration_feeds_the_next_round(svx):
    """Commit-aware tiering end to end: Eq. (5) picks [H, E), the history rows move device -> pinned
    host asynchronously, H advances only once the copy is done, and the next round streams the
    Sealed History [0, H) from host memory while reading the Active Tail [H, C) in place."""
    import time as _time
    import torch
    w = W.Workload("tier", 2, 8, 2, 128, (1500, 700), 256, 5, seed=50)
    x, t = gpu_inputs(w, resident=True)
    row_bytes = w.n_kv_heads * w.head_dim * 2
    T, g = 512, 128
    host_k = [torch.zeros_like(k, device="cpu").pin_memory() for k in t["kh"]]
    host_v = [torch.zeros_like(v, device="cpu").pin_memory() for v in t["vh"]]
    tiers = []
    stream = torch.cuda.Stream()
    for b in range(w.n_req):
        tr = svx.Tier()
        C = w.hist_len[b]
        tr.round(C, C + w.n_query)
        E = tr.migrate(T, g, row_bytes, t["kh"][b], t["vh"][b], host_k[b], host_v[b], stream=stream)
        assert E == max(0, g * ((C - T) // g)) and tr.H == 0  # nothing confirmed yet
        deadline = _time.time() + 30
        while not tr.poll():
            assert _time.time() < deadline
            _time.sleep(0.001)
        assert tr.H == E and tr.pending is None
        assert torch.equal(host_k[b][:E], t["kh"][b][:E].cpu()) and torch.equal(host_v[b][:E], t["vh"][b][:E].cpu())
        tiers.append(tr)
    o = torch.empty((w.n_req, w.n_q_heads, w.n_query, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.n_req, w.n_q_heads, w.n_query), dtype=torch.float32, device="cuda")
    with make_verifier(svx, w) as v:
        v.round_begin(t["q"], w.hist_len)
        v.candidate_attn(t["kc"], t["vc"], x.parent)
        for b, tr in enumerate(tiers):  # Sealed History from host, chunk by chunk
            for t0 in range(0, tr.H, w.chunk_tokens):
                n = min(w.chunk_tokens, tr.H - t0)
                v.push_chunk([(b, t0, host_k[b][t0:t0 + n], host_v[b][t0:t0 + n])])
        v.push_chunk([(b, tr.H, t["kh"][b][tr.H:], t["vh"][b][tr.H:]) for b, tr in enumerate(tiers)])
        v.round_finish(o, lse, timeout_ms=60000)
    check_parity(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                 *oracle_out(w, x))
    for tr in tiers:  # two of five candidates accepted; the rejected suffix never meets [0, H)
        C0, L0 = tr.C, tr.L
        rel = tr.commit(C0 + 2)
        assert rel == (C0 + 2, L0) and rel[0] >= tr.H and tr.C == tr.L == C0 + 2


def test_a_wait_that_runs_out_is_reported_and_the_context_runs_on(svx):
    """Failure path without a fault: a kernel whose bounded wait on a barrier that nothing completes
    runs out (0.2 s) raises the device error word; the next round's finish reports it, clears it, and
    the round after that is correct again.  Inside an open round the hook is refused."""
    w = SMALL[2]
    x, t = gpu_inputs(w)
    ref = oracle_out(w, x)
    with make_verifier(svx, w) as v:
        check_parity(*run_gpu(v, w, t, x, timeout_ms=60000), *ref)
        v.debug_expire_wait(200)
        with pytest.raises(svx.SvxError) as ei:
            run_gpu(v, w, t, x, timeout_ms=60000)
        assert ei.value.status == svx.ERR_CUDA and "gave up waiting" in ei.value.message
        check_parity(*run_gpu(v, w, t, x, timeout_ms=60000), *ref)
        v.round_begin(t["q"], w.hist_len)
        with pytest.raises(svx.SvxError) as ei:
            v.debug_expire_wait(200)
        assert ei.value.status == svx.ERR_BAD_STATE
