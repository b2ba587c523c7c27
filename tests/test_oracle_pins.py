"""Pins of the float64 oracle against things other than itself.

Each test is chosen so that a plausible slip in the oracle (wrong scale, a
transposed mask, h % G instead of h // G, a dropped history or candidate
term, a mis-signed LSE, a bad merge of empty chunks) fails at least one of
them.  All run on the CPU.

Sources: "Resource-Efficient Speculative Decoding for Long-Context LLM
Serving", section 4.2, Eqs. (6)-(9); "Speculative Streaming" blog, section 2
mask-topology figure (printed mask example).
"""
import math
import os

import numpy as np
import pytest

import oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(B=2, Hq=4, Hkv=2, d=8, hist=(7, 3), nq=3, tree=False, seed=0, scale_k=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, nq, d))
    kh = [rng.standard_normal((C, Hkv, d)) * scale_k for C in hist]
    vh = [rng.standard_normal((C, Hkv, d)) for C in hist]
    kc = rng.standard_normal((B, nq, Hkv, d)) * scale_k
    vc = rng.standard_normal((B, nq, Hkv, d))
    parents = None
    if tree:
        parents = np.stack([W.random_tree(np.random.default_rng([seed, b]), nq, 3) for b in range(B)])
    vis = O.visibility_table(B, nq, parents)
    return q, kh, vh, kc, vc, vis, parents


# ------------------------------------------------------------ masks


def test_printed_block_causal_mask_example():
    rows = []
    with open(os.path.join(GOLDEN, "block_causal_mask_example.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x) for x in line.split()[1:]])
    n_hist, n_cand = 4, 2
    words = O.candidate_visibility(n_cand)
    ours = [[1] * n_hist + [(int(words[j]) >> i) & 1 for i in range(n_cand)] for j in range(n_cand)]
    assert ours == rows


def test_tree_visibility_matches_graph_library_ancestors():
    nx = pytest.importorskip("networkx")
    for seed in range(20):
        n = 1 + seed % 16 + (16 if seed % 3 == 0 else 0)
        parent = W.random_tree(np.random.default_rng(seed), n, 5)
        g = nx.DiGraph()
        g.add_nodes_from(range(n))
        g.add_edges_from((int(parent[i]), i) for i in range(1, n))
        words = O.candidate_visibility(n, parent)
        for j in range(n):
            expect = nx.ancestors(g, j) | {j}
            got = {i for i in range(n) if (int(words[j]) >> i) & 1}
            assert got == expect


def test_chain_equals_linear_tree():
    for n in range(1, 33):
        parent = np.arange(-1, n - 1, dtype=np.int32)
        assert np.array_equal(O.candidate_visibility(n), O.candidate_visibility(n, parent))


def test_tree_generator_depth_and_order():
    for b in range(50):
        p = W.random_tree(np.random.default_rng(b), 16, 5)
        assert p[0] == -1 and all(0 <= p[i] < i for i in range(1, 16))
        for i in range(16):
            depth, node = 0, i
            while p[node] >= 0:
                node, depth = p[node], depth + 1
            assert depth <= 5


def test_bad_parents_rejected():
    with pytest.raises(ValueError):
        O.candidate_visibility(3, [-1, 2, 0])
    with pytest.raises(ValueError):
        O.candidate_visibility(3, [0, 0, 1])
    with pytest.raises(ValueError):
        O.candidate_visibility(33)


# ------------------------------------------------------------ chunk plan


def test_chunk_plan_hand_example():
    # histories of 5, 0 and 9 tokens in chunks of 4 over 2 staging buffers
    expect = [(0, 0, 0, 0, 4), (0, 0, 2, 0, 4), (1, 1, 0, 4, 1), (1, 1, 2, 4, 4), (2, 0, 2, 8, 1)]
    assert O.cohort_chunk_plan([5, 0, 9], 4, 2) == expect


def test_chunk_plan_properties():
    rng = np.random.default_rng(3)
    for _ in range(30):
        hist = [int(x) for x in rng.integers(0, 50, size=int(rng.integers(1, 6)))]
        c = int(rng.integers(1, 9))
        ns = int(rng.integers(2, 4))
        plan = O.cohort_chunk_plan(hist, c, ns)
        assert O.covers_exactly_once(hist, [(b, t0, n) for _, _, b, t0, n in plan])
        assert all(s == j % ns for j, s, _, _, _ in plan)
        assert max([j for j, *_ in plan], default=-1) + 1 == max([-(-C // c) for C in hist])


def test_coverage_detects_gaps_and_overlaps():
    hist = [10, 4]
    good = [(0, 0, 4), (0, 4, 6), (1, 0, 4)]
    assert O.covers_exactly_once(hist, good)
    assert not O.covers_exactly_once(hist, good[:2])  # request 1 missing
    assert not O.covers_exactly_once(hist, good + [(1, 0, 4)])  # duplicate
    assert not O.covers_exactly_once(hist, [(0, 0, 5), (0, 4, 6), (1, 0, 4)])  # overlap
    assert not O.covers_exactly_once(hist, [(0, 0, 4), (0, 4, 7), (1, 0, 4)])  # past the end
    assert O.covers_exactly_once([0, 0], [])


# ------------------------------------------------------------ attention


def test_brute_force_high_precision():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    for seed, hist, nq in [(0, (3, 0), 2), (1, (1, 5), 3), (2, (0, 2), 1), (3, (4, 4), 4)]:
        B, Hq, Hkv, d = 2, 2, 1, 4
        rng = np.random.default_rng(seed)
        q = rng.uniform(-1, 1, (B, Hq, nq, d))
        kh = [rng.uniform(-1, 1, (C, Hkv, d)) for C in hist]
        vh = [rng.uniform(-1, 1, (C, Hkv, d)) for C in hist]
        kc = rng.uniform(-1, 1, (B, nq, Hkv, d))
        vc = rng.uniform(-1, 1, (B, nq, Hkv, d))
        vis = O.visibility_table(B, nq, None)
        Ov, Lv = O.verify_attention(q, kh, vh, kc, vc, vis)
        for b in range(B):
            for h in range(Hq):
                for j in range(nq):
                    keys = [(kh[b][t, 0], vh[b][t, 0]) for t in range(hist[b])]
                    keys += [(kc[b, i, 0], vc[b, i, 0]) for i in range(j + 1)]  # chain: candidates 0..j
                    w = [mp.exp(mp.fsum(mp.mpf(float(x)) * mp.mpf(float(y)) for x, y in zip(q[b, h, j], k))
                                / mp.sqrt(d)) for k, _ in keys]
                    Z = mp.fsum(w)
                    assert abs(float(mp.log(Z)) - Lv[b, h, j]) < 1e-13
                    for c in range(d):
                        o = mp.fsum(wi * mp.mpf(float(v[c])) for wi, (_, v) in zip(w, keys)) / Z
                        assert abs(float(o) - Ov[b, h, j, c]) < 1e-13


def test_library_sdpa_and_logsumexp():
    torch = pytest.importorskip("torch")
    from scipy.special import logsumexp
    for tree in (False, True):
        q, kh, vh, kc, vc, vis, _ = rand_case(B=3, Hq=8, Hkv=2, d=16, hist=(9, 0, 17), nq=5, tree=tree, seed=5)
        Ov, Lv = O.verify_attention(q, kh, vh, kc, vc, vis)
        B, Hq, nq, d = q.shape
        G = Hq // kc.shape[2]
        for b in range(B):
            K = torch.from_numpy(np.concatenate([kh[b], kc[b]], 0)).permute(1, 0, 2)  # [Hkv][T][d]
            V = torch.from_numpy(np.concatenate([vh[b], vc[b]], 0)).permute(1, 0, 2)
            K = K.repeat_interleave(G, dim=0)
            V = V.repeat_interleave(G, dim=0)
            C = kh[b].shape[0]
            allow = torch.ones(nq, C + nq, dtype=torch.bool)
            for j in range(nq):
                for i in range(nq):
                    allow[j, C + i] = bool((int(vis[b, j]) >> i) & 1)
            ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q[b]), K, V, attn_mask=allow)
            assert np.max(np.abs(ref.numpy() - Ov[b])) < 1e-12
            s = torch.matmul(torch.from_numpy(q[b]), K.transpose(1, 2)).numpy() / math.sqrt(d)
            s = np.where(allow.numpy()[None], s, -np.inf)
            assert np.max(np.abs(logsumexp(s, axis=-1) - Lv[b])) < 1e-12


def test_equal_keys_closed_form():
    q, kh, vh, kc, vc, vis, _ = rand_case(B=2, Hq=4, Hkv=2, d=8, hist=(6, 11), nq=4, tree=True, seed=1)
    kconst = np.linspace(-1, 1, 8)
    kh = [np.broadcast_to(kconst, k.shape).copy() for k in kh]
    kc = np.broadcast_to(kconst, kc.shape).copy()
    Ov, Lv = O.verify_attention(q, kh, vh, kc, vc, vis)
    for b in range(2):
        for h in range(4):
            g = h // 2
            for j in range(4):
                cand = [i for i in range(4) if (int(vis[b, j]) >> i) & 1]
                Vvis = np.concatenate([vh[b][:, g], vc[b, cand, g]], 0)
                s = float(q[b, h, j] @ kconst) / math.sqrt(8)
                assert abs(Lv[b, h, j] - (s + math.log(len(Vvis)))) < 1e-12
                assert np.max(np.abs(Ov[b, h, j] - Vvis.mean(0))) < 1e-12


def test_zero_query_gives_uniform_weights():
    q, kh, vh, kc, vc, vis, _ = rand_case(B=1, Hq=2, Hkv=1, d=4, hist=(13,), nq=3, seed=2)
    q[:] = 0
    Ov, Lv = O.verify_attention(q, kh, vh, kc, vc, vis)
    for j in range(3):
        Vvis = np.concatenate([vh[0][:, 0], vc[0, :j + 1, 0]], 0)
        assert abs(Lv[0, 0, j] - math.log(13 + j + 1)) < 1e-12
        assert np.max(np.abs(Ov[0, 1, j] - Vvis.mean(0))) < 1e-12


def test_three_two_one_weights():
    # d=4, scale 1/2: q = (2,0,0,0) makes each score equal to the key's first
    # component.  Keys ln1, ln3 (history) and ln2 (the query's own candidate)
    # give weights 1:3:2 -> O = (v0 + 3 v1 + 2 v2) / 6 and LSE = ln 6.
    d = 4
    q = np.zeros((1, 1, 1, d)); q[0, 0, 0, 0] = 2.0
    kh = [np.zeros((2, 1, d))]; kh[0][1, 0, 0] = math.log(3)
    kc = np.zeros((1, 1, 1, d)); kc[0, 0, 0, 0] = math.log(2)
    v = np.array([[1.0, 0, 0, 5], [0, 1.0, 0, -1], [0, 0, 1.0, 2]])
    vh = [v[:2, None, :].copy()]
    vc = v[2][None, None, None, :].copy()
    vis = O.visibility_table(1, 1, None)
    Ov, Lv = O.verify_attention(q, kh, vh, kc, vc, vis)
    assert abs(Lv[0, 0, 0] - math.log(6)) < 1e-14
    assert np.max(np.abs(Ov[0, 0, 0] - np.array([1, 3, 2, 5 - 3 + 4]) / 6)) < 1e-14


def test_spike_key_dominates():
    q, kh, vh, kc, vc, vis, _ = rand_case(B=1, Hq=1, Hkv=1, d=8, hist=(50,), nq=1, seed=4)
    q[0, 0, 0] = 0
    q[0, 0, 0, 0] = math.sqrt(8)  # score = key component 0
    for k in kh[0][:, 0]:
        k[0] = 0.0
    kc[0, 0, 0, 0] = 0.0
    kh[0][17, 0, 0] = 60.0
    Ov, _ = O.verify_attention(q, kh, vh, kc, vc, vis)
    assert np.max(np.abs(Ov[0, 0, 0] - vh[0][17, 0])) < 1e-20 + 1e-24


def test_grouped_query_head_mapping():
    q, kh, vh, kc, vc, vis, _ = rand_case(B=1, Hq=8, Hkv=4, d=4, hist=(9,), nq=2, seed=6)
    for g in range(4):
        vh[0][:, g, :] = g + 1
        vc[0, :, g, :] = g + 1
    Ov, _ = O.verify_attention(q, kh, vh, kc, vc, vis)
    for h in range(8):
        assert np.allclose(Ov[0, h], h // 2 + 1, atol=1e-13)


@pytest.mark.parametrize("tree", [False, True])
def test_streamed_equals_full_any_chunking(tree):
    q, kh, vh, kc, vc, vis, _ = rand_case(B=3, Hq=4, Hkv=2, d=8, hist=(200, 0, 131), nq=6, tree=tree, seed=7,
                                          scale_k=3.0)
    Ov, Lv = O.verify_attention(q, kh, vh, kc, vc, vis)
    rng = np.random.default_rng(0)
    for c in (1, 3, 128, 200):
        n = -(-200 // c)
        for order in (None, list(range(n))[::-1], list(rng.permutation(n))):
            Os, Ls = O.verify_attention_streamed(q, kh, vh, kc, vc, vis, c, chunk_order=order)
            assert np.max(np.abs(Os - Ov)) < 1e-12
            assert np.max(np.abs(Ls - Lv)) < 1e-12


def test_k0_reduces_to_single_token_decode():
    torch = pytest.importorskip("torch")
    q, kh, vh, kc, vc, vis, _ = rand_case(B=2, Hq=4, Hkv=4, d=16, hist=(33, 1), nq=1, seed=8)
    Ov, _ = O.verify_attention(q, kh, vh, kc, vc, vis)
    for b in range(2):
        K = torch.from_numpy(np.concatenate([kh[b], kc[b]], 0)).permute(1, 0, 2)
        V = torch.from_numpy(np.concatenate([vh[b], vc[b]], 0)).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q[b]), K, V)
        assert np.max(np.abs(ref.numpy() - Ov[b])) < 1e-12


def test_invisible_candidates_do_not_matter():
    q, kh, vh, kc, vc, vis, _ = rand_case(B=2, Hq=4, Hkv=2, d=8, hist=(5, 12), nq=8, tree=True, seed=9)
    O1, L1 = O.verify_attention(q, kh, vh, kc, vc, vis)
    for b in range(2):
        for j in range(8):
            kc2, vc2 = kc.copy(), vc.copy()
            for i in range(8):
                if not (int(vis[b, j]) >> i) & 1:
                    kc2[b, i] += 7.0
                    vc2[b, i] -= 3.0
            O2, L2 = O.verify_attention(q, kh, vh, kc2, vc2, vis)
            assert np.array_equal(O1[b, :, j], O2[b, :, j]) and np.array_equal(L1[b, :, j], L2[b, :, j])
            # and a visible candidate does matter
            i = j
            kc3 = kc.copy(); kc3[b, i] += 1.0
            O3, _ = O.verify_attention(q, kh, vh, kc3, vc, vis)
            assert not np.array_equal(O1[b, :, j], O3[b, :, j])


def test_history_is_visible_to_every_query():
    q, kh, vh, kc, vc, vis, _ = rand_case(B=1, Hq=2, Hkv=1, d=8, hist=(20,), nq=5, seed=10)
    O1, _ = O.verify_attention(q, kh, vh, kc, vc, vis)
    vh2 = [vh[0].copy()]
    vh2[0][19] += 1.0  # the last history token changes every query's output
    O2, _ = O.verify_attention(q, kh, vh2, kc, vc, vis)
    assert np.all(np.abs(O1 - O2).max(axis=-1) > 0)


def test_round_bf16_matches_nearest_representable():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))
    r = O.round_bf16(x)
    # every result is a bf16 value
    as_bf16 = torch.from_numpy(r).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(as_bf16, r)
    # and no bf16 neighbour is nearer
    bits = torch.from_numpy(r.astype(np.float32)).view(torch.int32).numpy()
    up = (torch.from_numpy(bits + (1 << 16)).view(torch.float32)).numpy().astype(np.float64)
    dn = (torch.from_numpy(bits - (1 << 16)).view(torch.float32)).numpy().astype(np.float64)
    assert np.all(np.abs(r - x) <= np.abs(up - x)) and np.all(np.abs(r - x) <= np.abs(dn - x))
    # ties go to the even mantissa
    assert O.round_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    assert O.round_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6


def test_parity_bar_allows_only_the_bf16_output_rounding_beyond_the_tolerance():
    """The GPU parity bar: O error beyond half a bf16 ulp of the exact value (max <= 1e-2), raw O
    error (mean <= 1e-3), LSE error relative to max(|LSE|, 1).  Pinned on hand-made errors at the
    boundaries."""
    import pytest as _pt
    from helpers import bf16_half_ulp, check_parity
    o_ref = np.zeros((1, 200))
    o_ref[0, :4] = [4.075, 0.3, -1.5, 0.0]
    l_ref = np.array([9.0, 0.001, -np.inf, 2.0])
    assert np.allclose(bf16_half_ulp(o_ref[0, :4]), [2.0 ** -6, 2.0 ** -10, 2.0 ** -8, 0.0])

    def bump(k, v):
        o = o_ref.copy()
        o[0, k] += v
        return o
    # 0.0156 of rounding at 4.075 plus 0.009 of error passes; 0.011 beyond it does not
    check_parity(bump(0, 2.0 ** -6 + 0.009), l_ref, o_ref, l_ref)
    with _pt.raises(AssertionError):
        check_parity(bump(0, 2.0 ** -6 + 0.011), l_ref, o_ref, l_ref)
    with _pt.raises(AssertionError):  # at 0.3 the rounding allowance is only 2^-10
        check_parity(bump(1, 0.0115), l_ref, o_ref, l_ref)
    with _pt.raises(AssertionError):  # the mean bar: 0.006 beyond rounding on every element
        check_parity(o_ref + 0.006 + bf16_half_ulp(o_ref), l_ref, o_ref, l_ref)
    # the mean bar is on the raw error: a systematic 1.1e-3 on every element fails even where half a
    # bf16 ulp would have covered it, and a 9e-4 one passes
    o_mid = np.full((1, 200), 0.3)
    l_mid = np.full(1, 5.0)
    with _pt.raises(AssertionError):
        check_parity(o_mid + 1.1e-3, l_mid, o_mid, l_mid)
    check_parity(o_mid + 9e-4, l_mid, o_mid, l_mid)
    # exact values rounded to bf16 (what a perfect kernel writes) pass at every magnitude the
    # configured workloads produce
    from oracle import round_bf16
    rng = np.random.default_rng(3)
    o_exact = rng.standard_normal((64, 128)) * 0.3
    l_exact = np.full(64, 9.0)
    _, mean_err, _ = check_parity(round_bf16(o_exact), l_exact, o_exact, l_exact)
    assert mean_err < 5e-4
    # an LSE near zero is held to 1e-4 absolute, a large one to 1e-4 relative
    check_parity(o_ref, l_ref + [8e-4, 9e-5, 0, 1.9e-4], o_ref, l_ref)
    with _pt.raises(AssertionError):
        check_parity(o_ref, l_ref + [0, 1.1e-4, 0, 0], o_ref, l_ref)
    with _pt.raises(AssertionError):
        check_parity(o_ref, l_ref + [1.0e-3, 0, 0, 0], o_ref, l_ref)
    l_bad = l_ref.copy()
    l_bad[2] = 0.0
    with _pt.raises(AssertionError):  # -inf (nothing visible) must stay -inf
        check_parity(o_ref, l_bad, o_ref, l_ref)
