"""The C library loads, exports every symbol its header declares, and its host-only
bookkeeping (chunk plan, candidate visibility words, coverage check) matches the
oracle bit for bit.  No GPU needed: none of these calls touches a device."""
import os
import re

import numpy as np
import pytest

import oracle as O
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "svx.h")


@pytest.fixture(scope="module")
def svx():
    from speculative_decoding_verification_chunked_gb300 import build
    if not (os.path.exists(build.LIB) and os.path.exists(build.LIB_CHECKED)):
        build.build()
    from speculative_decoding_verification_chunked_gb300 import svx as mod
    return mod


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(svx_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(svx):
    names = header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(svx.lib, n), n
    assert sorted(svx.SYMBOLS) == names
    assert "sm_103a" in svx.version()


def test_bounds_checked_library_exports_the_same_symbols(svx):
    """libsvx_checked.so (the bounds-checked build) is a drop-in for libsvx.so: same ABI."""
    import ctypes
    from speculative_decoding_verification_chunked_gb300 import build
    checked = ctypes.CDLL(build.LIB_CHECKED)
    for n in header_functions():
        assert hasattr(checked, n), n
    sizes = (ctypes.c_int64 * 16)()
    checked.svx_abi_sizes.restype = ctypes.c_int32
    n = checked.svx_abi_sizes(sizes, 16)
    assert list(sizes[:n]) == list(svx.abi_sizes().values())


def test_plan_matches_oracle_on_named_workloads(svx):
    for name in W.NAMES:
        w = W.named(name)
        for ns in (2, 3):
            assert svx.plan_chunks(w.hist_len, w.chunk_tokens, ns) == \
                [(j, s, b, t0, n) for j, s, b, t0, n in O.cohort_chunk_plan(w.hist_len, w.chunk_tokens, ns)]


def test_plan_matches_oracle_random(svx):
    rng = np.random.default_rng(0)
    for _ in range(200):
        hist = [int(x) for x in rng.integers(0, 3000, size=int(rng.integers(1, 20)))]
        if rng.random() < 0.2:
            hist[0] = 0
        c = int(rng.integers(1, 700))
        ns = int(rng.integers(1, 4))
        assert svx.plan_chunks(hist, c, ns) == O.cohort_chunk_plan(hist, c, ns)
    assert svx.plan_chunks([0, 0], 5, 2) == []


def test_masks_match_oracle(svx):
    rng = np.random.default_rng(1)
    for nq in (1, 2, 5, 7, 16, 31, 32):
        assert np.array_equal(svx.candidate_masks(3, nq), O.visibility_table(3, nq, None))
        par = np.stack([W.random_tree(np.random.default_rng([nq, b]), nq, 5) for b in range(4)])
        assert np.array_equal(svx.candidate_masks(4, nq, par), O.visibility_table(4, nq, par))
        par = np.stack([W.random_tree(np.random.default_rng([nq, b, 9]), nq, 40) for b in range(2)])
        assert np.array_equal(svx.candidate_masks(2, nq, par), O.visibility_table(2, nq, par))
    w = W.named("tree")
    par = W.tree_parents(w)
    assert np.array_equal(svx.candidate_masks(w.n_req, w.n_query, par), O.visibility_table(w.n_req, w.n_query, par))
    del rng


def test_masks_reject_bad_trees(svx):
    for bad in ([0, 0, 1], [-1, 1, 0], [-1, 0, 3], [-1, -1, 0]):
        with pytest.raises(svx.SvxError):
            svx.candidate_masks(1, 3, np.array([bad]))
        with pytest.raises(ValueError):
            O.candidate_visibility(3, bad)
    with pytest.raises(svx.SvxError):
        svx.candidate_masks(1, 33)


def test_coverage_matches_oracle(svx):
    rng = np.random.default_rng(2)
    for trial in range(400):
        hist = [int(x) for x in rng.integers(0, 40, size=int(rng.integers(1, 5)))]
        plan = O.cohort_chunk_plan(hist, int(rng.integers(1, 9)), 2)
        parts = [(b, t0, n) for _, _, b, t0, n in plan]
        kind = trial % 6
        if kind == 1 and parts:
            parts.pop(int(rng.integers(0, len(parts))))
        elif kind == 2 and parts:
            parts.append(parts[int(rng.integers(0, len(parts)))])
        elif kind == 3 and parts:
            i = int(rng.integers(0, len(parts)))
            b, t0, n = parts[i]
            parts[i] = (b, max(0, t0 + int(rng.integers(-2, 3))), max(1, n + int(rng.integers(-2, 3))))
        elif kind == 4:
            parts.append((int(rng.integers(-1, len(hist) + 1)), int(rng.integers(-1, 50)), int(rng.integers(-1, 9))))
        elif kind == 5:
            rng.shuffle(parts)
        assert svx.check_coverage(hist, parts) == O.covers_exactly_once(hist, parts), (hist, parts)


def test_coverage_rejects_parts_whose_end_does_not_fit_64_bits(svx):
    """A part's end (start + length) past the int64 range lies outside every history."""
    big = (1 << 63) - 1
    for parts in ([(0, big, 1)], [(0, big - 5, 10)], [(0, 0, 10), (0, 10, big)], [(0, 10, big), (0, 0, 10)]):
        assert not svx.check_coverage([10], parts), parts
        assert not O.covers_exactly_once([10], parts), parts
    assert svx.check_coverage([big], [(0, 0, big)])


def test_create_rejects_bad_config_without_touching_a_device(svx):
    bad = [dict(head_dim=96), dict(max_query=33), dict(n_q_heads=12, n_kv_heads=8), dict(n_slots=4),
           dict(max_req=0), dict(max_chunk_tokens=0)]
    for kw in bad:
        args = dict(max_req=2, n_q_heads=8, n_kv_heads=2, head_dim=128, max_query=5, max_chunk_tokens=64)
        args.update(kw)
        with pytest.raises(svx.SvxError) as e:
            svx.Verifier(**args)
        assert e.value.status in (svx.ERR_INVALID_ARG, svx.ERR_UNSUPPORTED)


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib.util
    src = os.path.join(ROOT, "speculative_decoding_verification_chunked_gb300", "svx.py")
    dst = tmp_path / "svx_copy.py"
    dst.write_text(open(src).read())
    spec = importlib.util.spec_from_file_location("svx_copy", dst)
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


def test_tiering_matches_oracle(svx):
    from oracle.tiering import TierState, migration_endpoint
    rng = np.random.default_rng(5)
    for _ in range(3000):
        g = int(rng.choice([1, 16, 128]))
        T = int(rng.integers(0, 1024))
        H = g * int(rng.integers(0, 50))
        C = H + int(rng.integers(0, 3000))
        assert svx.migration_endpoint(H, C, T, g) == migration_endpoint(H, C, T, g)
    with pytest.raises(svx.SvxError):
        svx.migration_endpoint(3, 10, 5, 2)
    for trial in range(100):
        T, g = int(rng.integers(0, 600)), int(rng.choice([32, 128]))
        a, o = svx.Tier(), TierState()
        for _ in range(50):
            k = int(rng.integers(1, 9))
            a.round(a.C, a.C + k)
            o.round(o.C, o.C + k)
            assert a.plan(T, g) == o.plan(T, g)
            if rng.random() < 0.6:
                a.complete()
                o.copy_completed()
            acc = int(rng.integers(0, k + 1))
            assert a.commit(a.C + acc) == o.commit(o.C + acc)
            assert (a.H, a.C, a.L, a.pending) == (o.H, o.C, o.L, o.pending)
    t = svx.Tier()
    t.round(10, 15)
    for bad in (lambda: t.round(9, 15), lambda: t.commit(16), lambda: t.commit(9)):
        with pytest.raises(svx.SvxError):
            bad()


def _begin(k, c, T):
    return (k * T) // c


def _cta_of(x, c, T):
    return ((x + 1) * c - 1) // T


def test_tensor_core_work_plan_invariants(svx):
    """svx_plan_tc on seeded random launches: the grid is one CTA group per (KV head, pass of <= 64
    rows); a group's tiles are every part's tiles in order; CTA j of a group takes
    [floor(jT/c), floor((j+1)T/c)); no part spans more than 8 CTAs, and the grid is the largest
    that keeps it so within the budget."""
    rng = np.random.default_rng(5)
    for _ in range(300):
        n = int(rng.integers(1, 65))
        n_tok = [int(x) for x in rng.integers(1, int(rng.choice([300, 5000, 200000])), size=n)]
        hkv = int(rng.choice([1, 2, 4, 8, 16, 40]))
        rows = int(rng.integers(1, 257))
        budget = int(rng.choice([1, 8, 32, 100, 152]))
        pl = svx.plan_tc(n_tok, hkv, rows, budget)
        rpp = 32 if rows <= 32 else 64
        groups = hkv * -(-rows // rpp)
        nt = [-(-t // 128) for t in n_tok]
        T = sum(nt)
        assert pl["n_groups"] == groups and pl["grid"] == groups * pl["ctas_per_group"]
        assert pl["tiles_per_group"] == T and pl["tile_base"] == list(np.cumsum([0] + nt[:-1]))
        c = pl["ctas_per_group"]

        def spans(cc):
            return max(_cta_of(b + t - 1, cc, T) - _cta_of(b, cc, T) + 1 for b, t in zip(pl["tile_base"], nt))
        top = min(max(1, budget // groups), T)
        assert 1 <= c <= top and pl["slots"] == spans(c) and (c == 1 or pl["slots"] <= 8)
        assert all(spans(cc) > 8 for cc in range(c + 1, top + 1))  # the largest grid within the slot limit
        # the CTA ranges tile [0, T) exactly once, and cta_of inverts them
        ranges = [(_begin(j, c, T), _begin(j + 1, c, T)) for j in range(c)]
        assert ranges[0][0] == 0 and ranges[-1][1] == T and all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
        for j, (lo, hi) in enumerate(ranges):
            if hi > lo:
                assert _cta_of(lo, c, T) == j and _cta_of(hi - 1, c, T) == j


def test_kernel_split_arithmetic_matches_the_plan():
    """The kernel splits a group's T tiles over c CTAs in 32-bit arithmetic as begin(k) = k*q +
    floor(k*r/c) with T = q*c + r, and finds the CTA holding tile x from a float estimate corrected in
    exact steps; both must equal the host's floor(kT/c) and ((x+1)c - 1) // T."""
    rng = np.random.default_rng(6)
    for _ in range(2000):
        c = int(rng.integers(1, 153))
        T = int(rng.integers(c, 2 ** 31 - 1)) if rng.random() < 0.5 else int(rng.integers(c, 5000))
        q, r = divmod(T, c)
        dev_begin = lambda k: k * q + (k * r) // c  # noqa: E731
        for k in {0, 1, c // 2, c - 1, c}:
            assert dev_begin(k) == _begin(k, c, T)
        for x in {0, T - 1, int(rng.integers(0, T)), dev_begin(c // 2), max(0, dev_begin(c // 2) - 1)}:
            k = min(int(np.float32(x) * (np.float32(c) / np.float32(T))), c - 1)
            while k + 1 < c and dev_begin(k + 1) <= x:
                k += 1
            while k > 0 and dev_begin(k) > x:
                k -= 1
            assert k == _cta_of(x, c, T)


def test_binding_refuses_tensors_not_in_the_c_layout(svx):
    """The C calls see addresses only, so the binding checks a tensor's type, density and shape
    against the C layout before passing its address on."""
    import torch
    q = torch.zeros((2, 8, 3, 128), dtype=torch.bfloat16)
    assert svx._tensor_ptr(q, "bf16", (8, 3, 128), 2, "q") == q.data_ptr()
    assert svx._tensor_ptr(q, "bf16", (8, 3, 128), 1, "q") == q.data_ptr()  # a buffer for more requests
    assert svx._tensor_ptr(12345, "bf16", (8, 3, 128), 2, "q") == 12345      # raw addresses pass through
    lse = torch.zeros((2, 8, 3), dtype=torch.float32)
    assert svx._tensor_ptr(lse, "f32", (8, 3), 2, "lse") == lse.data_ptr()
    bad = [(q.float(), (8, 3, 128), 2),          # element type
           (q.transpose(1, 2), (3, 8, 128), 2),  # strides of a view
           (q[:, :, :2], (8, 2, 128), 2),        # a slice inside a row
           (q, (8, 3, 64), 2),                   # head dimension
           (q, (8, 3, 128), 3),                  # fewer requests than the round has
           (q[0], (8, 3, 128), 2)]               # rank
    for t, tail, lead in bad:
        with pytest.raises(svx.SvxError) as e:
            svx._tensor_ptr(t, "bf16", tail, lead, "q")
        assert e.value.status == svx.ERR_INVALID_ARG
    with pytest.raises(svx.SvxError):
        svx._dense_ptr(q.transpose(0, 1), "k_host")
    assert svx._dense_ptr(q[1], "k_host") == q[1].data_ptr()


def test_manual_completion_is_refused_while_a_library_copy_is_in_flight(svx):
    """H may advance past rows only once they are in host memory: while svx_tier_migrate's copy is
    in flight (its event set), svx_tier_complete refuses, and H stays.  The event here is a stand-in
    pointer that no CUDA call ever sees: it is cleared before the state is used any further."""
    import ctypes
    s = svx.TierState(0, 100, 104, 64, ctypes.c_void_p(1))
    assert svx.lib.svx_tier_complete(ctypes.byref(s)) == svx.ERR_BAD_STATE
    assert s.H == 0 and s.pending == 64
    s.event = None
    assert svx.lib.svx_tier_complete(ctypes.byref(s)) == svx.OK
    assert s.H == 64 and s.pending == -1


def test_binding_structs_match_the_compiled_layouts(svx):
    """Every struct the binding passes by pointer has the size the library was compiled with."""
    import ctypes
    sizes = svx.abi_sizes()
    assert set(sizes) == set(svx.ABI_STRUCTS)
    for name, size in sizes.items():
        assert ctypes.sizeof(getattr(svx, name)) == size, name
