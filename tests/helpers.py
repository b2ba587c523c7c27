"""Shared test plumbing: seeded inputs -> torch tensors, one GPU round through the
C ABI, the oracle on the same inputs, and the parity bar.

Tolerances (written here, used by every parity test): O max abs error <= 1e-2 and
mean abs error <= 1e-3 against the float64 oracle (bf16 output); LSE relative error
<= 1e-4 (fp32 output).
"""
import numpy as np

import oracle as O
import workloads as W

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_REL = 1e-4


def bf16_tensor(bits, device=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device is not None else t


def pinned_alloc(shape):
    import torch
    return torch.empty(shape, dtype=torch.int16, pin_memory=True).numpy().view(np.uint16)


def gpu_inputs(w, layer=0, resident=False):
    """Draw one layer; history in pinned host memory (streamed) or in device memory (resident)."""
    import torch
    alloc = (lambda s: np.empty(s, dtype=np.uint16)) if resident else pinned_alloc
    x = W.layer_inputs(w, layer, hist_alloc=alloc)
    dev = torch.device("cuda")
    t = {
        "q": bf16_tensor(x.q, dev),
        "kc": bf16_tensor(x.k_cand, dev),
        "vc": bf16_tensor(x.v_cand, dev),
        "kh": [bf16_tensor(k, dev if resident else None) if k.shape[0] else None for k in x.k_hist],
        "vh": [bf16_tensor(v, dev if resident else None) if v.shape[0] else None for v in x.v_hist],
    }
    return x, t


def run_gpu(v, w, t, x, chunk_order=None, with_candidates=True, timeout_ms=60000):
    """One round through the C ABI.  The finish waits with a timeout, so it also reads the device
    error word: a kernel whose bounded wait ran out fails the test that launched it."""
    import torch
    B, Hq, nq, d = w.n_req, w.n_q_heads, w.n_query, w.head_dim
    o = torch.empty((B, Hq, nq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, nq), dtype=torch.float32, device="cuda")
    v.run_round(t["q"], w.hist_len, t["kh"], t["vh"], w.chunk_tokens, o, lse,
                cand_k=t["kc"] if with_candidates else None, cand_v=t["vc"], parent=x.parent,
                chunk_order=chunk_order, timeout_ms=timeout_ms)
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def oracle_out(w, x, rows=None, with_candidates=True):
    f = W.bf16_to_f64
    vis = O.visibility_table(w.n_req, w.n_query, x.parent)
    if not with_candidates:
        vis = np.zeros_like(vis)
    return O.verify_attention(f(x.q), [f(k) for k in x.k_hist], [f(v) for v in x.v_hist], f(x.k_cand),
                              f(x.v_cand), vis, scale=w.scale, rows=rows)


def bf16_half_ulp(x):
    """Half the spacing of bf16 values around |x| (8 significant bits): the most that rounding an
    exact value to the bf16 output can change it."""
    ax = np.abs(x)
    return np.where(ax > 0, np.exp2(np.floor(np.log2(np.where(ax > 0, ax, 1.0))) - 8), 0.0)


def check_parity(o_gpu, l_gpu, o_ref, l_ref, rows=None):
    """The bar (the stated tolerances, read for a bf16 output and an LSE that may sit near zero):
    - O mean: mean |O - O_ref| <= 1e-3 on the raw error.  Rounding the exact value to bf16 averages
      about a quarter of a bf16 ulp, far under 1e-3 where |O| < 1, so this bar sees any systematic
      error above that;
    - O max: the error beyond the output format's own rounding, max(0, |O - O_ref| - half a bf16 ulp
      at |O_ref|), is <= 1e-2.  No bf16 output can meet an absolute 1e-2 on |O| >= 4 (the rounding
      alone can be 0.0156), and rows with few visible keys reach such values;
    - LSE: |LSE - LSE_ref| <= 1e-4 * max(|LSE_ref|, 1), i.e. relative, except that near LSE = 0
      (a handful of keys) it is absolute;
    - LSE finiteness (no visible key: -inf) matches exactly."""
    if rows is not None:
        idx = tuple(np.array(rows).T)
        o_gpu, l_gpu, o_ref, l_ref = o_gpu[idx], l_gpu[idx], o_ref[idx], l_ref[idx]
    raw = np.abs(o_gpu - o_ref)
    err = np.maximum(raw - bf16_half_ulp(o_ref), 0.0)
    fin = np.isfinite(l_ref)
    rel = np.abs(l_gpu[fin] - l_ref[fin]) / np.maximum(np.abs(l_ref[fin]), 1.0)
    assert np.array_equal(np.isfinite(l_gpu), fin), "LSE finiteness differs"
    assert err.max() <= O_MAX_ABS, f"O max abs err beyond bf16 rounding {err.max():.3e}"
    assert raw.mean() <= O_MEAN_ABS, f"O mean abs err {raw.mean():.3e}"
    if rel.size:
        assert rel.max() <= LSE_REL, f"LSE err {rel.max():.3e} (relative to max(|LSE|, 1))"
    return float(err.max()), float(raw.mean()), float(rel.max()) if rel.size else 0.0


def sample_rows(w, n, seed=0):
    """About n random (request, q-head, query) rows, plus the first and the last."""
    rng = np.random.default_rng(seed)
    rows = {(int(rng.integers(0, w.n_req)), int(rng.integers(0, w.n_q_heads)), int(rng.integers(0, w.n_query)))
            for _ in range(n)}
    rows |= {(w.n_req - 1, w.n_q_heads - 1, w.n_query - 1), (0, 0, 0)}
    return sorted(rows)


def oracle_pair(args):
    """Oracle rows of one (request, KV head) pair: all G * nq query rows of that KV head.  A top-level
    function, so that a spawn process pool can run pairs in parallel."""
    import oracle
    q, kh, vh, kc, vc, vis, scale = args
    f = W.bf16_to_f64
    return oracle.verify_attention(f(q), [f(kh)], [f(vh)], f(kc), f(vc), vis, scale=scale)


def oracle_all_rows_parallel(w, x, processes=None):
    """Every row of one layer from the oracle, one (request, KV head) pair per task on a spawn pool (a
    forked pool could inherit a CUDA context).  Returns O [B][Hq][nq][d] and LSE [B][Hq][nq]."""
    import multiprocessing as mp
    import os
    vis = O.visibility_table(w.n_req, w.n_query, x.parent)
    G = w.group
    tasks, keys = [], []
    for b in range(w.n_req):
        for g in range(w.n_kv_heads):
            tasks.append((x.q[b:b + 1, g * G:(g + 1) * G], x.k_hist[b][:, g:g + 1], x.v_hist[b][:, g:g + 1],
                          x.k_cand[b:b + 1, :, g:g + 1], x.v_cand[b:b + 1, :, g:g + 1], vis[b:b + 1], w.scale))
            keys.append((b, g))
    o_ref = np.full((w.n_req, w.n_q_heads, w.n_query, w.head_dim), np.nan)
    l_ref = np.full((w.n_req, w.n_q_heads, w.n_query), np.nan)
    with mp.get_context("spawn").Pool(processes or os.cpu_count() or 1) as pool:
        for (b, g), (o, lse) in zip(keys, pool.imap(oracle_pair, tasks)):
            o_ref[b, g * G:(g + 1) * G] = o[0]
            l_ref[b, g * G:(g + 1) * G] = lse[0]
    return o_ref, l_ref
