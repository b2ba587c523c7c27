"""Float64 CPU oracle for chunked multi-query verification attention.

TEST INFRASTRUCTURE.  This is a plain, slow, obviously correct statement of
what the verification round computes.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; the product path never calls it.
It shares no code with the CUDA library.

Source: "Resource-Efficient Speculative Decoding for Long-Context LLM
Serving" (SpecStream), section 4.2 "KV Streaming for Multi-Query
Verification", Eqs. (6)-(9), and section 4.1 Eq. (4) for the KV regions.

Readings where the page is silent (each is also listed in the design notes):
  * k draft tokens give k+1 verification queries and k+1 candidate KV entries;
    query j sits at absolute position C_b + j (section 2.2: tokens whose KV is
    not yet computed lie past the committed boundary C_r).
  * Query j sees candidate j itself (section 4.2 only excludes *subsequent*
    candidates); in a token tree it sees itself and its ancestors.
  * All committed history [0, C_b) is visible to every query (section 4.2,
    "Chunked verification shared across queries").
  * Grouped-query attention maps query head h to KV head floor(h / G) (the
    page never mentions GQA; contiguous grouping is the plain reading).
  * Default scale 1/sqrt(d_h) (Eq. 6); natural exponent and natural-log LSE
    (Eqs. 7-8).

Pins (what fixes this code to something other than itself) live in
``tests/test_oracle_pins.py``: high-precision brute force, a library SDPA,
closed forms (equal keys, zero query, a 3:1 two-key case), the chunked =
full invariant (Eq. 9) over chunk sizes and orders, k=0 decode, causality by
perturbation, the printed block-causal mask example and graph-library tree
ancestry.
"""
from __future__ import annotations

from typing import Iterable, Optional, Sequence

import numpy as np

# ------------------------------------------------------------------ masks


def candidate_visibility(n_query: int, parent: Optional[Sequence[int]] = None) -> np.ndarray:
    """Visibility words of the candidate region for one request.

    Returns uint32[n_query]; bit i of word j is set iff query j may attend to
    candidate i.  Chain (``parent is None``): i <= j, the causal mask by
    absolute position of section 4.2.  Tree: i == j or i is an ancestor of j
    (token-tree verification).  Candidates are limited to 32 per request.
    """
    if n_query > 32:
        raise ValueError("at most 32 candidates per request")
    if parent is not None:
        if len(parent) != n_query or (n_query and int(parent[0]) != -1):
            raise ValueError("parent[0] must be -1 (the root)")
        for i in range(1, n_query):
            if not 0 <= int(parent[i]) < i:
                raise ValueError("parent[i] must lie in [0, i-1]")
    words = np.zeros(n_query, dtype=np.uint32)
    for j in range(n_query):
        w = 0
        if parent is None:
            for i in range(j + 1):
                w |= 1 << i
        else:
            node = j  # walk from j up to the root: j and all its ancestors
            while node >= 0:
                w |= 1 << node
                node = int(parent[node])
        words[j] = w
    return words


def visibility_table(n_req: int, n_query: int, parents: Optional[np.ndarray]) -> np.ndarray:
    """uint32[n_req][n_query]: candidate_visibility for every request."""
    return np.stack([candidate_visibility(n_query, None if parents is None else parents[b])
                     for b in range(n_req)]) if n_req else np.zeros((0, n_query), np.uint32)


# ------------------------------------------------------------------ chunk plan


def cohort_chunk_plan(hist_len: Sequence[int], chunk_tokens: int, n_slots: int) -> list:
    """Cohort chunk plan of a round (section 4.2, "Pipelined KV transfers"
    and "Cohort batching").

    The Sealed History of each request is cut into contiguous chunks of
    ``chunk_tokens`` along token positions.  Cohort chunk j holds, for every
    request b whose history reaches past j*c, the part
    (b, t0=j*c, n=min(c, C_b - t0)); it is staged in buffer j mod n_slots.
    Returns a list of (j, slot, b, t0, n) tuples in (j, b) order.
    """
    plan = []
    j = 0
    while True:
        t0 = j * chunk_tokens
        parts = [(j, j % n_slots, b, t0, min(chunk_tokens, int(C) - t0))
                 for b, C in enumerate(hist_len) if int(C) > t0]
        if not parts:
            return plan
        plan.extend(parts)
        j += 1


def covers_exactly_once(hist_len: Sequence[int], parts: Iterable[tuple]) -> bool:
    """True iff the (b, t0, n) parts tile every [0, C_b) exactly once
    (each history token enters the reduction once, Eq. (9))."""
    count = [np.zeros(int(C), dtype=np.int64) for C in hist_len]
    for b, t0, n in parts:
        if b < 0 or b >= len(hist_len) or n <= 0 or t0 < 0 or t0 + n > int(hist_len[b]):
            return False
        count[b][t0:t0 + n] += 1
    return all(bool(np.all(c == 1)) for c in count)


# ------------------------------------------------------------------ attention


def _visible_keys(k_hist_b, v_hist_b, k_cand_b, v_cand_b, g, vis_word, n_cand):
    """Gather the KV rows visible to one query of KV head g: the whole
    history plus the candidates whose visibility bit is set."""
    cand = [i for i in range(n_cand) if (int(vis_word) >> i) & 1]
    K = np.concatenate([k_hist_b[:, g, :], k_cand_b[cand, g, :]], axis=0)
    V = np.concatenate([v_hist_b[:, g, :], v_cand_b[cand, g, :]], axis=0)
    return K, V


def verify_attention(q, k_hist, v_hist, k_cand, v_cand, vis, scale: Optional[float] = None,
                     rows: Optional[Sequence[tuple]] = None):
    """Full attention of every verification query over its visible KV, Eq. (6).

    q       float64 [B][Hq][nq][d]
    k_hist  list over requests of float64 [C_b][H_kv][d] (committed history)
    v_hist  same
    k_cand  float64 [B][n_cand][H_kv][d] (GPU-resident candidate region)
    v_cand  same
    vis     uint32 [B][nq] candidate visibility words
    rows    optional list of (b, h, j); default all rows

    Returns (O float64 [B][Hq][nq][d], LSE float64 [B][Hq][nq]); rows not
    asked for are NaN.  Per row, two passes: M = max s, LSE = M + ln sum
    exp(s - M), O = sum exp(s - LSE) v  (Eq. 9 with the denominator over all
    visible positions).
    """
    B, Hq, nq, d = q.shape
    Hkv = k_cand.shape[2]
    n_cand = k_cand.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    O = np.full((B, Hq, nq, d), np.nan)
    LSE = np.full((B, Hq, nq), np.nan)
    if rows is None:
        rows = [(b, h, j) for b in range(B) for h in range(Hq) for j in range(nq)]
    for b, h, j in rows:
        g = h // G
        K, V = _visible_keys(k_hist[b], v_hist[b], k_cand[b], v_cand[b], g, vis[b][j], n_cand)
        s = (K @ q[b, h, j]) * scale
        M = np.max(s)
        lse = M + np.log(np.sum(np.exp(s - M)))
        O[b, h, j] = np.exp(s - lse) @ V
        LSE[b, h, j] = lse
    return O, LSE


def _chunk_state(S, V, visible):
    """Eq. (7): chunk-local (m_j, l_j, a_j) over the visible positions of
    each query row.  A row with no visible position gets (-inf, 0, 0)."""
    S = np.where(visible, S, -np.inf)
    mj = S.max(axis=1) if S.shape[1] else np.full(S.shape[0], -np.inf)
    E = np.zeros_like(S)
    ok = np.isfinite(mj)
    E[ok] = np.exp(S[ok] - mj[ok, None])
    return mj, E.sum(axis=1), E @ V


def _merge_state(m, l, a, mj, lj, aj):
    """Eq. (8): m' = max(m, m_j), alpha = e^(m - m'), beta = e^(m_j - m'),
    l' = alpha l + beta l_j, a' = alpha a + beta a_j.  Where both maxima are
    -inf the row is still empty: alpha = beta = 0 keeps (-inf, 0, 0)."""
    mn = np.maximum(m, mj)
    alpha = np.zeros_like(m)
    beta = np.zeros_like(m)
    ok = np.isfinite(mn)
    alpha[ok] = np.exp(m[ok] - mn[ok])
    beta[ok] = np.exp(mj[ok] - mn[ok])
    return mn, alpha * l + beta * lj, alpha[:, None] * a + beta[:, None] * aj


def verify_attention_streamed(q, k_hist, v_hist, k_cand, v_cand, vis, chunk_tokens: int,
                              scale: Optional[float] = None, chunk_order: Optional[Sequence[int]] = None):
    """The same result by the streaming recurrence of section 4.2.

    State (m, l, a) per query and head starts at (-inf, 0, 0).  Each history
    chunk (K_j, V_j) serves all queries of the request: its local state
    (Eq. 7) is merged into the running state by the rescale of Eq. (8).  The
    GPU-resident candidate region follows under the visibility mask, and
    finally O = a / l and LSE = m + ln l (Eq. 9).  ``chunk_order`` permutes
    the history chunks.
    """
    B, Hq, nq, d = q.shape
    Hkv = k_cand.shape[2]
    n_cand = k_cand.shape[1]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    O = np.zeros((B, Hq, nq, d))
    LSE = np.zeros((B, Hq, nq))
    for b in range(B):
        C = k_hist[b].shape[0]
        n_chunks = -(-C // chunk_tokens)
        order = range(n_chunks) if chunk_order is None else [c for c in chunk_order if c < n_chunks]
        cand_visible = np.array([[(int(vis[b][j]) >> i) & 1 == 1 for i in range(n_cand)]
                                 for j in range(nq)], dtype=bool).reshape(nq, n_cand)
        for h in range(Hq):
            g = h // G
            m, l, a = np.full(nq, -np.inf), np.zeros(nq), np.zeros((nq, d))
            for c in order:
                t0, t1 = c * chunk_tokens, min(C, (c + 1) * chunk_tokens)
                S = (q[b, h] @ k_hist[b][t0:t1, g, :].T) * scale
                m, l, a = _merge_state(m, l, a, *_chunk_state(S, v_hist[b][t0:t1, g, :],
                                                              np.ones_like(S, dtype=bool)))
            S = (q[b, h] @ k_cand[b][:, g, :].T) * scale
            m, l, a = _merge_state(m, l, a, *_chunk_state(S, v_cand[b][:, g, :], cand_visible))
            O[b, h] = a / l[:, None]
            LSE[b, h] = m + np.log(l)
    return O, LSE


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> nearest bf16 value (ties to even), returned as float64.

    Used where the tests compare a bf16 output: the oracle's float64 value is
    rounded once, the way the round's output tensor is defined."""
    f = np.asarray(x, dtype=np.float64)
    # exact: split by frexp so the rounding happens on the float64 itself
    m, e = np.frexp(f)  # f = m * 2**e, 0.5 <= |m| < 1
    scaled = np.ldexp(m, 8)  # 8 significant bits (bf16 has 7 stored + 1 implicit)
    r = np.round(scaled)  # numpy rounds half to even
    return np.ldexp(r, e - 8)
