"""Seeded synthetic workloads for chunked multi-query verification attention.

This module only draws inputs: shapes, random bf16 tensors, ragged history
lengths and random token trees.  It holds none of the attention arithmetic, so
both the CUDA path and the float64 oracle can be fed from it without sharing
any of the method's code.

Recipe (the same on every machine that has numpy >= 2):
  * every tensor has its own stream ``numpy.random.default_rng([seed, layer,
    tensor_id, request])``;
  * values are float32 standard normals (times a per-KV-head factor for keys
    where the workload asks for it, multiplied in float32) rounded to bf16 with
    round-to-nearest-even;
  * bf16 tensors are held as uint16 bit patterns (numpy has no bf16 type).

Shapes follow the verification round of "Resource-Efficient Speculative
Decoding for Long-Context LLM Serving", section 4.2: Q holds the k+1
verification queries of each request (or one query per token-tree node), the
committed history of each request is token-major ``[C_b][H_kv][d]`` (the unit
that is streamed in chunks), and the candidate KV is ``[B][n_cand][H_kv][d]``.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Optional, Sequence

import numpy as np

# tensor ids of the per-tensor random streams
_T_Q, _T_KH, _T_VH, _T_KC, _T_VC, _T_TREE, _T_LEN, _T_KSCALE = range(8)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One verification-round workload (all layers share the shape)."""

    name: str
    n_req: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    hist_len: tuple  # committed history length C_b per request
    chunk_tokens: int  # tokens per streamed chunk
    n_query: int  # k+1 verification queries, or the token-tree node count
    tree: bool = False  # token-tree candidates (else a causal chain)
    tree_max_depth: int = 5
    k_head_scale: bool = False  # keys scaled per KV head by U(0.5, 2)
    n_layers: int = 1
    seed: int = 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def n_cand(self) -> int:
        # one candidate KV entry per verification query (query j sits at
        # absolute position C_b + j)
        return self.n_query

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.head_dim))

    @property
    def hist_bytes(self) -> int:
        """bf16 K+V bytes of the committed history of one layer."""
        return 2 * 2 * self.n_kv_heads * self.head_dim * int(sum(self.hist_len))

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _ragged_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    rng = np.random.default_rng([seed, 0, _T_LEN, 0])
    return tuple(int(x) for x in rng.integers(lo, hi, size=n, endpoint=True))


def named(name: str, seed: Optional[int] = None) -> Workload:
    """The five named synthetic workloads.

    tiny      1 request, 4/1 heads, d=64, history 512 in chunks of 128, k=4.
    qwen3     Qwen3-8B-shaped layer: 8 requests, 32/8 heads, d=128, history
              32768 per request in chunks of 2048, k=4.
    internlm  InternLM2.5-7B-shaped ragged batch: 16 requests, 32/8 heads,
              d=128, history uniform in [8192, 65536], chunks of 4096, k=6,
              keys scaled per KV head by U(0.5, 2).
    tree      8 requests, 32/8 heads, d=128, history 65536 in chunks of 4096,
              16-node random token tree (depth <= 5).
    fulldepth 36 layers of the qwen3 shape, 2 requests x 131072 tokens,
              chunks of 8192, k=4.
    """
    s = {"tiny": 1, "qwen3": 2, "internlm": 3, "tree": 4, "fulldepth": 5}[name] if seed is None else seed
    if name == "tiny":
        return Workload("tiny", 1, 4, 1, 64, (512,), 128, 5, seed=s)
    if name == "qwen3":
        return Workload("qwen3", 8, 32, 8, 128, (32768,) * 8, 2048, 5, seed=s)
    if name == "internlm":
        return Workload("internlm", 16, 32, 8, 128, _ragged_lengths(16, 8192, 65536, s), 4096, 7,
                        k_head_scale=True, seed=s)
    if name == "tree":
        return Workload("tree", 8, 32, 8, 128, (65536,) * 8, 4096, 16, tree=True, seed=s)
    if name == "fulldepth":
        return Workload("fulldepth", 2, 32, 8, 128, (131072,) * 2, 8192, 5, n_layers=36, seed=s)
    raise KeyError(name)


NAMES = ("tiny", "qwen3", "internlm", "tree", "fulldepth")


# ---------------------------------------------------------------- bf16 bits

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit pattern (uint16) -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------- generators

def _normal_bf16(rng: np.random.Generator, shape, out: Optional[np.ndarray] = None,
                 scale: Optional[np.ndarray] = None, block: int = 1 << 22) -> np.ndarray:
    """Fill ``out`` (uint16, C-contiguous) with bf16 N(0,1) draws.

    ``scale`` (float32, broadcast over the last two axes [H_kv][d] by head)
    multiplies the float32 draw before rounding.  Draws are made in blocks so
    the float32 temporary stays small for multi-GiB histories.
    """
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    n = flat.size
    row = int(np.prod(shape[-2:])) if scale is not None else 1
    if scale is not None:
        per_row = np.repeat(np.asarray(scale, dtype=np.float32), shape[-1])  # [H_kv*d]
        block = max(row, (block // row) * row)
    for s0 in range(0, n, block):
        s1 = min(n, s0 + block)
        x = rng.standard_normal(s1 - s0, dtype=np.float32)
        if scale is not None:
            x = (x.reshape(-1, row) * per_row[None, :]).reshape(-1)
        flat[s0:s1] = bf16_bits(x)
    return out


def random_tree(rng: np.random.Generator, n: int, max_depth: int) -> np.ndarray:
    """Parents of an n-node token tree: node 0 is the root (parent -1); for
    i >= 1 the parent is uniform in [0, i-1], redrawn from the same stream
    while the child would sit deeper than ``max_depth``."""
    parent = np.full(n, -1, dtype=np.int32)
    depth = np.zeros(n, dtype=np.int64)
    for i in range(1, n):
        while True:
            p = int(rng.integers(0, i))
            if depth[p] + 1 <= max_depth:
                break
        parent[i] = p
        depth[i] = depth[p] + 1
    return parent


def key_head_scale(w: Workload) -> Optional[np.ndarray]:
    if not w.k_head_scale:
        return None
    rng = np.random.default_rng([w.seed, 0, _T_KSCALE, 0])
    return rng.uniform(0.5, 2.0, size=w.n_kv_heads).astype(np.float32)


def tree_parents(w: Workload) -> Optional[np.ndarray]:
    """[B][n_cand] int32 parents, or None for the causal chain."""
    if not w.tree:
        return None
    return np.stack([random_tree(np.random.default_rng([w.seed, 0, _T_TREE, b]), w.n_cand, w.tree_max_depth)
                     for b in range(w.n_req)])


Alloc = Callable[[tuple], np.ndarray]


def _np_alloc(shape) -> np.ndarray:
    return np.empty(shape, dtype=np.uint16)


@dataclasses.dataclass
class LayerInputs:
    """bf16 bit patterns of one layer's round inputs."""

    q: np.ndarray  # [B][Hq][nq][d]
    k_hist: list  # per request [C_b][H_kv][d]
    v_hist: list
    k_cand: np.ndarray  # [B][n_cand][H_kv][d]
    v_cand: np.ndarray
    parent: Optional[np.ndarray]  # [B][n_cand] int32, or None (causal chain)


def layer_inputs(w: Workload, layer: int = 0, hist_alloc: Alloc = _np_alloc,
                 requests: Optional[Sequence[int]] = None) -> LayerInputs:
    """Draw one layer's inputs.  ``hist_alloc(shape)`` provides the uint16
    storage of each request's history (e.g. a view of pinned host memory)."""
    B, Hq, Hkv, d, nq = w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query
    rs = range(B) if requests is None else requests
    ks = key_head_scale(w)
    q = _normal_bf16(np.random.default_rng([w.seed, layer, _T_Q, 0]), (B, Hq, nq, d))
    k_hist, v_hist = [], []
    for b in rs:
        C = w.hist_len[b]
        k_hist.append(_normal_bf16(np.random.default_rng([w.seed, layer, _T_KH, b]), (C, Hkv, d),
                                   out=hist_alloc((C, Hkv, d)), scale=ks))
        v_hist.append(_normal_bf16(np.random.default_rng([w.seed, layer, _T_VH, b]), (C, Hkv, d),
                                   out=hist_alloc((C, Hkv, d))))
    k_cand = _normal_bf16(np.random.default_rng([w.seed, layer, _T_KC, 0]), (B, w.n_cand, Hkv, d), scale=ks)
    v_cand = _normal_bf16(np.random.default_rng([w.seed, layer, _T_VC, 0]), (B, w.n_cand, Hkv, d))
    return LayerInputs(q, k_hist, v_hist, k_cand, v_cand, tree_parents(w))


# ---------------------------------------------------------------- fast device-side draws

def layer_inputs_device(w: Workload, layer: int, device, hist_out_k=None, hist_out_v=None):
    """Draw one layer with torch's seeded device generator (Philox) instead of numpy.

    For the multi-GiB full-depth workload, where numpy would take minutes.  Values
    are float32 standard normals (times the per-KV-head key factor) rounded to
    bf16 by torch (round-to-nearest-even), the same recipe as ``layer_inputs``
    with a different random stream.  Returns torch tensors on ``device``; if
    ``hist_out_k[b]`` / ``hist_out_v[b]`` are given (e.g. pinned host tensors of
    shape [C_b][H_kv][d], bf16) the history is written there instead and those
    tensors are returned.  Parents (token trees) come from the numpy recipe.
    """
    import torch
    B, Hq, Hkv, d, nq = w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query
    g = torch.Generator(device=device)
    ks = key_head_scale(w)
    kscale = None if ks is None else torch.from_numpy(ks).to(device).view(1, Hkv, 1)

    def draw(shape, tid, b, scale=None):
        g.manual_seed(((w.seed * 1000003 + layer) * 16 + tid) * 4099 + b)
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if scale is not None:
            x = x * scale
        return x.to(torch.bfloat16)

    q = draw((B, Hq, nq, d), _T_Q, 0)
    k_hist, v_hist = [], []
    for b in range(B):
        C = w.hist_len[b]
        kk = draw((C, Hkv, d), _T_KH, b, kscale)
        vv = draw((C, Hkv, d), _T_VH, b)
        if hist_out_k is not None:
            hist_out_k[b].copy_(kk)
            hist_out_v[b].copy_(vv)
            kk, vv = hist_out_k[b], hist_out_v[b]
        k_hist.append(kk)
        v_hist.append(vv)
    k_cand = draw((B, w.n_cand, Hkv, d), _T_KC, 0, None if kscale is None else kscale.view(1, 1, Hkv, 1))
    v_cand = draw((B, w.n_cand, Hkv, d), _T_VC, 0)
    return q, k_hist, v_hist, k_cand, v_cand, tree_parents(w)
