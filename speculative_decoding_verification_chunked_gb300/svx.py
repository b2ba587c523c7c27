"""Python binding of the svx C ABI (``include/svx.h``): argument marshalling only.

Every step of the verification round runs in the CUDA library; this module
turns torch tensors and Python sequences into the pointers and sizes the C
calls take.  Importing it loads ``libsvx.so`` and fails loudly if the library
has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

# SVX_LIBRARY=checked loads the bounds-checked build (libsvx_checked.so) instead of libsvx.so.
_LIB_NAME = {"": "libsvx.so", "checked": "libsvx_checked.so"}.get(os.environ.get("SVX_LIBRARY", ""))
if _LIB_NAME is None:
    raise ImportError(f"SVX_LIBRARY={os.environ['SVX_LIBRARY']!r}: expected unset or 'checked'")
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), _LIB_NAME)

OK, ERR_INVALID_ARG, ERR_BAD_STATE, ERR_OOM, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED = range(7)
STATUS_NAMES = {0: "SVX_OK", 1: "SVX_ERR_INVALID_ARG", 2: "SVX_ERR_BAD_STATE", 3: "SVX_ERR_OOM",
                4: "SVX_ERR_CUDA", 5: "SVX_ERR_TIMEOUT", 6: "SVX_ERR_UNSUPPORTED"}
FLAG_TIMING = 1
FLAG_NO_TENSOR_CORES = 2
FLAG_ZERO_COPY = 4
FLAG_ADAPTIVE = 8


class SvxError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


class Config(ctypes.Structure):
    _fields_ = [("max_req", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("max_query", ctypes.c_int32), ("max_chunk_tokens", ctypes.c_int32),
                ("n_slots", ctypes.c_int32), ("device", ctypes.c_int32), ("compute_stream", ctypes.c_void_p),
                ("copy_stream", ctypes.c_void_p), ("flags", ctypes.c_uint32), ("zero_copy_ctas", ctypes.c_int32),
                ("staged_ctas", ctypes.c_int32)]


class Part(ctypes.Structure):
    _fields_ = [("req", ctypes.c_int32), ("n_tok", ctypes.c_int32), ("tok_start", ctypes.c_int64),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p)]


class Stats(ctypes.Structure):
    _fields_ = [("round_ms", ctypes.c_double), ("copy_busy_ms", ctypes.c_double),
                ("chunk_kernel_ms", ctypes.c_double), ("cand_kernel_ms", ctypes.c_double),
                ("finish_kernel_ms", ctypes.c_double), ("h2d_bytes", ctypes.c_int64),
                ("device_bytes", ctypes.c_int64), ("n_chunk_launches", ctypes.c_int32),
                ("n_copies", ctypes.c_int32), ("chunk_kernel_exposed_ms", ctypes.c_double),
                ("transfer_busy_ms", ctypes.c_double), ("n_zero_copy_pushes", ctypes.c_int32)]


class WindowStats(ctypes.Structure):
    _fields_ = [("window_ms", ctypes.c_double), ("copy_busy_ms", ctypes.c_double), ("copy_gap_ms", ctypes.c_double),
                ("chunk_kernel_ms", ctypes.c_double), ("chunk_kernel_exposed_ms", ctypes.c_double),
                ("finish_kernel_ms", ctypes.c_double), ("transfer_busy_ms", ctypes.c_double),
                ("zero_copy_kernel_ms", ctypes.c_double), ("n_zero_copy_pushes", ctypes.c_int32), ("pad", ctypes.c_int32),
                ("h2d_bytes", ctypes.c_int64), ("device_bytes", ctypes.c_int64), ("n_rounds", ctypes.c_int32), ("n_pushes", ctypes.c_int32), ("n_chunk_launches", ctypes.c_int32),
                ("n_copies", ctypes.c_int32)]


class TierState(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int64), ("C", ctypes.c_int64), ("L", ctypes.c_int64), ("pending", ctypes.c_int64),
                ("event", ctypes.c_void_p)]


class SchedConfig(ctypes.Structure):
    _fields_ = [("eps_target", ctypes.c_double), ("delta", ctypes.c_double), ("ema", ctypes.c_double),
                ("t_draft", ctypes.c_double), ("delta_target", ctypes.c_double), ("alloc", ctypes.c_int32)]


class DraftInstr(ctypes.Structure):
    _fields_ = [("req", ctypes.c_int64), ("round", ctypes.c_int64), ("seq", ctypes.c_int64),
                ("alloc", ctypes.c_int32), ("t_latest", ctypes.c_double)]


class PlanEntry(ctypes.Structure):
    _fields_ = [("chunk", ctypes.c_int32), ("slot", ctypes.c_int32), ("req", ctypes.c_int32),
                ("n_tok", ctypes.c_int32), ("tok_start", ctypes.c_int64)]


# name -> (restype, argtypes); every symbol declared in include/svx.h
_P = ctypes.c_void_p
_SIGS = {
    "svx_create": (ctypes.c_int, [ctypes.POINTER(Config), ctypes.POINTER(_P)]),
    "svx_destroy": (ctypes.c_int, [_P]),
    "svx_round_begin": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int32, _P, ctypes.POINTER(ctypes.c_int64),
                                       ctypes.c_float]),
    "svx_push_chunk": (ctypes.c_int, [_P, ctypes.POINTER(Part), ctypes.c_int32]),
    "svx_candidate_attn": (ctypes.c_int, [_P, _P, _P, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "svx_round_finish": (ctypes.c_int, [_P, _P, _P, ctypes.c_int32]),
    "svx_last_error": (ctypes.c_char_p, [_P]),
    "svx_round_stats": (ctypes.c_int, [_P, ctypes.POINTER(Stats)]),
    "svx_window_rounds": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_double), ctypes.c_int64,
                                         ctypes.POINTER(ctypes.c_int64)]),
    "svx_adaptive_state": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(ctypes.c_int32)]),
    "svx_window_reset": (ctypes.c_int, [_P]),
    "svx_window_stats": (ctypes.c_int, [_P, ctypes.POINTER(WindowStats)]),
    "svx_window_intervals": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_double), ctypes.c_int64,
                                            ctypes.POINTER(ctypes.c_int64)]),
    "svx_plan_chunks": (ctypes.c_int, [ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), ctypes.c_int32,
                                       ctypes.c_int32, ctypes.POINTER(PlanEntry), ctypes.c_int64,
                                       ctypes.POINTER(ctypes.c_int64)]),
    "svx_candidate_masks": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                                           ctypes.POINTER(ctypes.c_uint32)]),
    "svx_check_coverage": (ctypes.c_int, [ctypes.c_int32, ctypes.POINTER(ctypes.c_int64),
                                          ctypes.POINTER(ctypes.c_int64), ctypes.c_int64,
                                          ctypes.POINTER(ctypes.c_int32)]),
    "svx_debug_expire_wait": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    "svx_debug_fail_copy": (ctypes.c_int, [_P, ctypes.c_int64]),
    "svx_debug_delay_copy": (ctypes.c_int, [_P, ctypes.c_int64, ctypes.c_int32]),
    "svx_debug_clip_q_rows": (ctypes.c_int, [_P, ctypes.c_int64]),
    "svx_plan_tc": (ctypes.c_int, [ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32, ctypes.c_int32,
                                   ctypes.c_int64, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32),
                                   ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64),
                                   ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)]),
    "svx_verify_static": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, _P, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(_P),
                                         ctypes.POINTER(_P), _P, _P, ctypes.POINTER(ctypes.c_int32), ctypes.c_float,
                                         _P, _P, _P]),
    "svx_static_check": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32)]),
    "svx_migration_endpoint": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                              ctypes.POINTER(ctypes.c_int64)]),
    "svx_tier_round": (ctypes.c_int, [ctypes.POINTER(TierState), ctypes.c_int64, ctypes.c_int64]),
    "svx_tier_plan": (ctypes.c_int, [ctypes.POINTER(TierState), ctypes.c_int64, ctypes.c_int64,
                                     ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
    "svx_tier_complete": (ctypes.c_int, [ctypes.POINTER(TierState)]),
    "svx_tier_commit": (ctypes.c_int, [ctypes.POINTER(TierState), ctypes.c_int64, ctypes.POINTER(ctypes.c_int64),
                                       ctypes.POINTER(ctypes.c_int64)]),
    "svx_tier_migrate": (ctypes.c_int, [ctypes.POINTER(TierState), ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                        _P, _P, _P, _P, _P, ctypes.POINTER(ctypes.c_int64)]),
    "svx_tier_poll": (ctypes.c_int, [ctypes.POINTER(TierState), ctypes.POINTER(ctypes.c_int32)]),
    "svx_tier_release": (ctypes.c_int, [ctypes.POINTER(TierState)]),
    "svx_sched_create": (ctypes.c_int, [ctypes.POINTER(SchedConfig), ctypes.POINTER(_P)]),
    "svx_sched_destroy": (ctypes.c_int, [_P]),
    "svx_sched_new_round": (ctypes.c_int, [_P]),
    "svx_sched_try_admit": (ctypes.c_int, [_P, ctypes.c_int64, ctypes.c_int64, ctypes.c_double, ctypes.c_double,
                                           ctypes.POINTER(DraftInstr), ctypes.POINTER(ctypes.c_int32)]),
    "svx_sched_check_start": (ctypes.c_int, [_P, ctypes.POINTER(DraftInstr), ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_double, ctypes.POINTER(ctypes.c_int32)]),
    "svx_sched_ack": (ctypes.c_int, [_P, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                                     ctypes.POINTER(ctypes.c_int32)]),
    "svx_sched_observe_target": (ctypes.c_int, [_P, ctypes.c_double, ctypes.c_double]),
    "svx_sched_estimates": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_int32)]),
    "svx_width_create": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32), ctypes.c_int32, ctypes.c_double,
                                        ctypes.c_double, ctypes.c_int32, ctypes.POINTER(_P)]),
    "svx_width_destroy": (ctypes.c_int, [_P]),
    "svx_width_record": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                        ctypes.c_double, ctypes.c_double]),
    "svx_width_next": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int32)]),
    "svx_width_cost": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.POINTER(ctypes.c_double)]),
    "svx_version": (ctypes.c_char_p, []),
    "svx_abi_sizes": (ctypes.c_int32, [ctypes.POINTER(ctypes.c_int64), ctypes.c_int32]),
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"CUDA library not built: {_LIB_PATH} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()
SYMBOLS = tuple(_SIGS)


def version() -> str:
    return lib.svx_version().decode()


ABI_STRUCTS = ("Config", "Part", "Stats", "WindowStats", "PlanEntry", "TierState", "SchedConfig", "DraftInstr")


def abi_sizes() -> dict:
    """sizeof of each C ABI struct as the library was compiled, keyed by the binding's class name."""
    out = (ctypes.c_int64 * len(ABI_STRUCTS))()
    n = lib.svx_abi_sizes(out, len(ABI_STRUCTS))
    return dict(zip(ABI_STRUCTS, list(out[:min(n, len(ABI_STRUCTS))])))


def _i64(seq) -> ctypes.Array:
    a = np.ascontiguousarray(np.asarray(seq, dtype=np.int64))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


# ------------------------------------------------------------ host-only bookkeeping


def plan_chunks(hist_len: Sequence[int], chunk_tokens: int, n_slots: int) -> list:
    """Cohort chunk plan as (chunk, slot, req, tok_start, n_tok) tuples."""
    h, hp = _i64(hist_len)
    n = ctypes.c_int64(0)
    st = lib.svx_plan_chunks(len(h), hp, chunk_tokens, n_slots, None, 0, ctypes.byref(n))
    if st != OK:
        raise SvxError(st, "svx_plan_chunks: invalid arguments")
    buf = (PlanEntry * max(1, n.value))()
    st = lib.svx_plan_chunks(len(h), hp, chunk_tokens, n_slots, buf, n.value, ctypes.byref(n))
    if st != OK:
        raise SvxError(st, "svx_plan_chunks: invalid arguments")
    return [(e.chunk, e.slot, e.req, e.tok_start, e.n_tok) for e in buf[:n.value]]


def candidate_masks(n_req: int, n_query: int, parent: Optional[np.ndarray] = None) -> np.ndarray:
    out = np.zeros((n_req, n_query), dtype=np.uint32)
    par = None
    if parent is not None:
        parent = np.ascontiguousarray(np.asarray(parent, dtype=np.int32).reshape(n_req, n_query))
        par = parent.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    st = lib.svx_candidate_masks(n_req, n_query, par, out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32)))
    if st != OK:
        raise SvxError(st, "svx_candidate_masks: invalid tree or sizes")
    return out


def plan_tc(n_tok: Sequence[int], n_kv_heads: int, rows: int, cta_budget: int) -> dict:
    """Work plan of one tensor-core chunk launch (see svx_plan_tc): grid, n_groups, ctas_per_group,
    tiles_per_group, slots and tile_base (per part)."""
    n = len(n_tok)
    nt = (ctypes.c_int32 * max(1, n))(*[int(x) for x in n_tok])
    grid, tpg, = ctypes.c_int64(0), ctypes.c_int64(0)
    ng, cpg, sl = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    tb = (ctypes.c_int64 * max(1, n))()
    st = lib.svx_plan_tc(n, nt, n_kv_heads, rows, cta_budget, ctypes.byref(grid), ctypes.byref(ng), ctypes.byref(cpg),
                         ctypes.byref(tpg), ctypes.byref(sl), tb)
    if st != OK:
        raise SvxError(st, "svx_plan_tc: invalid arguments")
    return {"grid": grid.value, "n_groups": ng.value, "ctas_per_group": cpg.value, "tiles_per_group": tpg.value,
            "slots": sl.value, "tile_base": list(tb[:n])}


def check_coverage(hist_len: Sequence[int], parts: Sequence[tuple]) -> bool:
    """parts: (req, tok_start, n_tok) triples."""
    h, hp = _i64(hist_len)
    p, pp = _i64(np.asarray(parts, dtype=np.int64).reshape(-1, 3) if len(parts) else np.zeros((0, 3)))
    ok = ctypes.c_int32(-1)
    st = lib.svx_check_coverage(len(h), hp, pp, len(parts), ctypes.byref(ok))
    if st != OK:
        raise SvxError(st, "svx_check_coverage: invalid arguments")
    return bool(ok.value)


# ------------------------------------------------------------ commit-aware tiering


def migration_endpoint(H: int, C: int, T: int, g: int) -> int:
    E = ctypes.c_int64(0)
    st = lib.svx_migration_endpoint(H, C, T, g, ctypes.byref(E))
    if st != OK:
        raise SvxError(st, "svx_migration_endpoint: invalid arguments")
    return E.value


class Tier:
    """One request's Sealed History / Active Tail / Speculative Frontier boundaries."""

    def __init__(self, H: int = 0, C: int = 0, L: int = 0):
        self.s = TierState(H, C, L, -1, None)

    def _call(self, fn, *args):
        st = fn(ctypes.byref(self.s), *args)
        if st != OK:
            raise SvxError(st, fn.__name__)

    @property
    def H(self):
        return self.s.H

    @property
    def C(self):
        return self.s.C

    @property
    def L(self):
        return self.s.L

    @property
    def pending(self):
        return None if self.s.pending < 0 else self.s.pending

    def round(self, C: int, L: int):
        self._call(lib.svx_tier_round, C, L)

    def plan(self, T: int, g: int):
        b, e = ctypes.c_int64(0), ctypes.c_int64(0)
        self._call(lib.svx_tier_plan, T, g, ctypes.byref(b), ctypes.byref(e))
        return (b.value, e.value) if e.value > b.value else None

    def complete(self):
        self._call(lib.svx_tier_complete)

    def commit(self, C_new: int):
        b, e = ctypes.c_int64(0), ctypes.c_int64(0)
        self._call(lib.svx_tier_commit, C_new, ctypes.byref(b), ctypes.byref(e))
        return b.value, e.value

    def migrate(self, T: int, g: int, row_bytes: int, k_dev_at_H, v_dev_at_H, k_host, v_host, stream=None) -> int:
        E = ctypes.c_int64(0)
        ptrs = [_dense_ptr(t, what) for t, what in ((k_dev_at_H, "k_dev_at_H"), (v_dev_at_H, "v_dev_at_H"),
                                                     (k_host, "k_host"), (v_host, "v_host"))]
        self._call(lib.svx_tier_migrate, T, g, row_bytes, *ptrs, _stream_handle(stream), ctypes.byref(E))
        return E.value

    def poll(self) -> bool:
        d = ctypes.c_int32(0)
        self._call(lib.svx_tier_poll, ctypes.byref(d))
        return bool(d.value)

    def release(self):
        self._call(lib.svx_tier_release)


# ------------------------------------------------------------ Target-priority admission


class Scheduler:
    """Host-side Draft admission (svx_sched_*)."""

    def __init__(self, eps_target: float, delta: float, ema: float, t_draft: float, delta_target: float,
                 alloc: int = 0):
        self._h = ctypes.c_void_p(None)
        st = lib.svx_sched_create(ctypes.byref(SchedConfig(eps_target, delta, ema, t_draft, delta_target, alloc)),
                                  ctypes.byref(self._h))
        if st != OK:
            raise SvxError(st, "svx_sched_create: invalid configuration")

    def __del__(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib.svx_sched_destroy(self._h)
            self._h = ctypes.c_void_p(None)

    def new_round(self):
        lib.svx_sched_new_round(self._h)

    def try_admit(self, req: int, rnd: int, now: float, window: float) -> Optional[DraftInstr]:
        ins, ok = DraftInstr(), ctypes.c_int32(0)
        st = lib.svx_sched_try_admit(self._h, req, rnd, now, window, ctypes.byref(ins), ctypes.byref(ok))
        if st != OK:
            raise SvxError(st, "svx_sched_try_admit")
        return ins if ok.value else None

    def check_start(self, ins: DraftInstr, cur_req: int, cur_round: int, now: float) -> bool:
        ok = ctypes.c_int32(0)
        lib.svx_sched_check_start(self._h, ctypes.byref(ins), cur_req, cur_round, now, ctypes.byref(ok))
        return bool(ok.value)

    def ack(self, req: int, seq: int, t_obs: float) -> bool:
        ok = ctypes.c_int32(0)
        lib.svx_sched_ack(self._h, req, seq, t_obs, ctypes.byref(ok))
        return bool(ok.value)

    def observe_target(self, t_co: float, t_alone: float):
        st = lib.svx_sched_observe_target(self._h, t_co, t_alone)
        if st != OK:
            raise SvxError(st, "svx_sched_observe_target")

    def estimates(self):
        a, b, c = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_int32(0)
        lib.svx_sched_estimates(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
        return a.value, b.value, bool(c.value)


# ------------------------------------------------------------ dynamic verification width


class WidthController:
    """svx_width_*: argmin_q T_round_hat(q) / U_hat(q) with initial sampling and a switching threshold."""

    def __init__(self, widths: Sequence[int], ema: float, threshold: float, n_init: int):
        arr = (ctypes.c_int32 * len(widths))(*widths)
        self._h = ctypes.c_void_p(None)
        st = lib.svx_width_create(arr, len(widths), ema, threshold, n_init, ctypes.byref(self._h))
        if st != OK:
            raise SvxError(st, "svx_width_create: invalid configuration")

    def __del__(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib.svx_width_destroy(self._h)
            self._h = ctypes.c_void_p(None)

    def record(self, q: int, t_draft: float, t_h2d: float, t_attn: float, t_correct: float, committed: float):
        st = lib.svx_width_record(self._h, q, t_draft, t_h2d, t_attn, t_correct, committed)
        if st != OK:
            raise SvxError(st, "svx_width_record: unknown width")

    def next_width(self) -> int:
        q = ctypes.c_int32(0)
        lib.svx_width_next(self._h, ctypes.byref(q))
        return q.value

    def cost(self, q: int) -> Optional[float]:
        c = ctypes.c_double(0)
        st = lib.svx_width_cost(self._h, q, ctypes.byref(c))
        if st != OK:
            raise SvxError(st, "svx_width_cost: unknown width")
        return None if c.value < 0 else c.value


# ------------------------------------------------------------ a round that allocates nothing


STATIC_SCRATCH_BYTES = 32 << 20


def static_check() -> bool:
    """svx_static_check: True if a kernel of some static round since the last check gave up a
    bounded wait (that round's outputs are invalid); clears the flag.  Synchronises the device."""
    e = ctypes.c_int32(0)
    st = lib.svx_static_check(ctypes.byref(e))
    if st != OK:
        raise SvxError(st, lib.svx_last_error(None).decode())
    return bool(e.value)


def verify_static(q, hist_len: Sequence[int], hist_k: Sequence, hist_v: Sequence, o, lse, cand_k=None, cand_v=None,
                  parent: Optional[np.ndarray] = None, scale: float = 0.0, stream=None,
                  n_kv_heads: Optional[int] = None):
    """svx_verify_static: a whole round over device-resident KV using the library's static device
    scratch instead of any allocation (for callers that cannot call cudaMalloc).

    q: device bf16 [B][Hq][nq][d]; hist_k[b], hist_v[b]: device bf16 [C_b][Hkv][d] (or None when
    C_b = 0); cand_k, cand_v: device bf16 [B][nq][Hkv][d] or None; o, lse: device outputs.
    """
    B, Hq, nq, d = (int(x) for x in q.shape)
    if len(hist_len) != B or len(hist_k) != B or len(hist_v) != B:
        raise SvxError(ERR_INVALID_ARG, f"hist_len, hist_k and hist_v need one entry per request ({B})")
    if n_kv_heads is None:
        src = next((k for k in hist_k if k is not None), cand_k)
        if src is None:
            raise SvxError(ERR_INVALID_ARG, "n_kv_heads is required when no history or candidate tensor is given")
        n_kv_heads = int(src.shape[-2])
    h, hp = _i64(hist_len)
    qp = _tensor_ptr(q, "bf16", (Hq, nq, d), B, "q")
    kv = (n_kv_heads, d)
    ks = (_P * B)(*[None if k is None else _tensor_ptr(k, "bf16", kv, int(C), f"history k of request {b}")
                    for b, (k, C) in enumerate(zip(hist_k, hist_len))])
    vs = (_P * B)(*[None if v is None else _tensor_ptr(v, "bf16", kv, int(C), f"history v of request {b}")
                    for b, (v, C) in enumerate(zip(hist_v, hist_len))])
    ckp = None if cand_k is None else _tensor_ptr(cand_k, "bf16", (nq,) + kv, B, "candidate k")
    cvp = None if cand_v is None else _tensor_ptr(cand_v, "bf16", (nq,) + kv, B, "candidate v")
    par = None
    if parent is not None:  # the C call reads n_req * n_query parents
        parent = np.asarray(parent, dtype=np.int32)
        if parent.size != B * nq:
            raise SvxError(ERR_INVALID_ARG, f"parent: {parent.size} entries, expected [{B}, {nq}]")
        parent = np.ascontiguousarray(parent.reshape(B, nq))
        par = parent.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    op = _tensor_ptr(o, "bf16", (Hq, nq, d), B, "o")
    lp = _tensor_ptr(lse, "f32", (Hq, nq), B, "lse")
    st = lib.svx_verify_static(B, Hq, n_kv_heads, d, nq, qp, hp, ks, vs, ckp, cvp, par, ctypes.c_float(scale), op, lp,
                               _stream_handle(stream))
    if st != OK:
        raise SvxError(st, lib.svx_last_error(None).decode())


# ------------------------------------------------------------ the round


def _ptr(t) -> int:
    """Device or host address of a torch tensor (or an int address)."""
    if isinstance(t, int):
        return t
    return t.data_ptr()


_DTYPES = {"bf16": "torch.bfloat16", "f32": "torch.float32"}


def _dense_ptr(t, what: str) -> int:
    """Address of a dense row-major tensor (rows the C call steps over by a byte count)."""
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise SvxError(ERR_INVALID_ARG, f"{what}: not contiguous (the C layout is dense row-major)")
    return t.data_ptr()


def _tensor_ptr(t, dtype: str, tail: tuple, lead: Optional[int], what: str) -> int:
    """Address of a tensor laid out as the C call expects it: element type, dense row-major, the
    trailing dimensions `tail` and at least `lead` entries along the first.  The C calls see only an
    address, so a view with other strides or another type would be read as garbage; such tensors
    raise SvxError(SVX_ERR_INVALID_ARG) here.  Raw int addresses pass unchecked."""
    if isinstance(t, int):
        return t
    if str(t.dtype) != _DTYPES[dtype]:
        raise SvxError(ERR_INVALID_ARG, f"{what}: dtype {t.dtype}, expected {_DTYPES[dtype]}")
    if not t.is_contiguous():
        raise SvxError(ERR_INVALID_ARG, f"{what}: not contiguous (the C layout is dense row-major)")
    shape = tuple(int(n) for n in t.shape)
    if len(shape) != len(tail) + 1 or shape[1:] != tuple(int(n) for n in tail) or \
            (lead is not None and shape[0] < lead):
        want = (f">={lead}" if lead is not None else "n",) + tuple(tail)
        raise SvxError(ERR_INVALID_ARG, f"{what}: shape {list(shape)}, expected [{', '.join(map(str, want))}]")
    return t.data_ptr()


def _stream_handle(s) -> Optional[int]:
    if s is None:
        return None
    return int(getattr(s, "cuda_stream", s))


class Verifier:
    """One svx context: staging slots, state workspace, streams and events."""

    def __init__(self, max_req: int, n_q_heads: int, n_kv_heads: int, head_dim: int, max_query: int,
                 max_chunk_tokens: int, n_slots: int = 2, device: int = 0, compute_stream=None, copy_stream=None,
                 timing: bool = False, tensor_cores: bool = True, zero_copy: bool = False,
                 zero_copy_ctas: int = 0, staged_ctas: int = 0, adaptive: bool = False):
        self._keep = (compute_stream, copy_stream)
        flags = ((FLAG_TIMING if timing else 0) | (0 if tensor_cores else FLAG_NO_TENSOR_CORES)
                 | (FLAG_ZERO_COPY if zero_copy else 0) | (FLAG_ADAPTIVE if adaptive else 0))
        cfg = Config(max_req, n_q_heads, n_kv_heads, head_dim, max_query, max_chunk_tokens, n_slots, device,
                     _stream_handle(compute_stream), _stream_handle(copy_stream), flags, zero_copy_ctas, staged_ctas)
        h = ctypes.c_void_p(None)
        st = lib.svx_create(ctypes.byref(cfg), ctypes.byref(h))
        if st != OK:
            raise SvxError(st, lib.svx_last_error(None).decode())
        self._h = h
        self.cfg = cfg

    def _check(self, st: int):
        if st != OK:
            raise SvxError(st, lib.svx_last_error(self._h).decode())

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib.svx_destroy(self._h)
            self._h = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def round_begin(self, q, hist_len: Sequence[int], n_query: Optional[int] = None, scale: float = 0.0):
        """q: device bf16 [B][Hq][nq][d]."""
        n_req = len(hist_len)
        nq = n_query if n_query is not None else int(q.shape[2])
        c = self.cfg
        qp = _tensor_ptr(q, "bf16", (c.n_q_heads, nq, c.head_dim), n_req, "q")
        h, hp = _i64(hist_len)
        self._check(lib.svx_round_begin(self._h, n_req, nq, qp, hp, ctypes.c_float(scale)))
        self._round = (n_req, nq)

    def push_chunk(self, parts: Sequence[tuple]):
        """parts: (req, tok_start, k, v) with k, v bf16 [n_tok][Hkv][d] (pinned host or device)."""
        arr = (Part * max(1, len(parts)))()
        tail = (self.cfg.n_kv_heads, self.cfg.head_dim)
        for i, (req, t0, k, v) in enumerate(parts):
            n_tok = int(k.shape[0])
            kp = _tensor_ptr(k, "bf16", tail, None, f"part {i} k")
            vp = _tensor_ptr(v, "bf16", tail, n_tok, f"part {i} v")
            arr[i] = Part(req, n_tok, t0, kp, vp)
        self._check(lib.svx_push_chunk(self._h, arr, len(parts)))

    def push_raw(self, parts: Sequence[tuple]):
        """parts: (req, tok_start, n_tok, k_addr, v_addr) with raw addresses."""
        arr = (Part * max(1, len(parts)))()
        for i, (req, t0, n, k, v) in enumerate(parts):
            arr[i] = Part(req, n, t0, k, v)
        self._check(lib.svx_push_chunk(self._h, arr, len(parts)))

    def candidate_attn(self, k, v, parent: Optional[np.ndarray] = None, n_cand: Optional[int] = None):
        """k, v: device bf16 [B][n_cand][Hkv][d]; parent: int32 [B][n_cand] or None (chain)."""
        nc = n_cand if n_cand is not None else int(k.shape[1])
        n_req = getattr(self, "_round", (None, None))[0]
        tail = (nc, self.cfg.n_kv_heads, self.cfg.head_dim)
        kp = _tensor_ptr(k, "bf16", tail, n_req, "candidate k")
        vp = _tensor_ptr(v, "bf16", tail, n_req, "candidate v")
        par = None
        if parent is not None:
            self._parent = np.ascontiguousarray(np.asarray(parent, dtype=np.int32))
            par = self._parent.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        self._check(lib.svx_candidate_attn(self._h, kp, vp, nc, par))

    def round_finish(self, o, lse, timeout_ms: int = 0):
        """o: device bf16 [B][Hq][nq][d]; lse: device fp32 [B][Hq][nq]."""
        n_req, nq = getattr(self, "_round", (None, None))
        if nq is None:  # no round begun: the library reports the state error
            self._check(lib.svx_round_finish(self._h, _ptr(o), _ptr(lse), timeout_ms))
            return
        op = _tensor_ptr(o, "bf16", (self.cfg.n_q_heads, nq, self.cfg.head_dim), n_req, "o")
        lp = _tensor_ptr(lse, "f32", (self.cfg.n_q_heads, nq), n_req, "lse")
        self._check(lib.svx_round_finish(self._h, op, lp, timeout_ms))

    def debug_expire_wait(self, wait_ms: int):
        """Test hook: a kernel whose bounded wait runs out raises the device error word."""
        self._check(lib.svx_debug_expire_wait(self._h, wait_ms))

    def debug_fail_copy(self, nth: int):
        """Test hook: the nth copy submission from now is refused (0 disarms)."""
        self._check(lib.svx_debug_fail_copy(self._h, nth))

    def debug_delay_copy(self, nth: int, delay_ms: int):
        """Test hook: the host sleeps delay_ms before the nth copy submission from now (0 disarms)."""
        self._check(lib.svx_debug_delay_copy(self._h, nth, delay_ms))

    def debug_clip_q_rows(self, rows: int):
        """Test hook of the bounds-checked build: the chunk launches until round_finish state that q has at
        most `rows` rows (< 0: the real count)."""
        self._check(lib.svx_debug_clip_q_rows(self._h, rows))

    def stats(self) -> dict:
        s = Stats()
        self._check(lib.svx_round_stats(self._h, ctypes.byref(s)))
        return {f: getattr(s, f) for f, _ in Stats._fields_}

    def adaptive_state(self) -> dict:
        """The adaptive policy's figures: ms per GB of each engine (None before measured), preference."""
        a, b, p = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_int32(0)
        self._check(lib.svx_adaptive_state(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(p)))
        return {"copy_engine_ms_per_gb": None if a.value < 0 else a.value,
                "in_place_ms_per_gb": None if b.value < 0 else b.value, "prefer_in_place": bool(p.value)}

    def window_reset(self):
        """Opens a new timing window at the next round."""
        self._check(lib.svx_window_reset(self._h))

    def window_stats(self) -> dict:
        s = WindowStats()
        self._check(lib.svx_window_stats(self._h, ctypes.byref(s)))
        return {f: getattr(s, f) for f, _ in WindowStats._fields_}

    def window_intervals(self) -> np.ndarray:
        """[n_pushes][4] float64: copy start, copy end (NaN without copies), kernel start, end (ms from the
        window's first round begin)."""
        n = ctypes.c_int64(0)
        self._check(lib.svx_window_intervals(self._h, None, 0, ctypes.byref(n)))
        out = np.zeros((max(1, n.value), 4), dtype=np.float64)
        self._check(lib.svx_window_intervals(self._h, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), n.value,
                                             ctypes.byref(n)))
        return out[:n.value]

    def window_rounds(self) -> np.ndarray:
        """[n_rounds][3] float64: round begin, finish-kernel start, end (ms from the window's first round)."""
        n = ctypes.c_int64(0)
        self._check(lib.svx_window_rounds(self._h, None, 0, ctypes.byref(n)))
        out = np.zeros((max(1, n.value), 3), dtype=np.float64)
        self._check(lib.svx_window_rounds(self._h, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), n.value,
                                          ctypes.byref(n)))
        return out[:n.value]

    def run_round(self, q, hist_len: Sequence[int], hist_k: Sequence, hist_v: Sequence, chunk_tokens: int,
                  o, lse, cand_k=None, cand_v=None, parent: Optional[np.ndarray] = None,
                  chunk_order: Optional[Sequence[int]] = None, timeout_ms: int = 0, scale: float = 0.0):
        """One round through the C ABI: begin, the candidate region (issued first so it runs under the
        first transfer), one push per cohort chunk of the plan, finish.

        hist_k[b], hist_v[b]: bf16 [C_b][Hkv][d] tensors (pinned host or device) or None when C_b = 0.
        """
        self.round_begin(q, hist_len, scale=scale)
        if cand_k is not None:
            self.candidate_attn(cand_k, cand_v, parent)
        row_bytes = self.cfg.n_kv_heads * self.cfg.head_dim * 2
        chunks = {}
        for j, _slot, b, t0, n in plan_chunks(hist_len, chunk_tokens, self.cfg.n_slots):
            chunks.setdefault(j, []).append((b, t0, n))
        tail = (self.cfg.n_kv_heads, self.cfg.head_dim)
        base_k = [None if k is None else _tensor_ptr(k, "bf16", tail, int(C), f"history k of request {b}")
                  for b, (k, C) in enumerate(zip(hist_k, hist_len))]
        base_v = [None if v is None else _tensor_ptr(v, "bf16", tail, int(C), f"history v of request {b}")
                  for b, (v, C) in enumerate(zip(hist_v, hist_len))]
        for j in (chunk_order if chunk_order is not None else sorted(chunks)):
            parts = chunks[j]
            arr = (Part * len(parts))()
            for i, (b, t0, n) in enumerate(parts):
                arr[i] = Part(b, n, t0, base_k[b] + t0 * row_bytes, base_v[b] + t0 * row_bytes)
            self._check(lib.svx_push_chunk(self._h, arr, len(parts)))
        self.round_finish(o, lse, timeout_ms)
