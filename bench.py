#!/usr/bin/env python
"""Verification-attention benchmark (one JSON line on rank 0).

A step is one verification round of every layer of the workload, through the C
ABI: chunk plan, chunk attention, candidate-region attention and the final merge.
The default workload is the full-depth round: 36 layers of the Qwen3-8B-shaped
attention stack (32 query / 8 KV heads, d = 128), 2 requests x 131072 committed
tokens (38.65 GB of bf16 K and V per step), k = 4 (5 verification queries, causal
candidate chain), chunks of 8192 tokens.

  value  verification tokens/s with every input already in HBM (history read in
         place as device parts): the HBM-bound form of the step.
  e2e    the same metric through the same API with HOST buffers: Q and the
         candidate KV copied from pinned host memory, the committed history of
         every layer read from pinned host memory over the host link by the chunk
         kernel itself (in-place reads on up to every SM), O and LSE copied back and read
         on the host, all inside the timed region.  Overlap figures come from the
         same context's timing window over the same timed steps.  The copy engine
         (chunks staged through triple-buffered slots, the next layer's copies
         queued behind the current layer's) and the adaptive choice between the
         two engines are measured the same way under "streamed_copy_engine" and
         "streamed_adaptive".

The other named workloads (tiny, qwen3, internlm, tree) run as shorter
sub-records under "workloads".  Every step reads more than the 129 MB L2 except
tiny's (stated in its config), so no flush is needed.  --impl reference times
the float64 CPU oracle on a bounded sample of each step instead.
"""
from __future__ import annotations

import argparse
import gc
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "verify-attn tokens/s; streamed-KV GB/s vs host-link & HBM roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
SUB_WORKLOADS = "tiny,qwen3,internlm,tree"
# The pages' own figures for the method, all end to end with real models on other hardware: context for
# the numbers above, not a target for this path.
PAGES_CONTEXT = {
    "hardware": "2x NVIDIA A800 80GB PCIe Gen4 (TP = 2), 240 GB host memory; precision not stated",
    "vs_offloading_baseline": "1.41x (Qwen3) and 1.32x (InternLM2.5) average output throughput over TriForce",
    "vs_split_gpu_parallel_sd": "+55.4% output throughput per GPU versus SPECTRE+Offload on separate GPUs",
    "stream_and_reduce_vs_restore_then_verify": "+83.2% (Qwen3) and +117.1% (InternLM2.5), q = 4, 16K inputs",
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["svx", "reference"], default="svx")
    ap.add_argument("--workload", default="fulldepth", choices=list(W.NAMES))
    ap.add_argument("--layers", type=int, default=None,
                    help="layers per step (default: the workload's; fewer keep every launch's shape, for profiling)")
    ap.add_argument("--head-dim", type=int, choices=[64, 128], default=None,
                    help="the workload with another head dimension (same tokens, heads and queries)")
    ap.add_argument("--sub-workloads", default=SUB_WORKLOADS,
                    help="comma list of further workloads measured briefly under 'workloads' (empty = none)")
    ap.add_argument("--zero-copy-ctas", default="8,32,64",
                    help="comma list of CTA caps for further in-place (zero-copy) streamed variants (0 = all SMs; empty = skip)")
    ap.add_argument("--e2e-ctas", type=int, default=0,
                    help="CTAs of the e2e context's in-place chunk launches (reads of pinned host history)")
    ap.add_argument("--adaptive-ctas", type=int, default=0,
                    help="CTAs of the adaptive context's chunk launches when it reads in place")
    ap.add_argument("--staged-ctas", type=int, default=16,
                    help="CTA budget of staged chunk launches in the Target-priority variant of the copy engine")
    ap.add_argument("--tp-sub-workloads", default="qwen3,internlm,tree",
                    help="sub-workloads that also get the Target-priority record (Draft beside the streamed step)")
    ap.add_argument("--no-draft-load", dest="draft_load", action="store_false",
                    help="skip timing the streamed step beside a low-priority bf16 GEMM loop (Target priority)")
    ap.add_argument("--slots", type=int, default=3, choices=[2, 3])
    ap.add_argument("--resident-chunk", default="whole", choices=["whole", "plan"],
                    help="device-resident history pushed as one part per request, or in the plan's chunks")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-method", dest="method", action="store_false",
                    help="skip the method sub-records (dynamic width, tiering)")
    ap.add_argument("--profile-in-place", action="store_true",
                    help="only the e2e context's in-place steps (inputs, then --warmup and --steps steps), for a "
                         "profiler to capture its launches; prints their mean step time")
    ap.add_argument("--cpu-sample-pairs", type=int, default=0,
                    help="(layer, request, KV head) pairs in each CPU sample (default: one per core)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- distributed plumbing


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (the slowest rank sets the job time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, ms_per_rank: float, world: int, device=None) -> tuple:
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    ms = max_over_ranks(ms_per_rank, world, device)
    return units_per_rank * world / (ms / 1e3), ms


# ---------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.index)], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self) -> dict:
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- CPU oracle sample


def _oracle_pair(args):
    """Oracle rows of one (layer, request, KV head) triple: all G*nq queries of that KV head."""
    import oracle
    q_bits, kh_bits, vh_bits, kc_bits, vc_bits, vis, scale = args
    f = W.bf16_to_f64
    t0 = time.perf_counter()
    o, l = oracle.verify_attention(f(q_bits), [f(kh_bits)], [f(vh_bits)], f(kc_bits), f(vc_bits), vis, scale=scale)
    return time.perf_counter() - t0, float(np.nansum(l))


def oracle_tasks(w: W.Workload, x: W.LayerInputs, pairs):
    import oracle
    vis = oracle.visibility_table(w.n_req, w.n_query, x.parent)
    G = w.group
    tasks = []
    for b, g in pairs:
        tasks.append((x.q[b:b + 1, g * G:(g + 1) * G], x.k_hist[b][:, g:g + 1], x.v_hist[b][:, g:g + 1],
                      x.k_cand[b:b + 1, :, g:g + 1], x.v_cand[b:b + 1, :, g:g + 1], vis[b:b + 1], w.scale))
    return tasks


def cpu_sample_pairs(w: W.Workload, n: int):
    all_pairs = [(b, g) for b in range(w.n_req) for g in range(w.n_kv_heads)]
    rng = np.random.default_rng(123)
    idx = rng.permutation(len(all_pairs))[:n]
    return [all_pairs[i] for i in sorted(idx)]


def oracle_sample(pool, tasks, w: W.Workload, n_layers: int) -> dict:
    """One bounded CPU sample: the oracle over `tasks` (one (request, KV head) pair of one layer each) on
    the pool.  The fraction of a whole step it covers and the tokens/s that rate gives."""
    t0 = time.perf_counter()
    list(pool.map(_oracle_pair, tasks))
    dt = time.perf_counter() - t0
    frac = len(tasks) / (n_layers * w.n_req * w.n_kv_heads)
    return {"seconds": dt, "step_fraction": frac, "value": w.n_req * w.n_query * frac / dt}


# ---------------------------------------------------------------- reference arm


def run_reference(a, rank, world):
    """The float64 oracle on the host cores, on this arm's workload, metric and unit.  Each timed step is
    one bounded sample (one (request, KV head) pair of layer 0 per core); the line says what fraction of
    a whole step that is, and `value` is the sample's tokens/s (the fraction of the step's tokens over
    its time)."""
    if rank != 0:
        return 0
    import multiprocessing as mp
    w = workload_of(a)
    L = w.n_layers
    cores = os.cpu_count() or 1
    n_pairs = min(a.cpu_sample_pairs or cores, w.n_req * w.n_kv_heads)
    pairs = cpu_sample_pairs(w, n_pairs)
    x = W.layer_inputs(w, 0, requests=None) if w.n_layers == 1 or w.hist_bytes < (4 << 30) else None
    if x is None:  # multi-GiB layers: draw only the sampled requests' histories
        reqs = sorted({b for b, _g in pairs})
        xs = W.layer_inputs(w, 0, requests=reqs)
        full_k, full_v = [None] * w.n_req, [None] * w.n_req
        for i, b in enumerate(reqs):
            full_k[b], full_v[b] = xs.k_hist[i], xs.v_hist[i]
        x = W.LayerInputs(xs.q, full_k, full_v, xs.k_cand, xs.v_cand, xs.parent)
    tasks = oracle_tasks(w, x, pairs)
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(cores, len(tasks))) as pool:
        for _ in range(a.warmup):
            oracle_sample(pool, tasks[:1], w, L)
        samples = [oracle_sample(pool, tasks, w, L) for _ in range(a.steps)]
    value = statistics.median(s["value"] for s in samples)
    ms = statistics.median(s["seconds"] for s in samples) * 1e3
    frac = samples[0]["step_fraction"]
    sample = (f"each step: {len(tasks)} of {L * w.n_req * w.n_kv_heads} (layer, request, KV head) pairs of one step "
              f"({len(tasks) * w.group * w.n_query} of {L * w.n_req * w.n_q_heads * w.n_query} layer query rows), "
              f"a {frac:.4f} fraction of the step; value = that fraction of the step's tokens over the sample's time")
    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
           "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference", "sampled": True, "step_fraction": frac,
           "config": workload_config(w, a),
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(cores, len(tasks)), "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))
    return 0


def workload_of(a) -> W.Workload:
    w = W.named(a.workload)
    if a.head_dim:
        w = w.with_(head_dim=a.head_dim)
    if getattr(a, "layers", None):
        w = w.with_(n_layers=a.layers)
    return w


def workload_config(w: W.Workload, a) -> dict:
    l2_bytes = 129e6
    per_round = 4 * w.n_kv_heads * w.head_dim * sum(w.hist_len)
    layers = f"{w.n_layers} layers x " if w.n_layers > 1 else ""
    return {"workload": f"{w.name}: {layers}{w.n_req} requests, {w.n_q_heads}/{w.n_kv_heads} heads, d={w.head_dim}, "
                        f"history {min(w.hist_len)}..{max(w.hist_len)} tokens, chunk {w.chunk_tokens}, "
                        f"{w.n_query} verify queries ({'token tree' if w.tree else 'causal chain'})",
            "n_layers": w.n_layers, "n_req": w.n_req, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
            "head_dim": w.head_dim, "hist_tokens": int(sum(w.hist_len)), "chunk_tokens": w.chunk_tokens,
            "n_query": w.n_query, "slots": a.slots, "resident_chunk": a.resident_chunk,
            "l2": (f"no flush: one round reads {per_round / 2**20:.0f} MiB of history, more than the 129 MB L2"
                   if per_round > l2_bytes else
                   f"no flush: one round reads {per_round / 2**10:.0f} KiB of history, which stays in the 129 MB L2"),
            "seed": w.seed}


# ---------------------------------------------------------------- GPU arm


class DraftLoad:
    """Synthetic Draft co-execution (section 4.3's Draft model as a pure compute load): bf16
    4096^3 GEMMs (cuBLAS via torch.matmul) captured in a CUDA graph and replayed from a host thread
    on a lowest-priority stream, at most `per_replay` GEMMs in flight.  Warmed up (cuBLAS
    initialisation, graph capture) before any timing."""

    def __init__(self, dev, n=4096, per_replay=8):
        import torch
        self.torch = torch
        self.dev = dev
        lo, _hi = torch.cuda.Stream.priority_range()
        self.stream = torch.cuda.Stream(device=dev, priority=lo)
        self.a = torch.randn((n, n), device=dev, dtype=torch.bfloat16)
        self.b = torch.randn((n, n), device=dev, dtype=torch.bfloat16)
        self.c = torch.empty((n, n), device=dev, dtype=torch.bfloat16)
        with torch.cuda.stream(self.stream):
            for _ in range(3):
                torch.matmul(self.a, self.b, out=self.c)
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            for _ in range(per_replay):
                torch.matmul(self.a, self.b, out=self.c)
        torch.cuda.synchronize(dev)
        self.flops = 2.0 * n ** 3
        self.per_replay = per_replay
        self.count = 0
        self.stop_flag = False
        self.thread = None

    def _run(self):
        torch = self.torch
        torch.cuda.set_device(self.dev)
        ev = torch.cuda.Event()
        while not self.stop_flag:
            with torch.cuda.stream(self.stream):
                self.graph.replay()
                ev.record(self.stream)
            ev.synchronize()
            self.count += self.per_replay

    def start(self):
        import threading
        self.stop_flag = False
        self.count = 0
        self.t0 = time.perf_counter()
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self) -> float:
        self.stop_flag = True
        self.thread.join()
        dt = time.perf_counter() - self.t0
        return self.count * self.flops / dt / 1e12


class AdmittedDraft:
    """Draft steps admitted by the library's Target-priority scheduler (section 4.3, "Target-priority
    scheduling" and the two paragraphs after it), in place of a free-running Draft.

    The Draft stand-in runs one bf16 4096^3 GEMM (cuBLAS) per Draft step on a lowest-priority stream,
    from a host thread.  For each request it asks svx_sched_try_admit with the time left in the
    Target's current round (the round began at t0 and is predicted to take S ms); an admitted
    instruction is checked again with svx_sched_check_start right before the launch (the Draft side of
    the protocol: same request and round, t_latest not passed) and acknowledged from the step's
    completion event with its measured time.  The Target side calls begin_round before each
    verification round and end_round with the round's measured time, which feeds
    svx_sched_observe_target (an observed increase over eps_T pauses new submissions)."""

    def __init__(self, dev, n_req, eps_target=0.05, delta_ms=0.5, ema=0.3, t_draft_ms=0.1, n=4096):
        import threading
        import torch
        from speculative_decoding_verification_chunked_gb300 import svx
        self.torch, self.dev, self.n_req = torch, dev, n_req
        lo, _hi = torch.cuda.Stream.priority_range()
        self.stream = torch.cuda.Stream(device=dev, priority=lo)
        self.a = torch.randn((n, n), device=dev, dtype=torch.bfloat16)
        self.b = torch.randn((n, n), device=dev, dtype=torch.bfloat16)
        self.c = torch.empty((n, n), device=dev, dtype=torch.bfloat16)
        with torch.cuda.stream(self.stream):
            torch.matmul(self.a, self.b, out=self.c)
        torch.cuda.synchronize(dev)
        self.flops = 2.0 * n ** 3
        self.eps = eps_target
        self.sched = svx.Scheduler(eps_target, delta_ms, ema, t_draft_ms, 0.0, alloc=0)
        self.lock = threading.Lock()
        self.round, self.t0, self.S = -1, 0.0, 0.0
        self.log = []  # (host time at launch, t_latest) of every executed step
        self.rejected = self.admitted = self.paused_rounds = 0
        self.stop_flag = False

    @staticmethod
    def now_ms():
        return time.perf_counter() * 1e3

    def begin_round(self, r, predicted_ms):
        with self.lock:
            self.sched.new_round()
            if self.sched.estimates()[2]:
                self.paused_rounds += 1
            self.round, self.t0, self.S = r, self.now_ms(), predicted_ms

    def end_round(self, t_co_ms, t_alone_ms):
        with self.lock:
            self.sched.observe_target(t_co_ms, t_alone_ms)

    def _run(self):
        torch = self.torch
        torch.cuda.set_device(self.dev)
        while not self.stop_flag:
            launched = False
            for req in range(self.n_req):
                with self.lock:
                    now = self.now_ms()
                    ins = self.sched.try_admit(req, self.round, now, self.t0 + self.S - now)
                if ins is None:
                    continue
                self.admitted += 1
                with self.lock:  # the Draft side's check right before it starts the step
                    now = self.now_ms()
                    ok = self.sched.check_start(ins, req, self.round, now)
                if not ok:
                    self.rejected += 1
                    continue
                self.log.append((now, ins.t_latest))
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(self.stream):
                    e0.record(self.stream)
                    torch.matmul(self.a, self.b, out=self.c)
                    e1.record(self.stream)
                e1.synchronize()
                with self.lock:
                    self.sched.ack(req, ins.seq, e0.elapsed_time(e1))
                launched = True
            if not launched:
                time.sleep(0.0002)

    def start(self):
        import threading
        self.stop_flag = False
        self.log.clear()
        self.rejected = self.admitted = self.paused_rounds = 0
        self.t_start = time.perf_counter()
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self) -> float:
        """Stops the Draft thread; returns the Draft's TFLOP/s since start()."""
        self.stop_flag = True
        self.thread.join()
        return len(self.log) * self.flops / (time.perf_counter() - self.t_start) / 1e12


def run_admitted(R, step_fn, steps, ms_alone, draft):
    """Target steps with Draft steps admitted by the scheduler: each step is one verification round,
    timed with CUDA events on the compute stream and reported to the scheduler.  Returns the mean step
    time and the admission figures."""
    torch = R.torch
    draft.start()
    times = []
    for r in range(steps):
        draft.begin_round(r, ms_alone)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(R.cs)
        step_fn()
        e1.record(R.cs)
        e1.synchronize()
        t = e0.elapsed_time(e1)
        times.append(t)
        draft.end_round(t, ms_alone)
    tf = draft.stop()
    late = sum(1 for t_launch, t_latest in draft.log if t_launch > t_latest)
    ms = statistics.mean(times)
    return ms, {"delta_T": (ms - ms_alone) / ms_alone, "target_ms_alone": ms_alone, "target_ms_co": ms,
                "draft_tflops_co": tf, "eps_T": draft.eps, "draft_steps": len(draft.log),
                "instructions": draft.admitted, "expired_or_stale": draft.rejected,
                "started_after_t_latest": late, "paused_rounds": draft.paused_rounds}


class Inputs:
    """One workload's inputs on the device and in pinned host memory, per layer.

    History: each layer's K and V as rows of one pinned [B][C_max][Hkv][d] tensor per tensor (the layout
    of a batched host KV cache: a chunk's parts are equally strided, and the library stages each chunk
    with one 2D copy for K and one for V), filled from the device-side seeded generator; optionally the
    same history resident in HBM (device parts, the HBM-bound form)."""

    def __init__(self, w: W.Workload, dev, resident=True):
        import torch
        self.w = w
        B, Hq, Hkv, d, nq = w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query
        bf = torch.bfloat16
        self.row_bytes = Hkv * d * 2
        self.layers = []
        for layer in range(w.n_layers):
            kb = torch.empty((B, max(w.hist_len), Hkv, d), dtype=bf, pin_memory=True)
            vb = torch.empty((B, max(w.hist_len), Hkv, d), dtype=bf, pin_memory=True)
            kh_h = [kb[b, :C] for b, C in enumerate(w.hist_len)]
            vh_h = [vb[b, :C] for b, C in enumerate(w.hist_len)]
            q, kh_d, vh_d, kc, vc, parent = W.layer_inputs_device(w, layer, dev)
            for b in range(B):
                kh_h[b].copy_(kh_d[b])
                vh_h[b].copy_(vh_d[b])
            ly = dict(q_h=q.cpu().pin_memory(), kc_h=kc.cpu().pin_memory(), vc_h=vc.cpu().pin_memory(),
                      kh_h=kh_h, vh_h=vh_h, kh_d=kh_d if resident else None, vh_d=vh_d if resident else None,
                      q_d=q, kc_d=kc, vc_d=vc, parent=parent,
                      o_d=torch.empty((B, Hq, nq, d), dtype=bf, device=dev),
                      lse_d=torch.empty((B, Hq, nq), dtype=torch.float32, device=dev),
                      o_h=torch.empty((B, Hq, nq, d), dtype=bf).pin_memory(),
                      lse_h=torch.empty((B, Hq, nq), dtype=torch.float32).pin_memory())
            self.layers.append(ly)
            del kh_d, vh_d
        torch.cuda.synchronize(dev)
        from speculative_decoding_verification_chunked_gb300 import svx
        self.chunks = {}
        for j, _s, b, t0, n in svx.plan_chunks(w.hist_len, w.chunk_tokens, 3):
            self.chunks.setdefault(j, []).append((b, t0, n))

    def parts(self, kh, vh, whole: bool):
        """Pushes (lists of raw parts) of one layer: one part per request, or the plan's chunks."""
        w, rb = self.w, self.row_bytes
        if whole:
            return [[(b, 0, w.hist_len[b], kh[b].data_ptr(), vh[b].data_ptr()) for b in range(w.n_req)
                     if w.hist_len[b]]]
        return [[(b, t0, n, kh[b].data_ptr() + t0 * rb, vh[b].data_ptr() + t0 * rb) for b, t0, n in self.chunks[j]]
                for j in sorted(self.chunks)]

    def drop_resident(self, keep_first=True):
        """Free the device duplicates (a streaming deployment does not hold its history in HBM twice)."""
        import torch
        for ly in self.layers[1 if keep_first else 0:]:
            ly["kh_d"] = ly["vh_d"] = None
        torch.cuda.empty_cache()

    def oracle_layer0(self) -> W.LayerInputs:
        """Layer 0's inputs as drawn, read back from pinned host memory (bf16 bit patterns)."""
        import torch
        u16 = lambda t: t.view(torch.int16).numpy().view(np.uint16)  # noqa: E731
        ly = self.layers[0]
        return W.LayerInputs(u16(ly["q_h"]), [u16(k) for k in ly["kh_h"]], [u16(v) for v in ly["vh_h"]],
                             u16(ly["kc_h"]), u16(ly["vc_h"]), ly["parent"])


class Runner:
    """Timed steps of one workload on one GPU (rank)."""

    def __init__(self, a, w, dev, world, cs, xs):
        import torch
        self.torch, self.a, self.w, self.dev, self.world, self.cs, self.xs = torch, a, w, dev, world, cs, xs

    def verifier(self, **kw):
        from speculative_decoding_verification_chunked_gb300 import svx
        w = self.w
        return svx.Verifier(w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query, w.chunk_tokens,
                            n_slots=self.a.slots, device=self.dev.index, compute_stream=self.cs, copy_stream=self.xs,
                            **kw)

    def timed(self, step_fn, steps, warmup, between=None, lead_ms=0.0):
        """Mean ms per step over `steps` steps after `warmup`, CUDA events on the compute stream, a barrier and
        a device synchronisation on both sides.  `between()` runs after the warm-up, before the timing.
        lead_ms > 0: the compute stream first spins that long (before the start event), so the host has
        enqueued the steps' work before the GPU reaches it (for timing single launches inside the steps)."""
        torch = self.torch
        for _ in range(warmup):
            step_fn()
        torch.cuda.synchronize(self.dev)
        if between is not None:
            between()
        # Python's cycle collector stays out of the timed steps: a collection there can free an earlier
        # workload's pinned host buffers (cudaFreeHost of tens of GB stalls the device for ~100 ms)
        gc.collect()
        gc_on = gc.isenabled()
        gc.disable()
        try:
            barrier(self.world)
            torch.cuda.synchronize(self.dev)
            if lead_ms > 0:
                with torch.cuda.stream(self.cs):
                    torch.cuda._sleep(int(lead_ms * 2.0e6))  # ~2 GHz SM clock
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.cs)
            for _ in range(steps):
                step_fn()
            e1.record(self.cs)
            torch.cuda.synchronize(self.dev)
            barrier(self.world)
        finally:
            if gc_on:
                gc.enable()
        return e0.elapsed_time(e1) / steps

    def round_of(self, v, ly, pushes, timeout_ms=0):
        v.round_begin(ly["q_d"], self.w.hist_len)
        v.candidate_attn(ly["kc_d"], ly["vc_d"], ly["parent"])
        for p in pushes:
            v.push_raw(p)
        v.round_finish(ly["o_d"], ly["lse_d"], timeout_ms=timeout_ms)

    def host_step(self, v, inp, pushes_of):
        """One step with host inputs: Q and candidates copied in, every layer's round, O and LSE copied out
        and read by the host (the step ends when its result is on the host, as a decode loop needs it to
        accept or reject the drafts before the next round)."""
        torch, cs = self.torch, self.cs
        with torch.cuda.stream(cs):
            for ly in inp.layers:
                ly["q_d"].copy_(ly["q_h"], non_blocking=True)
                ly["kc_d"].copy_(ly["kc_h"], non_blocking=True)
                ly["vc_d"].copy_(ly["vc_h"], non_blocking=True)
        for li, ly in enumerate(inp.layers):  # layer l+1's chunk copies queue behind layer l's: prefetch
            self.round_of(v, ly, pushes_of(li))
            with torch.cuda.stream(cs):
                ly["o_h"].copy_(ly["o_d"], non_blocking=True)
                ly["lse_h"].copy_(ly["lse_d"], non_blocking=True)
        cs.synchronize()

    def checked(self, v, inp, pushes):
        """One round of layer 0 whose finish reads the context's device error word: a kernel whose bounded
        wait ran out in any earlier round of the context raises here, so no line rests on aborted launches."""
        self.round_of(v, inp.layers[0], pushes, timeout_ms=60000)


def copy_rates(iv, push_bytes):
    """Per-push copy-engine rates (GB/s) from window intervals: min, median, max and the share of pushes
    below 150 GB/s."""
    cp = iv[:, 1] - iv[:, 0]
    ok = np.isfinite(cp) & (cp > 0)
    if not ok.any():
        return None
    r = np.asarray(push_bytes, dtype=np.float64)[ok] / (cp[ok] / 1e3) / 1e9
    return {"min": float(r.min()), "median": float(np.median(r)), "max": float(r.max()),
            "below_150_frac": float((r < 150).mean()), "pushes": int(ok.sum())}


def step_overlap(iv, rounds, layers: int):
    """Per step of a timing window: (T_step, T_transfer) in ms.  T_step runs from the step's first round
    begin to its last finish-kernel end; T_transfer is the length of the union, inside the step, of the
    pushes' copy intervals and of the chunk kernels of pushes read in place (no copy interval).  Steps are
    separated by the host reading each step's result, so every interval belongs to the step it lies in
    (an adaptive context launches an in-place round's pushes together, so the number of intervals per
    step varies)."""
    iv = np.asarray(iv, dtype=np.float64).reshape(-1, 4)
    has_copy = np.isfinite(iv[:, 0])
    ta = np.where(has_copy, iv[:, 0], iv[:, 2])
    tb = np.where(has_copy, iv[:, 1], iv[:, 3])
    out = []
    for s in range(len(rounds) // layers):
        t0, t1 = rounds[s * layers, 0], rounds[(s + 1) * layers - 1, 2]
        sel = (tb > t0) & (ta < t1)
        tr = sorted(zip(ta[sel].tolist(), tb[sel].tolist()))
        busy, cur = 0.0, None
        for a, b in tr:
            a, b = max(a, t0), min(b, t1)
            if b <= a:
                continue
            if cur is None or a > cur[1]:
                if cur is not None:
                    busy += cur[1] - cur[0]
                cur = [a, b]
            else:
                cur[1] = max(cur[1], b)
        if cur is not None:
            busy += cur[1] - cur[0]
        out.append((t1 - t0, busy))
    return out


def link_probe(inp, dev, xs):
    """Pinned host -> HBM bandwidth now (one 256 MiB copy of layer 0's first K rows, best of 4)."""
    import torch
    src = inp.layers[0]["kh_h"][0]
    n = min(src.shape[0], (256 << 20) // inp.row_bytes)
    src = src[:n]
    dst = torch.empty_like(src, device=dev)
    best = 0.0
    for _ in range(4):
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(xs):
            e0.record(xs)
            dst.copy_(src, non_blocking=True)
            e1.record(xs)
        torch.cuda.synchronize(dev)
        best = max(best, src.numel() * 2 / (e0.elapsed_time(e1) / 1e3) / 1e9)
    return best


def measure(a, w, dev, world, cs, xs, hbm_peak, hbm_src, full: bool) -> dict:
    """All timed figures of one workload.  `full`: the headline record (every variant); otherwise a
    shorter sub-record (resident value, kernel roofline, and the e2e, copy-engine and adaptive streamed
    steps with their overlap figures)."""
    import torch
    B, nq, L = w.n_req, w.n_query, w.n_layers
    steps = a.steps if full else min(a.steps, 20)
    warmup = a.warmup if full else min(a.warmup, 3)
    inp = Inputs(w, dev)
    R = Runner(a, w, dev, world, cs, xs)
    hist_bytes = w.hist_bytes * L
    row_bytes = inp.row_bytes
    rec = {"config": workload_config(w, a)}

    # ---- value: resident history (HBM-bound form of the step)
    res_pushes = [inp.parts(ly["kh_d"], ly["vh_d"], a.resident_chunk == "whole") for ly in inp.layers]
    v_res = R.verifier()

    def resident_step():
        for ly, pushes in zip(inp.layers, res_pushes):
            R.round_of(v_res, ly, pushes)

    ms_res = R.timed(resident_step, steps, warmup)
    # the same steps with events around every chunk launch (an event between two kernels of a round keeps
    # the second from launching early, so these are not the value's steps): the dominant kernel's time
    kern_ev = []

    def resident_step_events():
        for ly, pushes in zip(inp.layers, res_pushes):
            v_res.round_begin(ly["q_d"], w.hist_len)
            v_res.candidate_attn(ly["kc_d"], ly["vc_d"], ly["parent"])
            for p in pushes:
                e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                e[0].record(cs)
                v_res.push_raw(p)
                e[1].record(cs)
                kern_ev.append((e, sum(n for _b, _t, n, _k, _v in p)))
            v_res.round_finish(ly["o_d"], ly["lse_d"])

    # The GPU first spins for about the host's time to enqueue every timed round, so that each launch's
    # interval is the launch alone, never the host's time to submit it (short launches, as a single qwen3
    # layer's 90 us, would otherwise wait on the host).  The first timed step is dropped as well.
    R.timed(resident_step_events, steps, 1, between=kern_ev.clear, lead_ms=min(200.0, 0.2 * steps * L))
    per_step = len(kern_ev) // steps
    kern = [(e[0].elapsed_time(e[1]), toks) for e, toks in kern_ev[per_step if steps > 1 else 0:]]
    k1_ms = statistics.mean(k for k, _ in kern)
    k1_bytes = statistics.mean(t for _, t in kern) * row_bytes * 2
    # the same step captured once in a CUDA graph and replayed: the shapes are fixed, so the host cost of
    # the API calls (validation, planning, launches) is paid at capture; the kernels are the same
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cs):
        resident_step()

    def replay():
        with torch.cuda.stream(cs):
            graph.replay()

    ms_graph = R.timed(replay, steps, warmup)
    R.checked(v_res, inp, res_pushes[0])
    ms_eager = ms_res
    ms_res = min(ms_eager, ms_graph)
    value, ms_res_job = job_throughput(B * nq, ms_res, world, dev)
    rec.update(value=value, ms_per_step=ms_res_job, steps=steps, warmup=warmup,
               launches_per_step=sum(len(p) for p in res_pushes) + L)
    rec["roofline"] = {"bound": "hbm", "achieved": k1_bytes / (k1_ms / 1e3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                       "frac": k1_bytes / (k1_ms / 1e3) / 1e9 / hbm_peak, "traffic": profiled_traffic(w),
                       "kernel": "chunk_attn_tc", "peak_source": f"{hbm_src} hbm_gbs (burst copy)",
                       "algorithmic_bytes_per_launch": int(k1_bytes), "ms_per_launch": k1_ms}
    rec["resident"] = {"hist_gb_per_s": hist_bytes / (ms_res / 1e3) / 1e9,
                       "hbm_frac": hist_bytes / (ms_res / 1e3) / 1e9 / hbm_peak,
                       "eager_ms_per_step": ms_eager, "graph_ms_per_step": ms_graph,
                       "value_from": "CUDA-graph replay" if ms_graph <= ms_eager else "eager API calls"}
    # the same chunks' kernels in resident mode (device parts in the plan's chunks): the compute the
    # streamed step has to hide, for the hidden fraction over the step
    v_rt = R.verifier(timing=True)
    plan_pushes0 = inp.parts(inp.layers[0]["kh_d"], inp.layers[0]["vh_d"], False)

    def resident_plan_step():
        for ly in inp.layers:
            R.round_of(v_rt, ly, plan_pushes0)

    R.timed(resident_plan_step, min(steps, 5), 1, between=v_rt.window_reset)
    res_chunk_ms_step = v_rt.window_stats()["chunk_kernel_ms"] / min(steps, 5)
    R.checked(v_rt, inp, plan_pushes0)
    v_rt.close()
    v_res.close()
    inp.drop_resident(keep_first=False)

    # ---- e2e: streamed from pinned host through the public API, every transfer in the timed region.  The
    # e2e engine is the chunk kernel's in-place reads of pinned host memory over the host link; the copy
    # engine (staging slots) and the adaptive choice between the two are measured the same way beside it.
    stream_pushes = [inp.parts(ly["kh_h"], ly["vh_h"], False) for ly in inp.layers]  # the plan's chunks
    whole_pushes = [inp.parts(ly["kh_h"], ly["vh_h"], True) for ly in inp.layers]    # one part per request
    push_bytes = [sum(n for _b, _t, n, _k, _v in p) * row_bytes * 2 for pl in stream_pushes for p in pl]
    link_before = link_probe(inp, dev, xs)

    def streamed(v, pushes, label):
        """Streamed steps through context v: throughput, overlap over the timed steps (the context's timing
        window), per-push copy rates."""
        ms = R.timed(lambda: R.host_step(v, inp, lambda li: pushes[li]), steps, warmup, between=v.window_reset)
        ws = v.window_stats()
        iv = v.window_intervals()
        so = step_overlap(iv, v.window_rounds(), L)
        val, ms_job = job_throughput(B * nq, ms, world, dev)
        covered = ws["n_rounds"] / L  # steps in the window (all timed steps unless it filled up)
        per_step = {k: ws[k] / covered for k in ("window_ms", "copy_busy_ms", "copy_gap_ms", "chunk_kernel_ms",
                                               "chunk_kernel_exposed_ms", "transfer_busy_ms",
                                               "zero_copy_kernel_ms", "finish_kernel_ms")}
        staged_kernel = ws["chunk_kernel_ms"] - ws["zero_copy_kernel_ms"]
        out = {"value": val, "unit": UNIT, "ms_per_step": ms_job, "what": label,
               "hist_gb_per_s": hist_bytes / (ms / 1e3) / 1e9,
               "per_step_ms": per_step,
               # rounds read in place (an adaptive context launches an in-place round's pushes together,
               # so it counts one in-place push per such round)
               "in_place_round_frac": min(1.0, ws["n_zero_copy_pushes"] / max(1, ws["n_rounds"])),
               # per-push copy rates when every planned push has its own interval (an adaptive context's
               # in-place rounds launch their pushes together)
               "copy_rate_gbs": (copy_rates(iv, push_bytes * steps)
                                 if pushes is stream_pushes and ws["n_rounds"] == steps * L
                                 and len(iv) == len(push_bytes) * steps else None),
               # chunk compute hidden under transfer: the time of chunk kernels over staged parts that lies
               # inside transfer intervals; a kernel that reads host memory in place is the transfer itself
               # (1.0 when every push is read in place)
               "hidden_frac": 1.0 - ws["chunk_kernel_exposed_ms"] / staged_kernel if staged_kernel > 0 else 1.0,
               # per step (first round begin to last finish end): whatever of the step is not transfer time
               # counts as exposed compute, against the same chunks' kernel time with resident history;
               # the median over the timed steps
               "hidden_frac_step": statistics.median(1.0 - max(0.0, t - tr) / res_chunk_ms_step for t, tr in so),
               "step_ms_median": statistics.median(t for t, _ in so),
               "step_transfer_ms_median": statistics.median(tr for _, tr in so),
               "resident_chunk_kernel_ms_per_step": res_chunk_ms_step}
        return out, ms

    e2e_ctas = a.e2e_ctas
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    e2e_name = f"in_place_{e2e_ctas}_ctas" if e2e_ctas > 0 else "in_place_all_sms"
    v_e2e = R.verifier(timing=True, zero_copy=True, zero_copy_ctas=e2e_ctas)
    e2e_rec, ms_e2e = streamed(v_e2e, whole_pushes, f"in-place reads: the chunk kernel reads each layer's pinned host "
                                                    f"history over the host link on "
                                                    f"{e2e_ctas if e2e_ctas > 0 else f'up to {n_sms}'} CTAs")
    R.checked(v_e2e, inp, whole_pushes[0])
    v_ce = R.verifier(timing=True)
    ce_rec, ms_ce = streamed(v_ce, stream_pushes, f"copy engine: every chunk staged through {a.slots} slots")
    R.checked(v_ce, inp, stream_pushes[0])
    v_ad = R.verifier(timing=True, adaptive=True, zero_copy_ctas=a.adaptive_ctas)
    ad_rec, ms_ad = streamed(v_ad, stream_pushes, f"adaptive: per round the copy engine, or in-place reads on "
                                                  f"{a.adaptive_ctas if a.adaptive_ctas > 0 else f'up to {n_sms}'} "
                                                  f"CTAs when measured 10% faster")
    ad_rec["adaptive_state"] = v_ad.adaptive_state()
    R.checked(v_ad, inp, stream_pushes[0])
    link_after = link_probe(inp, dev, xs)
    link_gbs = max(link_before, link_after)
    for r in (e2e_rec, ce_rec, ad_rec):
        r["link_frac"] = r["hist_gb_per_s"] / link_gbs
    e2e_value, ms_e2e_job = job_throughput(B * nq, ms_e2e, world, dev)
    h2d_step = hist_bytes + sum((ly["q_h"].numel() + ly["kc_h"].numel() + ly["vc_h"].numel()) * 2
                                for ly in inp.layers)
    d2h_step = sum(ly["o_h"].numel() * 2 + ly["lse_h"].numel() * 4 for ly in inp.layers)
    rec["e2e"] = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d_step),
                  "d2h_bytes_per_step": int(d2h_step), "ms_per_step": ms_e2e_job}
    rec["streamed"] = dict(e2e_rec, link_gbs=link_gbs, link_gbs_before_after=[link_before, link_after])
    rec["streamed_copy_engine"] = ce_rec
    rec["streamed_adaptive"] = ad_rec

    # ---- in-place reads on other CTA budgets
    zc = {}
    with_tp = a.draft_load and (full or w.name in [n.strip() for n in a.tp_sub_workloads.split(",")])
    caps = [int(x) for x in a.zero_copy_ctas.split(",") if x.strip() != "" and int(x) != e2e_ctas]
    if not full:  # a sub-record measures the budgets that leave most SMs to a Draft, if it reports one
        caps = [c_ for c_ in caps if c_ in (8, 32)] if with_tp else []
    zc_ctx = {}
    for cap in caps:
        vz = R.verifier(zero_copy=True, zero_copy_ctas=cap)
        ms = R.timed(lambda vz=vz: R.host_step(vz, inp, lambda li: whole_pushes[li]), steps, warmup)
        R.checked(vz, inp, whole_pushes[0])
        val, ms_job = job_throughput(B * nq, ms, world, dev)
        zc[str(cap)] = {"value": val, "unit": UNIT, "ms_per_step": ms_job,
                        "hist_gb_per_s": hist_bytes / (ms / 1e3) / 1e9,
                        "link_frac": hist_bytes / (ms / 1e3) / 1e9 / link_gbs,
                        "ctas": cap if cap > 0 else n_sms}
        zc_ctx[cap] = (vz, whole_pushes, ms)
    zc[str(e2e_ctas)] = {"value": e2e_rec["value"], "unit": UNIT, "ms_per_step": e2e_rec["ms_per_step"],
                         "hist_gb_per_s": e2e_rec["hist_gb_per_s"], "link_frac": e2e_rec["link_frac"],
                         "ctas": e2e_ctas if e2e_ctas > 0 else n_sms, "what": "the e2e context"}
    rec["streamed_zero_copy"] = zc

    if full:
        # ---- restore then verify (the paper's K1 ablation point, SD+Offload): each layer's whole history is
        # copied to HBM first (one copy per request and tensor), then attended in place
        restore_k = [torch.empty_like(k, device=dev) for k in inp.layers[0]["kh_h"]]
        restore_v = [torch.empty_like(v_, device=dev) for v_ in inp.layers[0]["vh_h"]]
        restored, consumed = torch.cuda.Event(), torch.cuda.Event()
        consumed.record(cs)
        rs_pushes = inp.parts(restore_k, restore_v, True)
        v_rs = R.verifier()

        def restore_step():
            with torch.cuda.stream(cs):
                for ly in inp.layers:
                    ly["q_d"].copy_(ly["q_h"], non_blocking=True)
                    ly["kc_d"].copy_(ly["kc_h"], non_blocking=True)
                    ly["vc_d"].copy_(ly["vc_h"], non_blocking=True)
            for ly in inp.layers:
                xs.wait_event(consumed)  # the restore buffer is free once the previous layer was attended
                with torch.cuda.stream(xs):
                    for b in range(B):
                        if w.hist_len[b]:
                            restore_k[b].copy_(ly["kh_h"][b], non_blocking=True)
                            restore_v[b].copy_(ly["vh_h"][b], non_blocking=True)
                restored.record(xs)
                cs.wait_event(restored)
                R.round_of(v_rs, ly, rs_pushes)
                consumed.record(cs)
                with torch.cuda.stream(cs):
                    ly["o_h"].copy_(ly["o_d"], non_blocking=True)
                    ly["lse_h"].copy_(ly["lse_d"], non_blocking=True)
            cs.synchronize()

        ms_rs = R.timed(restore_step, steps, warmup)
        R.checked(v_rs, inp, rs_pushes)
        v_rs.close()
        val_rs, ms_rs_job = job_throughput(B * nq, ms_rs, world, dev)
        rec["restore_then_verify"] = {"value": val_rs, "unit": UNIT, "ms_per_step": ms_rs_job,
                                      "streamed_over_restore": ms_rs / ms_e2e,
                                      "what": "copy each layer's whole history to HBM, then attend (verification "
                                              "waits for the restore)"}
        del restore_k, restore_v

    # ---- Target priority: the streamed step again beside a low-priority Draft GEMM loop
    if with_tp:
        dl = DraftLoad(dev)
        dl.start()
        time.sleep(1.0)
        draft_alone = dl.stop()
        v_st = R.verifier(staged_ctas=a.staged_ctas, timing=True)
        st_rec, ms_st = streamed(v_st, stream_pushes, f"copy engine, staged chunk launches on {a.staged_ctas} CTAs")
        rec["streamed_copy_engine_staged"] = dict(st_rec, link_frac=st_rec["hist_gb_per_s"] / link_gbs)
        modes = [(e2e_name, v_e2e, whole_pushes, ms_e2e),
                 ("copy_engine", v_ce, stream_pushes, ms_ce),
                 (f"copy_engine_staged_{a.staged_ctas}_ctas", v_st, stream_pushes, ms_st)]
        for cap, (vz, zp, ms) in zc_ctx.items():
            if cap in (8, 32):  # the budgets that leave most SMs to a co-running Draft
                modes.append((f"in_place_{cap}_ctas", vz, zp, ms))
        tp = {"draft": "bf16 GEMM 4096^3, CUDA-graph replays of 8 on a lowest-priority stream",
              "draft_tflops_alone": draft_alone, "modes": {},
              "baseline": "each mode's Target steps timed alone right before its co-run"}
        tp_steps = max(3, min(steps, 10))

        def tp_n(ms_step):
            """Steps per timed region: at least tp_steps, and about a second of steps for short ones, so that
            one host hiccup does not decide a mean."""
            return max(tp_steps, min(200, int(math.ceil(1000.0 / max(ms_step, 1e-3)))))

        for name, vx, pushes, ms_mode in modes:
            timing = bool(vx.cfg.flags & 1)
            n = tp_n(ms_mode)
            ms_alone = R.timed(lambda vx=vx, pushes=pushes: R.host_step(vx, inp, lambda li: pushes[li]), n, 1)
            dl.start()
            time.sleep(0.2)
            ms_co = R.timed(lambda vx=vx, pushes=pushes: R.host_step(vx, inp, lambda li: pushes[li]), n, 1,
                            between=vx.window_reset if timing else None)
            tf = dl.stop()
            m = {"delta_T": (ms_co - ms_alone) / ms_alone, "target_ms_alone": ms_alone, "target_ms_co": ms_co,
                 "draft_tflops_co": tf, "steps": n}
            if timing:  # where the Target's time went beside the Draft: slower copies, or a stalled pipeline
                ws = vx.window_stats()
                cov = ws["n_rounds"] / L
                m["co_per_step_ms"] = {k: ws[k] / cov for k in ("copy_busy_ms", "copy_gap_ms", "chunk_kernel_ms",
                                                                "zero_copy_kernel_ms", "transfer_busy_ms")}
                ivx = vx.window_intervals()
                m["co_copy_rate_gbs"] = copy_rates(ivx, push_bytes * n) \
                    if pushes is stream_pushes and ws["n_rounds"] == n * L and len(ivx) == len(push_bytes) * n else None
            tp["modes"][name] = m
        # the same steps with Draft steps admitted by the scheduler instead of a free-running Draft (a new
        # scheduler per mode, each against its own baseline timed right before)
        tp["admission"] = {"draft": "one bf16 GEMM 4096^3 per Draft step, admitted per request by "
                                    "svx_sched_try_admit, checked by svx_sched_check_start, ACKed",
                           "modes": {}}
        for name, vx, pushes, ms_mode in modes:
            if name in ("copy_engine", e2e_name):
                continue  # in-place reads on few SMs and the copy engine's launches on a few SMs
            fn = (lambda vx=vx, pushes=pushes: R.host_step(vx, inp, lambda li: pushes[li]))
            n = tp_n(ms_mode)
            ms_alone = R.timed(fn, n, 1)
            _ms, rec_ad = run_admitted(R, fn, 2 * n, ms_alone, AdmittedDraft(dev, B))
            tp["admission"]["modes"][name] = rec_ad
        R.checked(v_st, inp, stream_pushes[0])
        v_st.close()
        rec["target_priority"] = tp
    for vz, _zp, _ms in zc_ctx.values():
        vz.close()
    v_e2e.close()
    v_ce.close()
    v_ad.close()
    rec["_inputs"] = inp
    return rec


def measure_width(a, dev, world, cs, xs, rounds=48, seed=7):
    """The I/O-aware dynamic verification width (section 4.2) on real rounds: the qwen3-shaped layer,
    history read in place from pinned host memory; each round runs at the width the library's controller
    chose (q drafts, q + 1 queries and candidates) and feeds it the round's measured kernel time (the
    transfer fused with the attention) plus a synthetic Draft cost and acceptance (no Draft model here):
    q x 0.3 ms to draft, 0.1 ms of rejection correction, each request's drafts accepted with probability
    0.75 each until the first rejection.  Reports the widths chosen and the committed tokens per second
    (all requests of the Cohort)."""
    import torch
    from speculative_decoding_verification_chunked_gb300 import svx
    widths, acc, t_tok, t_corr = [2, 4, 6, 8], 0.75, 0.3, 0.1
    w = W.named("qwen3").with_(n_query=max(widths) + 1)
    B, Hq, Hkv, d = w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim
    inp = Inputs(w, dev, resident=False)
    R = Runner(a, w, dev, world, cs, xs)
    ly = inp.layers[0]
    pushes = inp.parts(ly["kh_h"], ly["vh_h"], True)
    g = torch.Generator(device=dev).manual_seed(seed)
    per_q = {}
    for q in widths:
        nq = q + 1
        per_q[q] = dict(q=(torch.randn((B, Hq, nq, d), generator=g, device=dev)).to(torch.bfloat16),
                        kc=(torch.randn((B, nq, Hkv, d), generator=g, device=dev)).to(torch.bfloat16),
                        vc=(torch.randn((B, nq, Hkv, d), generator=g, device=dev)).to(torch.bfloat16),
                        o=torch.empty((B, Hq, nq, d), dtype=torch.bfloat16, device=dev),
                        lse=torch.empty((B, Hq, nq), dtype=torch.float32, device=dev))
    rng = np.random.default_rng(seed)
    ctl = svx.WidthController(widths, ema=0.5, threshold=0.05, n_init=3)
    v = R.verifier(zero_copy=True, zero_copy_ctas=a.e2e_ctas, timing=True)
    chosen, total_ms, committed = [], 0.0, 0.0
    for r in range(rounds):
        q = ctl.next_width()
        t = per_q[q]
        v.round_begin(t["q"], w.hist_len)
        v.candidate_attn(t["kc"], t["vc"])
        for p in pushes:
            v.push_raw(p)
        v.round_finish(t["o"], t["lse"], timeout_ms=60000 if r == rounds - 1 else 0)
        st = v.stats()
        # each request's drafts are accepted until the first rejection; it commits that prefix plus the
        # Target's own token; the controller sees the Cohort's mean
        ok = rng.random((B, q)) < acc
        per_req = 1.0 + np.where(ok.all(axis=1), q, np.argmin(ok, axis=1))
        u = float(per_req.mean())
        attn = st["chunk_kernel_ms"] + st["finish_kernel_ms"]
        ctl.record(q, q * t_tok, st["chunk_kernel_ms"], attn, t_corr, u)
        chosen.append(q)
        total_ms += q * t_tok + st["round_ms"] + t_corr
        committed += float(per_req.sum())
    v.close()
    costs = {q: ctl.cost(q) for q in widths}
    steady = chosen[len(widths) * 3:]
    return {"what": "dynamic verification width on the qwen3-shaped layer (in-place reads); Draft cost and "
                    "acceptance synthetic: q x 0.3 ms, 0.1 ms correction, acceptance 0.75 per draft",
            "rounds": rounds, "widths_chosen": {str(q): chosen.count(q) for q in widths},
            "after_sampling": {str(q): steady.count(q) for q in widths},
            "cost_ms_per_committed_token": {str(q): c for q, c in costs.items()},
            "committed_tokens_per_s": committed / (total_ms / 1e3)}


def measure_tiering(a, dev, world, cs, xs, rounds=40, seed=9, T=512, g=256):
    """Commit-aware tiering (section 4.1, Eqs. 4-5) beside streaming rounds: on the qwen3-shaped layer each
    request's Sealed History [0, H) is read in place from pinned host memory and its Active Tail [H, C)
    in place from HBM; after every round the accepted candidates (a seeded number, 1-5 per request) are
    committed to the tail, and whenever Eq. 5 moves the endpoint the rows [H, E) migrate to host memory
    on a side stream while the next rounds run; H advances once a migration has completed.  Reports the
    round time with and without migrations and the migration's device-to-host rate."""
    import torch
    from speculative_decoding_verification_chunked_gb300 import svx
    w = W.named("qwen3")
    B, Hq, Hkv, d, nq = w.n_req, w.n_q_heads, w.n_kv_heads, w.head_dim, w.n_query
    C0 = w.hist_len[0]
    tail0 = T + g  # initial Active Tail
    cap = C0 + 6 * rounds * 2
    row = Hkv * d
    inp = Inputs(w, dev, resident=False)
    R = Runner(a, w, dev, world, cs, xs)
    ly = inp.layers[0]
    bf = torch.bfloat16
    # host copy of each request's history (capacity for the committed growth), device tail buffers
    host_k = torch.zeros((B, cap, Hkv, d), dtype=bf, pin_memory=True)
    host_v = torch.zeros((B, cap, Hkv, d), dtype=bf, pin_memory=True)
    dev_k = torch.zeros((B, cap, Hkv, d), dtype=bf, device=dev)
    dev_v = torch.zeros((B, cap, Hkv, d), dtype=bf, device=dev)
    for b in range(B):
        host_k[b, :C0].copy_(ly["kh_h"][b])
        host_v[b, :C0].copy_(ly["vh_h"][b])
        dev_k[b, C0 - tail0:C0].copy_(ly["kh_h"][b][C0 - tail0:])
        dev_v[b, C0 - tail0:C0].copy_(ly["vh_h"][b][C0 - tail0:])
    torch.cuda.synchronize(dev)
    rb = row * 2
    mig_stream = torch.cuda.Stream(device=dev)
    rng = np.random.default_rng(seed)
    v = R.verifier(zero_copy=True, zero_copy_ctas=a.e2e_ctas)

    def run(migrate: bool):
        tiers = [svx.Tier(C0 - tail0, C0 - tail0, C0 - tail0) for _ in range(B)]
        for tr in tiers:
            tr.round(C0, C0 + nq)
        times, moved, mig_events = [], 0, []
        for r in range(rounds):
            hist = [tr.C for tr in tiers]
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cs)
            v.round_begin(ly["q_d"], hist)
            v.candidate_attn(ly["kc_d"], ly["vc_d"])
            v.push_raw([(b, 0, tr.H, host_k[b].data_ptr(), host_v[b].data_ptr()) for b, tr in enumerate(tiers)])
            v.push_raw([(b, tr.H, tr.C - tr.H, dev_k[b, tr.H].data_ptr(), dev_v[b, tr.H].data_ptr())
                        for b, tr in enumerate(tiers)])
            v.round_finish(ly["o_d"], ly["lse_d"], timeout_ms=60000 if r == rounds - 1 else 0)
            e1.record(cs)
            # commit: the accepted candidates' KV joins the Active Tail (the rejected ones are released)
            acc = rng.integers(1, nq + 1, size=B)
            with torch.cuda.stream(cs):
                for b, tr in enumerate(tiers):
                    c = tr.C
                    dev_k[b, c:c + acc[b]].copy_(ly["kc_d"][b, :acc[b]])
                    dev_v[b, c:c + acc[b]].copy_(ly["vc_d"][b, :acc[b]])
                    tr.commit(c + int(acc[b]))
                    tr.round(tr.C, tr.C + nq)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
            if migrate:
                for b, tr in enumerate(tiers):
                    if tr.pending is not None:
                        tr.poll()
                    if tr.pending is None:
                        m0 = torch.cuda.Event(enable_timing=True)
                        m1 = torch.cuda.Event(enable_timing=True)
                        mig_stream.wait_stream(cs)  # the committed rows are written
                        m0.record(mig_stream)
                        H = tr.H
                        E = tr.migrate(T, g, rb, dev_k[b, H].data_ptr(), dev_v[b, H].data_ptr(), host_k[b].data_ptr(),
                                       host_v[b].data_ptr(), stream=mig_stream)
                        m1.record(mig_stream)
                        if E > H:
                            moved += 2 * (E - H) * rb
                            mig_events.append((m0, m1))
        torch.cuda.synchronize(dev)
        for tr in tiers:
            if tr.pending is not None:
                tr.release()
        mig_ms = sum(m0.elapsed_time(m1) for m0, m1 in mig_events)
        return statistics.median(times), moved, mig_ms, len(mig_events), tiers

    ms_plain, _, _, _, _ = run(False)
    ms_tier, moved, mig_ms, n_mig, tiers = run(True)
    v.close()
    return {"what": "rounds on the qwen3-shaped layer with the Sealed History read in place from host and the "
                    "Active Tail from HBM, accepted candidates committed each round; with and without "
                    "asynchronous Eq. 5 migrations of [H, E) to host memory (T = 512, g = 256)",
            "rounds": rounds, "round_ms_median_without_migration": ms_plain,
            "round_ms_median_with_migration": ms_tier, "slowdown": ms_tier / ms_plain - 1.0,
            "migrations": n_mig, "migrated_bytes": int(moved),
            "migration_gb_per_s": moved / (mig_ms / 1e3) / 1e9 if mig_ms > 0 else None,
            "final_H": [tr.H for tr in tiers], "final_C": [tr.C for tr in tiers]}


def main(argv=None):
    a = parse_args(argv)
    rank, world, local = dist_init()
    if a.impl == "reference":
        return run_reference(a, rank, world)

    import multiprocessing as mp
    w = workload_of(a)
    w = w.with_(seed=w.seed + 1000 * rank)
    do_cpu = rank == 0 and world == 1 and not a.no_cpu_baseline
    cores = os.cpu_count() or 1
    pool = None
    if do_cpu:  # the oracle's process pool is started (spawn) before the first GPU call
        pool = mp.get_context("spawn").Pool(cores)

    import torch
    from speculative_decoding_verification_chunked_gb300 import svx  # noqa: F401  (fails loudly if unbuilt)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    hbm_peak = float(peaks.get("hbm_gbs") or FALLBACK_HBM_GBS)
    hbm_src = "measured" if peaks.get("hbm_gbs") else "fallback"
    cs = torch.cuda.Stream(device=dev, priority=-1)
    xs = torch.cuda.Stream(device=dev, priority=-1)

    if a.profile_in_place:  # the e2e context's launches alone (the first chunk launch is the first in-place one)
        inp = Inputs(w, dev, resident=False)
        R = Runner(a, w, dev, world, cs, xs)
        vz = R.verifier(zero_copy=True, zero_copy_ctas=a.e2e_ctas)
        pushes = [inp.parts(ly["kh_h"], ly["vh_h"], True) for ly in inp.layers]
        ms = R.timed(lambda: R.host_step(vz, inp, lambda li: pushes[li]), a.steps, a.warmup)
        R.checked(vz, inp, pushes[0])
        vz.close()
        if rank == 0:
            print(json.dumps({"profile_in_place": True, "ms_per_step": ms, "ctas": a.e2e_ctas,
                              "hist_gb_per_s": w.hist_bytes * w.n_layers / (ms / 1e3) / 1e9,
                              "config": workload_config(w, a)}))
        return 0
    clk = ClockSampler(local).__enter__()  # sampled over every timed region
    head = measure(a, w, dev, world, cs, xs, hbm_peak, hbm_src, full=True)
    inp = head.pop("_inputs")
    cpu = None
    if do_cpu:  # the oracle on a bounded sample of the headline step (layer 0's inputs as drawn)
        n_pairs = min(a.cpu_sample_pairs or cores, w.n_req * w.n_kv_heads)
        tasks = oracle_tasks(w, inp.oracle_layer0(), cpu_sample_pairs(w, n_pairs))
        s = oracle_sample(pool, tasks, w, w.n_layers)
        cpu = {"value": s["value"], "unit": UNIT, "cores": min(cores, len(tasks)), "kind": "oracle",
               "sample": f"{len(tasks)} of {w.n_layers * w.n_req * w.n_kv_heads} (layer, request, KV head) pairs of "
                         f"one step in {s['seconds']:.1f} s (a {s['step_fraction']:.4f} fraction of the step); value "
                         f"= that fraction of the step's tokens over the sample's time"}
        pool.close()
    del inp
    gc.collect()  # the headline's pinned history is freed here, not in a later timed region
    torch.cuda.empty_cache()
    subs = {}
    for name in [n.strip() for n in a.sub_workloads.split(",") if n.strip()]:
        if name == w.name:
            continue
        ws = W.named(name)
        ws = ws.with_(seed=ws.seed + 1000 * rank)
        r = measure(a, ws, dev, world, cs, xs, hbm_peak, hbm_src, full=False)
        r.pop("_inputs")
        gc.collect()
        torch.cuda.empty_cache()
        subs[name] = r
    method = {}
    for key, fn in ((("dynamic_width", measure_width), ("tiering", measure_tiering)) if a.method else ()):
        try:
            method[key] = fn(a, dev, world, cs, xs)
        except Exception as e:  # a failing sub-record is reported, not silently dropped
            method[key] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
    clk.__exit__(None, None, None)
    clocks = clk.summary()

    out = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": head["steps"],
           "warmup": head["warmup"], "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": head["config"],
           "e2e": head["e2e"], "gpu_launches": head["launches_per_step"] * head["steps"],
           "roofline": head["roofline"], "clocks": clocks}
    for k in ("streamed", "streamed_copy_engine", "streamed_adaptive", "streamed_copy_engine_staged", "resident",
              "restore_then_verify", "streamed_zero_copy", "target_priority"):
        if k in head:
            out[k] = head[k]
    if cpu:
        out["cpu_baseline"] = cpu
    if subs:
        out["workloads"] = subs
    out["method"] = method
    out["pages_context"] = PAGES_CONTEXT
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def code_digest(path: str) -> str:
    """sha256 of a CUDA source with its // comments, trailing blanks and empty lines removed, so that
    an edit of comments alone does not mark the counters taken on it as stale."""
    import hashlib
    import re
    lines = []
    for line in open(path, encoding="utf-8"):
        line = re.sub(r"//.*$", "", line.rstrip("\n")).rstrip()
        if line:
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def profiled_traffic(w: W.Workload):
    """DRAM bytes per launch of the tensor-core chunk kernel on this workload from the committed ncu
    summary, if that summary was taken on the kernel source as it is now (else None)."""
    src = os.path.join(ROOT, "speculative_decoding_verification_chunked_gb300", "csrc", "svx_tc_kernel.cu")
    summ = os.path.join(ROOT, "profiles", "chunk_attn_tc_traffic.txt")
    try:
        kv = {k.strip(): v.strip() for k, v in
              (line.split(":", 1) for line in open(summ) if ":" in line and not line.startswith("#"))}
        if kv.get("kernel_code_sha256", "") != code_digest(src):
            return None
        key = w.name if w.head_dim == 128 else f"{w.name}_d{w.head_dim}"
        return float(kv[f"{key}.dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


if __name__ == "__main__":
    sys.exit(main())
