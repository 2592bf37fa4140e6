#!/usr/bin/env python
"""LOCKS decode-step benchmark on GB300.

One step = one pass of the whole decode hot path over one batch: summary-only
page scoring of every page, group-shared top-k selection, and sparse attention
over the kept pages (the two kernels ``locks_decode_step`` launches, called here
as ``locks_score_pages`` + ``locks_select_attend`` so that the scoring kernel can
be bracketed by CUDA events inside the timed region).

Default workload: the 1M-token context, batch 1, 32 query / 8 kv heads,
budget 2048 tokens (``--workload`` / ``--budget`` select the others). Inputs
are synthetic (the seeded generator in ``synth``) and resident in HBM when the
timed region starts; L2 is flushed (512 MiB write) between timed steps.

Prints ONE JSON line (rank 0). ``--impl reference`` times the float64 CPU
oracle on the host cores instead (the reference arm of this project).
Multi-GPU (torchrun): every rank runs an independent replica of the workload
(the step has no cross-request exchange); timing is the max over ranks.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode-step µs and effective HBM GB/s (% of GB300 roofline) at 128K–1M ctx"
UNIT_BYTES = 776                 # summary bytes per (page, kv head)
PAGE_KV_BYTES = 2 * 16 * 128 * 2  # K + V bytes per (page, kv head)
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------- distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    os.environ.setdefault("MASTER_PORT", "29533")
    dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clock, power and clock-event reasons through NVML (read-only) in a thread."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, uuid: str | None, period_s: float = 0.002):
        self.samples = []
        self.period = period_s
        self.ok = False
        self._stop = threading.Event()
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            r = -1
            if uuid:
                r = self.nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h))
            if r != 0:
                idx = int(os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0] or 0)
                r = self.nv.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(self.h))
            if r != 0:
                return
            mx = ctypes.c_uint()
            rc = self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.max_mhz = float(mx.value) if rc == 0 else None
            fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None)
            self._reasons_fn = fn or self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except OSError:
            self.ok = False

    def _one(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        pw = ctypes.c_uint()
        self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk))
        self._reasons_fn(self.h, ctypes.byref(rs))
        self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(pw))
        self.samples.append((float(clk.value), int(rs.value), pw.value / 1000.0))

    def _loop(self):
        while not self._stop.is_set():
            self._one()
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self._t = threading.Thread(target=self._loop, daemon=True)
            self._t.start()

    def stop(self):
        if self.ok:
            self._stop.set()
            self._t.join()
            self._one()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        clocks = [s[0] for s in self.samples]
        bits = 0
        for s in self.samples:
            bits |= s[1]
        reasons = [name for bit, name in self.REASONS.items() if bits & bit]
        return {"sm_mhz": statistics.median(clocks), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "power_w_max": max(s[2] for s in self.samples)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    from sparse_kv_page_gb300 import build as B
    ent = rec.get(kernel)
    if not ent:
        return None
    try:
        if ent.get("source_hash") != B.source_hash(ent.get("sources", []))[:16]:
            return None   # the kernel changed since the counters were taken
    except OSError:
        return None
    return ent


# ----------------------------------------------------------------- workload

def workload_of(args) -> tuple[synth.Workload, int]:
    w = synth.WORKLOADS[args.workload]
    if args.pages is not None:
        w = w.scaled(pages=args.pages, name_suffix=f"-{args.pages}p")
    budget = args.budget if args.budget is not None else max(w.budgets)
    return w, budget


def algorithmic_bytes(w: synth.Workload, budget: int) -> tuple[int, int]:
    units = w.batch * w.pages * w.num_kv_heads
    k = min(budget // 16, w.pages)
    return units * UNIT_BYTES, w.batch * w.num_kv_heads * k * PAGE_KV_BYTES


def units_of(w: synth.Workload) -> int:
    """(physical page, kv head) units of the workload's cache."""
    return w.num_phys_pages * w.num_kv_heads


def config_of(w: synth.Workload, budget: int) -> dict:
    return {"workload": f"{w.name}: {w.description}", "batch": w.batch, "context_tokens": w.context,
            "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": 128, "page_size": 16,
            "rank": 8, "budget_tokens": budget, "pages_per_seq": w.pages,
            "l2": "flushed between timed steps (512 MiB write, outside the step events)"}


# ---------------------------------------------------------- oracle (CPU) arm

class OracleStep:
    """The float64 oracle's decode step on one (request, kv head) segment per call.

    A full step is every segment; one call times one segment (scores of all its
    pages for the group's query heads, group keys, selection, attention) and the
    per-step figure is that time times the number of segments, so a step stays
    bounded. Summary bytes are random (the oracle's cost does not depend on
    their values)."""

    def __init__(self, w: synth.Workload, budget: int, inp: synth.DecodeInputs):
        import oracle
        oracle.build()
        self.o = oracle
        self.w, self.budget, self.inp = w, budget, inp
        s = synth.random_summaries(w.num_phys_pages, w.num_kv_heads, seed=12345)
        self.seg = []
        for b in range(w.batch):
            for kvh in range(w.num_kv_heads):
                self.seg.append((b, kvh))
        self.per_kvh = [tuple(np.ascontiguousarray(a[:, kvh:kvh + 1]) for a in (s.mu, s.basis, s.coef, s.scales))
                        for kvh in range(w.num_kv_heads)]
        self.i = 0

    def run_one(self) -> float:
        """Seconds for one segment."""
        w, o = self.w, self.o
        b, kvh = self.seg[self.i % len(self.seg)]
        self.i += 1
        g = w.group
        q = np.ascontiguousarray(self.inp.q[b:b + 1, kvh * g:(kvh + 1) * g])
        table = np.ascontiguousarray(self.inp.page_table[b:b + 1])
        seq = self.inp.seq_pages[b:b + 1]
        mu, basis, coef, scales = self.per_kvh[kvh]
        t0 = time.perf_counter()
        s = o.scores(q, mu, basis, coef, scales, table, seq, 1)
        keys, _ = o.group_keys(s, seq, 1)
        sel, nsel = o.select(keys, seq, self.budget)
        t1 = time.perf_counter()
        full_sel = np.zeros((1, w.num_kv_heads, sel.shape[2]), np.int32)
        full_n = np.zeros((1, w.num_kv_heads), np.int32)
        full_sel[0, kvh] = sel[0, 0]
        full_n[0, kvh] = nsel[0, 0]
        qb = np.ascontiguousarray(self.inp.q[b:b + 1])
        t2 = time.perf_counter()
        o.attend(qb, self.inp.k_cache, self.inp.v_cache, table, full_sel, full_n)
        t3 = time.perf_counter()
        return (t1 - t0) + (t3 - t2)

    @property
    def segments(self) -> int:
        return len(self.seg)

    def cores(self) -> int:
        return self.o.max_threads()


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the baseline record."""
    import subprocess
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(step: OracleStep, budget_s: float = 12.0, max_calls: int = 64, single_s: float = 4.0) -> dict:
    def sample(seconds: float, calls: int) -> list:
        times = []
        t_end = time.perf_counter() + seconds
        while len(times) < calls and (not times or time.perf_counter() < t_end):
            times.append(step.run_one())
        return times

    cores = step.cores()
    times = sample(budget_s, max_calls)
    per_step_us = statistics.mean(times) * step.segments * 1e6
    # the same on one thread (a shorter bounded sample)
    step.o.set_threads(1)
    try:
        single = sample(single_s, 8)
    finally:
        step.o.set_threads(cores)
    return {"value": per_step_us, "unit": "us", "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{len(times)} of the step's {step.segments} (request, kv head) segments, each fully "
                      f"scored/selected/attended in float64; per-step time = mean segment time x segments; "
                      f"random summary bytes of the same shape",
            "single_thread": {"value": statistics.mean(single) * step.segments * 1e6, "unit": "us", "cores": 1,
                              "sample": f"{len(single)} segments, extrapolated the same way"}}


def run_reference(args, rank, world):
    if rank != 0:
        return
    w, budget = workload_of(args)
    inp = synth.make_decode_inputs(w, workers=min(16, os.cpu_count() or 1))
    step = OracleStep(w, budget, inp)
    for _ in range(args.warmup):
        step.run_one()
    times = [step.run_one() * step.segments * 1e6 for _ in range(args.steps)]
    value = statistics.mean(times)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "us", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1000.0, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, budget),
            "cpu_baseline": {"value": value, "unit": "us", "cores": step.cores(), "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": f"each step = one (request, kv head) segment of {step.segments}, "
                                       f"extrapolated x{step.segments}"},
            "e2e": {"value": value, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------------- GPU arm

def run_locks(args, rank, world, local):
    w, budget = workload_of(args)
    workers = min(16, os.cpu_count() or 1)
    inp = synth.make_decode_inputs(w, workers=workers)      # before any CUDA call (spawn pool)
    want_cpu = (rank == 0 and world == 1 and not args.no_cpu_baseline)
    cpu = cpu_baseline(OracleStep(w, budget, inp)) if want_cpu else None

    import torch
    import sparse_kv_page_gb300 as L
    from sparse_kv_page_gb300 import build as B
    B.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init(world, "nccl")
    L.load_library()

    def up(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(dev)

    q = up(inp.q)
    kc = up(inp.k_cache)
    vc = up(inp.v_cache)
    table = up(inp.page_table)
    seq = up(inp.seq_pages)
    del inp.k_cache, inp.v_cache
    dims = L.make_dims(w.batch, w.num_q_heads, w.num_kv_heads, w.pages, w.num_phys_pages)
    summ = L.Summaries.empty(w.num_phys_pages, w.num_kv_heads, dev)
    ids = torch.arange(w.num_phys_pages, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    # summary build (off the decode critical path): warm once, time once
    L.locks_build_summaries(dims, kc, ids, w.num_phys_pages, summ)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    L.locks_build_summaries(dims, kc, ids, w.num_phys_pages, summ)
    e1.record(stream)
    torch.cuda.synchronize()
    build_ms = e0.elapsed_time(e1)

    # the summary build at the GLM-4-9B-shaped 4 x 1M configuration (262,144 pages x 2 kv
    # heads of N(0,1) bf16 keys drawn on the device), timed as prefill pages/s
    glm = synth.WORKLOADS["glm9b_4x1m"]
    glm_pages = glm.batch * glm.pages
    glm_dims = L.make_dims(glm.batch, glm.num_q_heads, glm.num_kv_heads, glm.pages, glm_pages)
    gk = torch.randn((glm_pages, glm.num_kv_heads, 16, 128), device=dev, dtype=torch.bfloat16).view(torch.int16)
    gsumm = L.Summaries.empty(glm_pages, glm.num_kv_heads, dev)
    gids = torch.arange(glm_pages, dtype=torch.int32, device=dev)
    L.locks_build_summaries(glm_dims, gk, gids, glm_pages, gsumm)
    torch.cuda.synchronize()
    e0.record(stream)
    L.locks_build_summaries(glm_dims, gk, gids, glm_pages, gsumm)
    e1.record(stream)
    torch.cuda.synchronize()
    glm_build_ms = e0.elapsed_time(e1)
    del gk, gsumm, gids
    torch.cuda.empty_cache()

    k_cap = L.locks_k_cap(dims, budget)
    ws = L.alloc_workspace(dims, budget, dev)
    scores = torch.empty((w.batch, w.num_q_heads, w.pages), dtype=torch.float32, device=dev)
    sel = torch.empty((w.batch, w.num_kv_heads, k_cap), dtype=torch.int32, device=dev)
    nsel = torch.empty((w.batch, w.num_kv_heads), dtype=torch.int32, device=dev)
    out = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.int16, device=dev)
    lse = torch.empty((w.batch, w.num_q_heads), dtype=torch.float32, device=dev)
    partials = torch.empty(L.locks.lse_partials_shape(dims), dtype=torch.float32, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    # the two kernels locks_decode_step launches (scores + LSE partials, then selection + attention)
    def score():
        L.locks_score_pages(dims, q, summ, table, seq, scores, ws, lse_partials=partials)

    def select_attend():
        L.locks_select_attend(dims, q, kc, vc, table, scores, seq, budget, sel, nsel, out, lse, ws,
                              lse_partials=partials)

    # eager warm-up (first-call set-up), then CUDA graphs: the whole step (the two kernels
    # locks_decode_step launches, the selection programmatically dependent on the scorer) for
    # the timed steps, and one graph per kernel for the per-kernel breakdown
    score()
    select_attend()
    torch.cuda.synchronize()
    g_score, g_sa, g_step = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_score):
        score()
    with torch.cuda.graph(g_sa):
        select_attend()
    with torch.cuda.graph(g_step):
        score()
        select_attend()
    for _ in range(args.warmup):
        flush.zero_()
        g_step.replay()
        flush.zero_()
        g_score.replay()
        g_sa.replay()
    torch.cuda.synchronize()
    assert L.locks_get_device_status(ws) == 0, "device status after warm-up"

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    evk = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    t0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        evs[i][0].record(stream)
        g_step.replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    # per-kernel breakdown: the same K steps with an event between the two kernels
    for i in range(K):
        flush.zero_()
        evk[i][0].record(stream)
        g_score.replay()
        evk[i][1].record(stream)
        g_sa.replay()
        evk[i][2].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    sampler.stop()
    status = L.locks_get_device_status(ws)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    score_ms = [a.elapsed_time(b) for a, b, _ in evk]
    sa_ms = [b.elapsed_time(c) for _, b, c in evk]
    split_ms = [a.elapsed_time(c) for a, _, c in evk]
    mean_step_us = reduce_max(statistics.mean(step_ms) * 1000.0, world, dev)
    mean_score_us = reduce_max(statistics.mean(score_ms) * 1000.0, world, dev)
    mean_sa_us = reduce_max(statistics.mean(sa_ms) * 1000.0, world, dev)

    # end to end through the public call with host buffers: q in, output out
    q_host = torch.from_numpy(np.ascontiguousarray(synth.make_queries(w))).pin_memory()
    out_host = torch.empty(out.shape, dtype=torch.int16).pin_memory()
    n_e2e = min(K, 200)

    def e2e_step():
        q.copy_(q_host, non_blocking=True)
        L.locks_decode_step(dims, q, kc, vc, summ, table, seq, budget, out, ws, lse=lse)
        out_host.copy_(out, non_blocking=True)

    # the step as a serving loop runs it: copy-in, the decode step and copy-out captured in one
    # CUDA graph (the library's calls are graph-capturable), replayed and synchronised per step;
    # and the same three calls issued eagerly through the C ABI each step
    e2e_step()
    torch.cuda.synchronize()
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e):
        e2e_step()
    e2e_us, e2e_eager_us = [], []
    for run, acc in ((g_e2e.replay, e2e_us), (e2e_step, e2e_eager_us)):
        for i in range(n_e2e + 3):
            flush.zero_()
            torch.cuda.synchronize()
            t1 = time.perf_counter()
            run()
            torch.cuda.synchronize()
            if i >= 3:
                acc.append((time.perf_counter() - t1) * 1e6)
    e2e_value = reduce_max(statistics.mean(e2e_us), world, dev)
    e2e_eager = reduce_max(statistics.mean(e2e_eager_us), world, dev)

    # full-model decode graph (outside the timed region): 32 layers' decode steps
    # (locks_decode_step each) in one CUDA graph, every layer with its own query, K/V cache,
    # summaries, workspace and outputs (the page table is shared, as one block table serves
    # every layer). The caches hold N(0,1) bf16 keys and values drawn on the device and the
    # summaries are built from them; as many distinct layers as fit in 60% of the free
    # memory, layer i using set i mod n_distinct.
    model_graph = None
    if not args.no_model_graph:
        n_layers = 32
        kv_bytes_layer = 2 * kc.numel() * 2
        per_layer = kv_bytes_layer + units_of(w) * UNIT_BYTES + L.locks_workspace_size(dims, budget) + (1 << 20)
        free = torch.cuda.mem_get_info(dev)[0]
        n_distinct = max(2, min(n_layers, int(0.6 * free // per_layer)))
        gen = torch.Generator(device=dev)
        gen.manual_seed(4321)
        sets = []
        for i in range(n_distinct):
            kc_i = torch.randn(tuple(kc.shape), generator=gen, device=dev, dtype=torch.bfloat16).view(torch.int16)
            vc_i = torch.randn(tuple(vc.shape), generator=gen, device=dev, dtype=torch.bfloat16).view(torch.int16)
            summ_i = L.Summaries.empty(w.num_phys_pages, w.num_kv_heads, dev)
            L.locks_build_summaries(dims, kc_i, ids, w.num_phys_pages, summ_i)
            sets.append(dict(q=torch.randn(tuple(q.shape), generator=gen, device=dev), kc=kc_i, vc=vc_i,
                             summ=summ_i, ws=L.alloc_workspace(dims, budget, dev), out=torch.empty_like(out),
                             lse=torch.empty_like(lse)))
        torch.cuda.synchronize()

        def model_step():
            for layer in range(n_layers):
                z = sets[layer % n_distinct]
                L.locks_decode_step(dims, z["q"], z["kc"], z["vc"], z["summ"], table, seq, budget, z["out"],
                                    z["ws"], lse=z["lse"])

        model_step()
        torch.cuda.synchronize()
        g_model = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_model):
            model_step()
        g_model.replay()
        torch.cuda.synchronize()
        m_us = []
        for i in range(5):
            flush.zero_()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            g_model.replay()
            b_.record(stream)
            torch.cuda.synchronize()
            if i >= 1:
                m_us.append(a_.elapsed_time(b_) * 1000.0)
        model_us = reduce_max(statistics.mean(m_us), world, dev)
        model_graph = {"layers": n_layers, "distinct_layer_sets": n_distinct, "us": model_us,
                       "per_layer_us": model_us / n_layers,
                       "per_layer_vs_single_step": (model_us / n_layers) / mean_step_us, "replays": len(m_us),
                       "path": f"32 x locks_decode_step captured in one CUDA graph, L2 flushed before each "
                               f"replay; each layer has its own query, K/V cache (N(0,1) bf16 drawn on the "
                               f"device), summaries built from it, workspace and outputs: {n_distinct} distinct "
                               f"sets, layer i using set i mod {n_distinct} (layers sharing a set are "
                               f"{n_distinct} apart); the page table is shared by every layer"}
        for z in sets:
            assert L.locks_get_device_status(z["ws"]) == 0, "device status after the model graph"
        del sets
        torch.cuda.empty_cache()

    # page-fill refresh (outside the timed region): the one-page summary build a filled page
    # needs, alone and overlapped with a decode step on a second stream
    refresh = None
    if not args.no_model_graph:
        side = torch.cuda.Stream()
        one = ids[:1].clone()                                        # physical page 0
        fresh = L.Summaries.empty(1, w.num_kv_heads, dev)            # its new summary (not read by the step)
        L.locks_build_summaries(dims, kc, one, 1, fresh)
        # the step a caller runs while pages fill: locks_decode_step_tail (no tail tokens here),
        # whose scorer leaves one SM to the concurrent one-page builds
        tails = torch.zeros(w.batch, dtype=torch.int32, device=dev)

        def tail_step():
            L.locks_decode_step(dims, q, kc, vc, summ, table, seq, budget, out, ws, lse=lse, tail_tokens=tails)

        tail_step()
        torch.cuda.synchronize()
        g_tail = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_tail):
            tail_step()
        torch.cuda.synchronize()
        alone, with_refresh, plain = [], [], []
        for i in range(12):
            flush.zero_()
            torch.cuda.synchronize()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(side)
            L.locks_build_summaries(dims, kc, one, 1, fresh, stream=side)
            b_.record(side)
            torch.cuda.synchronize()
            # three consecutive steps, then the same with the one-page build launched on the
            # second stream right after the first step's kernels are queued
            for with_build, acc in ((False, plain), (True, with_refresh)):
                flush.zero_()
                torch.cuda.synchronize()
                c_, d_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                c_.record(stream)
                for k in range(3):
                    g_tail.replay()
                    if with_build and k == 0:
                        side.wait_stream(stream)
                        with torch.cuda.stream(side):
                            L.locks_build_summaries(dims, kc, one, 1, fresh, stream=side)
                d_.record(stream)
                torch.cuda.synchronize()
                if i >= 2:
                    acc.append(c_.elapsed_time(d_) * 1000.0)
            if i >= 2:
                alone.append(a_.elapsed_time(b_) * 1000.0)
        refresh = {"build_one_page_us": statistics.mean(alone), "three_steps_us": statistics.mean(plain),
                   "three_steps_with_refresh_us": statistics.mean(with_refresh),
                   "refresh_cost_us": statistics.mean(with_refresh) - statistics.mean(plain),
                   "samples": len(alone),
                   "tail_step_us": statistics.mean(plain) / 3.0,
                   "path": "locks_build_summaries(n_pages=1) for a page that just filled, on a second stream, "
                           "launched after the first of three consecutive steps is queued (the page stays in "
                           "the tail, attended whole, until the build completes); the steps are "
                           "locks_decode_step_tail in one graph each (its scorer leaves one SM to the build); "
                           "refresh_cost_us = the three steps' extra time"}
        assert L.locks_get_device_status(ws) == 0, "device status after the refresh timing"

    # dense comparator (outside the timed region): the same attention kernel with every page
    # of every sequence selected, i.e. exact attention over the whole cache
    dense = None
    if not args.no_dense:
        k_cap_all = L.locks_k_cap(dims, w.pages * 16)
        sel_all = torch.arange(w.pages, dtype=torch.int32, device=dev).repeat(w.batch * w.num_kv_heads, 1)
        sel_all = sel_all.view(w.batch, w.num_kv_heads, w.pages)[:, :, :k_cap_all].contiguous()
        nsel_all = seq.view(-1, 1).repeat(1, w.num_kv_heads).to(torch.int32).contiguous()
        out_d = torch.empty_like(out)

        def dense_attention():
            L.locks_sparse_attention(dims, q, kc, vc, table, sel_all, nsel_all, k_cap_all, out_d, None, ws)

        dense_attention()
        g_dense = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_dense):
            dense_attention()
        n_dense = max(3, min(K, 20))
        d_us = []
        for i in range(n_dense + 2):
            flush.zero_()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            g_dense.replay()
            b_.record(stream)
            torch.cuda.synchronize()
            if i >= 2:
                d_us.append(a_.elapsed_time(b_) * 1000.0)
        dense_us = reduce_max(statistics.mean(d_us), world, dev)
        dense_bytes = int(inp.seq_pages.astype(np.int64).sum()) * w.num_kv_heads * PAGE_KV_BYTES
        dense = {"attention_us": dense_us, "kv_bytes": dense_bytes, "GBps": dense_bytes / (dense_us * 1e-6) / 1e9,
                 "steps": n_dense, "locks_step_speedup": dense_us / mean_step_us,
                 "path": "locks_sparse_attention with every page selected (exact attention over the whole cache, "
                         "same attention kernel), one CUDA graph, L2 flushed before each"}
        assert L.locks_get_device_status(ws) == 0, "device status after the dense comparator"

    # selector ablations (outside the timed region): recall, attention mass and carrier retention of
    # the shipped summary, other ranks / code widths and shared bases against the exact selection
    ablation = None
    if rank == 0 and not args.no_ablation:
        from sparse_kv_page_gb300 import ablation as AB
        ablation = AB.run(dims, q, kc, table, seq, summ, budget, inp.carriers, dev)

    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    if dense:
        dense["frac_of_measured_hbm"] = dense["GBps"] / hbm
    summ_bytes, kv_bytes = algorithmic_bytes(w, budget)
    step_bytes = summ_bytes + kv_bytes
    score_gbs = summ_bytes / (mean_score_us * 1e-6) / 1e9
    step_gbs = step_bytes / (mean_step_us * 1e-6) / 1e9
    traffic = recorded_traffic("score_kernel")
    clocks = sampler.summary()
    units = w.batch * w.pages * w.num_kv_heads
    line = {
        "metric": METRIC, "value": mean_step_us, "unit": "us", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": mean_step_us / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "int4/int8 codes x f16 MMA, fp32 accumulate; bf16 K/V",
        "data": "synthetic (seeded page-local low-rank keys, N(0,1) values and queries)",
        "config": config_of(w, budget),
        "effective_GBps": step_gbs, "algorithmic_bytes_per_step": step_bytes,
        "frac_of_measured_hbm": step_gbs / hbm, "frac_of_8TBps": step_gbs / NOMINAL_HBM_GBS,
        "aggregate_effective_GBps": step_gbs * world,
        "kernels_us": {"score_pages": mean_score_us, "select_attend": mean_sa_us,
                       "step_p50": statistics.median(step_ms) * 1000.0,
                       "step_two_graphs": statistics.mean(split_ms) * 1000.0},
        "bytes_vs_dense": (w.batch * w.pages * w.num_kv_heads * PAGE_KV_BYTES) / step_bytes,
        "dense_comparator": dense,
        "model_graph": model_graph,
        "page_refresh": refresh,
        "ablation": ablation,
        "roofline": {"kernel": "score_pages (locks_score_pages)", "bound": "hbm", "achieved": score_gbs,
                     "peak": hbm, "peak_kind": f"{peak_kind} copy bandwidth", "unit": "GB/s",
                     "frac": score_gbs / hbm,
                     "algorithmic_bytes_per_launch": summ_bytes, "units_per_launch": units,
                     "traffic": traffic["dram_bytes_per_launch"] if traffic else None,
                     "traffic_source": traffic["source"] if traffic else None},
        "roofline_select_attend": {
            "kernel": "select_attend (the decode step's second launch: group keys, top-k, sparse attention)",
            "bound": "hbm", "achieved": kv_bytes / (mean_sa_us * 1e-6) / 1e9, "peak": hbm,
            "peak_kind": f"{peak_kind} copy bandwidth", "unit": "GB/s",
            "frac": kv_bytes / (mean_sa_us * 1e-6) / 1e9 / hbm,
            "algorithmic_bytes_per_launch": kv_bytes,
            "algorithmic_bytes": "selected K/V: 8 KiB per kept (page, kv head)",
            "l2_resident_bytes_per_launch": w.batch * w.num_q_heads * w.pages * 4 + L.locks_lse_partials_size(dims),
            "l2_resident_bytes": "the score table and LSE partials the scorer just wrote (read from L2)",
            "traffic": None},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "us", "h2d_bytes_per_step": int(q_host.numel() * 4),
                "d2h_bytes_per_step": int(out_host.numel() * 2),
                "path": "pinned q -> locks_decode_step -> output to pinned host, the three captured in one CUDA "
                        "graph, replayed and synchronised each step, wall clock",
                "eager_us": e2e_eager, "eager_path": "the same three calls issued eagerly through the C ABI "
                                                    "(ctypes) each step, synchronised, wall clock"},
        "launch": "timed steps: one CUDA graph per step (score_pages, then select_attend launched "
                  "programmatically dependent on it), L2 flushed before each; kernels_us: a second pass of "
                  "K steps with one graph per kernel and an event between them",
        "clocks": clocks, "gpu_launches": 2 * K, "device_status": status,
        "timed_wall_s": wall,
        "build": {"units": units, "ms": build_ms, "pages_per_s": w.batch * w.pages / (build_ms * 1e-3),
                  "units_per_s": units / (build_ms * 1e-3),
                  "glm9b_4x1m_prefill": {"pages": glm_pages, "kv_heads": glm.num_kv_heads, "ms": glm_build_ms,
                                         "pages_per_s": glm_pages / (glm_build_ms * 1e-3),
                                         "units_per_s": glm_pages * glm.num_kv_heads / (glm_build_ms * 1e-3),
                                         "keys": "N(0,1) bf16 drawn on the device"}},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["locks", "reference"], default="locks")
    ap.add_argument("--workload", choices=sorted(synth.WORKLOADS), default="ctx1m")
    ap.add_argument("--budget", type=int, default=None)
    ap.add_argument("--pages", type=int, default=None, help="override pages per sequence (smaller cases)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true", help="skip the dense-attention comparator")
    ap.add_argument("--no-model-graph", action="store_true", help="skip the 32-layer decode graph")
    ap.add_argument("--no-ablation", action="store_true", help="skip the selector ablations")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_locks(args, rank, world, local)


if __name__ == "__main__":
    main()
