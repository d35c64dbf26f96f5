"""Benchmark of the quantized-weight matvec / routed-expert library on GB300.

Default workload (one JSON line): the decode expert block at full size --
hidden 6144, expert intermediate 2048, 256 resident experts (fmt=4 grouped
int4, gs=64), top-8 softmax routing drawn afresh every step, S=1.  One step
is one coli_moe_block call (routing, gate/up, silu*mul, down, weighted
scatter-add: the whole hot path).  The metric is algorithmic HBM GB/s: the
packed codes and scales of the 8 routed experts plus x and y, divided by the
device time.  The 5.4 GB expert pool is far larger than L2 and every step
routes to a fresh random set, so no step finds its weights in L2.

Other workloads (--workload): gemv_sweep, moe_prefill, streaming, router
(all four are also in the by_workload part of a full run).  --impl reference times the CPU oracle (the reference arm of this
benchmark) on a bounded sample of the same workload.

Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torch.distributed.run, one rank per GPU, each running its own independent
replica (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402


# ---------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = "samples inside the timed region"
        if not inside and self.samples:
            nearest = min(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))
            inside = [nearest[1]]
            note = "timed region shorter than the sampling interval: nearest sample"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "note": note}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def aggregate(value_units: float, seconds: float, world: int):
    """Sum the units and take the max time over ranks (identity for one rank)."""
    if world == 1:
        return value_units, seconds
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([value_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(u.item()), float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- workloads
class DecodeBlock:
    """Decode expert block, S=1, 256 experts, top-8."""

    name = "moe_decode_block"
    metric_unit = "GB/s"

    def __init__(self, coli, torch, seed_offset=0, n_experts=None):
        self.coli, self.torch = coli, torch
        c = self.c = wl.MOE_DECODE
        g = wl.rng(c["seed"] + seed_offset)
        self.H, self.F, self.E, self.K = c["H"], c["F"], n_experts or c["E"], c["K"]
        self.host = []
        dev = []
        for _ in range(self.E):
            trip = wl.expert(g, self.H, self.F, c["fmt"], c["gs"])
            self.host.append(trip)
            dev.append(tuple(coli.tensor_upload(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in trip))
        self.table = coli.ExpertTable(dev)
        self.n_routes = 4096
        ids, w = wl.routing_topk_softmax(g, self.n_routes, self.E, self.K)
        self.ids_h, self.w_h = ids, w
        self.ids = torch.from_numpy(ids).cuda()
        self.w = torch.from_numpy(w).cuda()
        self.xs_h = wl.activations(g, 64, self.H)
        self.x = torch.from_numpy(self.xs_h).cuda()
        self.x_rows = [self.x[i: i + 1] for i in range(64)]
        self.id_rows = [self.ids[r: r + 1] for r in range(self.n_routes)]
        self.w_rows = [self.w[r: r + 1] for r in range(self.n_routes)]
        self.y = torch.empty(1, self.H, device="cuda")
        self.expert_bytes = wl.expert_bytes(self.H, self.F, c["fmt"], c["gs"])
        self.bytes_per_step = self.K * self.expert_bytes + 2 * 4 * self.H + 8 * self.K
        self.launches_per_step = 1

    def step(self, i, stream=None):
        r = i % self.n_routes
        self.coli.moe_block(self.x_rows[i % 64], self.table, self.id_rows[r], self.w_rows[r], self.y, stream=stream)

    def e2e_setup(self):
        """Each step's inputs (x, ids, w) packed in one pinned host record, so a
        step is one host-to-device copy, the block call and one device-to-host
        copy of y.  The steps are independent tokens, so they run pipelined over
        two device buffers: on a copy stream (the current stream of the whole
        loop) step i + 1's inputs go in before step i's y comes out, and the
        block calls run on a compute stream; events order each buffer's reuse."""
        t = self.torch
        H, K = self.H, self.K
        rec = np.zeros((64, H + 2 * K), np.float32)
        for r in range(64):
            rec[r, :H] = self.xs_h[r]
            rec[r, H:H + K] = self.ids_h[r].astype(np.int32).view(np.float32)
            rec[r, H + K:] = self.w_h[r]
        self.hin = [t.from_numpy(rec[r].copy()).pin_memory() for r in range(64)]
        self.din = [t.empty(H + 2 * K, device="cuda") for _ in range(2)]
        self.dx = [d[:H].view(1, H) for d in self.din]
        self.dids = [d[H:H + K].view(t.int32).view(1, K) for d in self.din]
        self.dw = [d[H + K:].view(1, K) for d in self.din]
        self.dy = [t.empty(1, H, device="cuda") for _ in range(2)]
        self.hy = [t.empty(1, H).pin_memory() for _ in range(2)]
        self.s_cp, self.s_cmp = t.cuda.Stream(), t.cuda.Stream()
        self.ev_in = [t.cuda.Event() for _ in range(2)]
        self.ev_cmp = [t.cuda.Event() for _ in range(2)]
        self.ev_out = [t.cuda.Event() for _ in range(2)]
        for b in range(2):   # every buffer starts out free
            self.ev_cmp[b].record(self.s_cmp)
            self.ev_out[b].record(self.s_cp)
        self.h2d = 4 * H + 8 * K
        self.d2h = 4 * H

    def e2e_begin(self, i0):
        """Step i0's inputs in (the copy stream must be current)."""
        b = i0 % 2
        self.s_cp.wait_event(self.ev_cmp[b])
        self.din[b].copy_(self.hin[i0 % 64], non_blocking=True)
        self.ev_in[b].record(self.s_cp)

    def e2e_step(self, i):
        """Step i (its inputs already on their way): step i + 1's inputs in,
        the block call, step i's y out.  The copy stream must be current."""
        b, nb = i % 2, (i + 1) % 2
        self.s_cp.wait_event(self.ev_cmp[nb])       # the call of step i - 1 has read din[nb]
        self.din[nb].copy_(self.hin[(i + 1) % 64], non_blocking=True)
        self.ev_in[nb].record(self.s_cp)
        self.s_cmp.wait_event(self.ev_in[b])
        self.s_cmp.wait_event(self.ev_out[b])      # y[b] of step i - 2 has reached the host
        self.coli.moe_block(self.dx[b], self.table, self.dids[b], self.dw[b], self.dy[b], stream=self.s_cmp)
        self.ev_cmp[b].record(self.s_cmp)
        self.s_cp.wait_event(self.ev_cmp[b])
        self.hy[b].copy_(self.dy[b], non_blocking=True)
        self.ev_out[b].record(self.s_cp)

    def e2e_join(self, stream):
        """Make `stream` wait for every copy and call issued so far."""
        for b in range(2):
            stream.wait_event(self.ev_out[b])
            stream.wait_event(self.ev_cmp[b])

    def oracle_sample(self, budget_s: float):
        """The oracle on whole decode steps of this workload, as many as fit."""
        from oracle import oracle as orc
        mats_cache = {}
        done, t0, nbytes = 0, time.time(), 0
        while True:
            r = done % self.n_routes
            ids = self.ids_h[r: r + 1]
            used = sorted(set(int(e) for e in ids[0]))
            mats = []
            remap = {}
            for j, e in enumerate(used):
                if e not in mats_cache:
                    mats_cache[e] = tuple(orc.Mat(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in self.host[e])
                mats.append(mats_cache[e])
                remap[e] = j
            ids_l = np.vectorize(remap.get)(ids).astype(np.int32)
            orc.moe_block(self.H, self.F, mats, self.xs_h[done % 64: done % 64 + 1], ids_l, self.w_h[r: r + 1])
            done += 1
            nbytes += self.bytes_per_step
            if time.time() - t0 > budget_s:
                break
        dt = time.time() - t0
        return nbytes / dt / 1e9, done, dt


# ---------------------------------------------------------------- other workloads of the metric
# The oracle timed beside each GPU number (bounded samples; off with --no-cpu-baseline).
CPU_TIMING = {"on": True, "budget": 0.4}


def oracle_time(fn, units_per_call: float, unit: str, sample: str):
    """The oracle, as it stands, on a bounded sample: fn() is one oracle call
    covering units_per_call units of the metric.  Timed single-threaded and on
    all the host's cores (each: one call, then more until the budget is spent)."""
    if not CPU_TIMING["on"]:
        return None
    from oracle import oracle as orc
    n_all = orc.threads()
    rate = {}
    for label, n in (("single_thread", 1), ("all_cores", n_all)):
        prev = orc.set_threads(n)
        try:
            calls, t0 = 0, time.perf_counter()
            while True:
                fn()
                calls += 1
                dt = time.perf_counter() - t0
                if dt >= CPU_TIMING["budget"]:
                    break
        finally:
            orc.set_threads(prev)
        rate[label] = units_per_call * calls / dt
    return {"value": rate["all_cores"], "unit": unit, "cores": n_all, "kind": "oracle",
            "single_thread": rate["single_thread"], "sample": sample}


def _orc():
    from oracle import oracle as orc
    return orc


def _omat(m):
    return _orc().Mat(m.fmt, m.gs, m.O, m.I, m.data, m.scales)


def _time_loop(torch, fn, n, warm=5):
    for i in range(warm):
        fn(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(n):
        fn(i)
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / n


def _time_graph(torch, fn, n, warm=3):
    """Average device time of fn(0..n-1) replayed from one CUDA graph (no
    Python launch overhead inside the timed region)."""
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):   # warm up on the capture stream: its scratch exists before capture
        for i in range(warm):
            fn(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        for i in range(n):
            fn(i)
    graph.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    graph.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / n


def bench_gemv(coli, torch, peaks, l2_bytes, only=None):
    """Single fmt=4 GEMV and the format sweep, each over enough distinct copies
    of the matrix that the rotation exceeds 4x L2 (no call finds its weights in L2)."""
    out = {}
    cases = [("gemv_single_fmt4_g64", 4, 64, wl.GEMV_SINGLE["O"], wl.GEMV_SINGLE["I"], (1,), wl.GEMV_SINGLE["seed"])]
    for fmt, gs in wl.GEMV_SWEEP["variants"]:
        name = f"sweep_fmt{fmt}" + (f"_g{gs}" if fmt == 4 else "")
        cases.append((name, fmt, gs, wl.GEMV_SWEEP["O"], wl.GEMV_SWEEP["I"], wl.GEMV_SWEEP["S"], wl.GEMV_SWEEP["seed"]))
    # FP8 E4M3 with 128 x 128 block scales (uniform over the finite bytes), same shape
    cases.append(("fp8_fmt7_b128", 7, 0, wl.GEMV_SWEEP["O"], wl.GEMV_SWEEP["I"], wl.GEMV_SWEEP["S"],
                  wl.GEMV_SWEEP["seed"]))
    # int3 (fmt=5) with groups of 64, quantised from the same N(0, 0.02) weights
    cases.append(("sweep_int3_fmt5_g64", 5, 64, wl.GEMV_SWEEP["O"], wl.GEMV_SWEEP["I"], wl.GEMV_SWEEP["S"],
                  wl.GEMV_SWEEP["seed"]))
    if only:
        cases = [c for c in cases if c[0] == only]
        if not cases:
            raise SystemExit(f"unknown --gemv-case {only}")
    for name, fmt, gs, O, I, Ss, seed in cases:
        g = wl.rng(seed + fmt + gs)
        if name.startswith("sweep"):
            m = wl.quantize(fmt, g.normal(0, 0.02, (O, I)).astype(np.float32), gs)
        else:
            m = wl.random_matrix(g, fmt, O, I, gs)
        ncopy = max(2, math.ceil(4 * l2_bytes / m.nbytes))
        Ws = [coli.tensor_upload(m.fmt, m.gs, O, I, m.data, m.scales) for _ in range(ncopy)]
        res = {}
        for S in Ss:
            x = torch.randn(S, I, device="cuda")
            y = torch.empty(S, O, device="cuda")
            t = _time_graph(torch, lambda i: coli.matmul(Ws[i % ncopy], x, y), max(200, 2 * ncopy))
            nbytes = m.nbytes + 4 * S * (I + O)
            xh = x.cpu().numpy()
            cpu = oracle_time(lambda: _orc().matmul(m.fmt, m.gs, O, I, m.data, m.scales, xh), nbytes / 1e9, "GB/s",
                              f"whole {O}x{I} product at S={S}")
            res[f"S{S}"] = {"us": t * 1e6, "GB/s": nbytes / t / 1e9, "frac_hbm": nbytes / t / 1e9 / peaks["hbm_gbs"],
                            "cpu_baseline": cpu}
        coli.sync_check()
        out[name] = {"bytes": m.nbytes, "copies": ncopy, **res}
        del Ws
    return out


def bench_prefill(coli, torch, peaks, steps=5, n_experts=None):
    """Prefill expert block: S=544, Zipf(1.1) top-8 over 256 experts, fmt=4
    gs=128; tokens/s and the fraction of the per-expert roofline
    sum_e max(bytes_e / HBM, flops_e / bf16 peak)."""
    c = wl.MOE_PREFILL
    g = wl.rng(c["seed"])
    H, F, E, K, S = c["H"], c["F"], n_experts or c["E"], c["K"], c["S"]
    dev, hosts = [], []
    for _ in range(E):
        trip = wl.expert(g, H, F, c["fmt"], c["gs"])
        dev.append(tuple(coli.tensor_upload(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in trip))
        hosts.append(trip if CPU_TIMING["on"] else None)
    table = coli.ExpertTable(dev)
    x_h = wl.activations(g, S, H, bf16_exact=True)
    x = torch.from_numpy(x_h).cuda()
    ids_h, w_h = wl.routing_zipf(g, S, E, K, c["zipf"])
    ids = torch.from_numpy(ids_h).cuda()
    w = torch.from_numpy(w_h).cuda()
    y = torch.empty(S, H, device="cuda")
    t = _time_loop(torch, lambda i: coli.moe_block(x, table, ids, w, y), steps, warm=2)
    coli.sync_check()
    counts = np.bincount(ids_h.reshape(-1), minlength=E)
    eb = wl.expert_bytes(H, F, c["fmt"], c["gs"])
    flops_per_row = 2 * 3 * H * F
    roof = sum(max(eb / (peaks["hbm_gbs"] * 1e9), n * flops_per_row / (peaks["bf16_tflops"] * 1e12))
               for n in counts if n > 0)
    touched = int((counts > 0).sum())
    cpu = None
    if CPU_TIMING["on"]:
        rows = 2   # the oracle on the first rows of the batch, with their own routing
        used = sorted(set(int(e) for e in ids_h[:rows].reshape(-1)))
        mats = [tuple(_omat(m) for m in hosts[e]) for e in used]
        ids_l = np.searchsorted(np.array(used), ids_h[:rows]).astype(np.int32)
        cpu = oracle_time(lambda: _orc().moe_block(H, F, mats, x_h[:rows], ids_l, w_h[:rows]), rows, "tokens/s",
                          f"the expert block on the batch's first {rows} rows (top-{K} each)")
    del hosts
    return {"tokens/s": S / t, "ms": t * 1e3, "experts_touched": touched, "max_rows_per_expert": int(counts.max()),
            "GB/s": touched * eb / t / 1e9, "GFLOP": float(counts.sum() * flops_per_row / 1e9),
            "roofline_ms": roof * 1e3, "frac_of_per_expert_roofline": roof / t, "cpu_baseline": cpu}


def bench_streaming(coli, torch, peaks, tokens=10, pool_gb=None, only_fmt=None):
    """Weight streaming: S=1 GEMVs of 2048x6144 over a 40 GB resident pool,
    8 random matrices per layer (one launch: shared input), 75 layers per token.
    pool_gb / only_fmt shrink the run (profiling captures)."""
    c = wl.STREAMING
    res = {}
    for fmt, gs in c["variants"]:
        if only_fmt is not None and fmt != only_fmt:
            continue
        g = wl.rng(c["seed"] + fmt)
        per = wl.tensor_bytes(fmt, c["O"], c["I"], gs)
        n_pool = int((pool_gb or c["pool_gb"]) * 1e9 // per)
        srcs = [wl.random_matrix(g, fmt, c["O"], c["I"], gs) for _ in range(16)]
        pool = [coli.tensor_upload(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in
                (srcs[i % 16] for i in range(n_pool))]
        sel = g.integers(0, n_pool, (c["layers"] * (tokens + 1), c["per_layer"]))
        x = torch.randn(1, c["I"], device="cuda")
        ys = [torch.empty(1, c["O"], device="cuda") for _ in range(c["per_layer"])]
        n_layers = c["layers"] * tokens
        t = _time_graph(torch, lambda i: coli.matmul_multi([pool[j] for j in sel[i]], x, ys), n_layers, warm=c["layers"])
        coli.sync_check()
        nbytes = c["per_layer"] * per
        xh = x.cpu().numpy()
        cpu = oracle_time(lambda: [_orc().matmul(m.fmt, m.gs, m.O, m.I, m.data, m.scales, xh)
                                   for m in srcs[:c["per_layer"]]], nbytes / 1e9, "GB/s",
                          f"one layer: {c['per_layer']} whole {c['O']}x{c['I']} products at S=1")
        res[f"fmt{fmt}" + (f"_g{gs}" if fmt == 4 else "")] = {
            "pool_matrices": n_pool, "pool_GB": n_pool * per / 1e9, "layer_us": t * 1e6,
            "GB/s": nbytes / t / 1e9, "frac_hbm": nbytes / t / 1e9 / peaks["hbm_gbs"],
            "tokens/s": 1.0 / (c["layers"] * t), "cpu_baseline": cpu}
        del pool
        torch.cuda.empty_cache()
    return res


def bench_router(coli, torch, peaks, steps=200):
    """Device-side router of the decode workload: logits of a 256 x 6144 f32
    router, sigmoid + bias greedy top-8 with norm_topk (coli_moe_router), alone
    and followed by the expert block (the whole routed-expert layer on the GPU,
    no host step between)."""
    c = wl.MOE_DECODE
    g = wl.rng(c["seed"] + 100)
    H, F, E, K = c["H"], c["F"], c["E"], c["K"]
    Wr = g.normal(0.0, 0.05, (E, H)).astype(np.float32)
    router = coli.tensor_upload(0, 0, E, H, Wr, None)
    bias = torch.from_numpy(g.normal(0.0, 0.01, E).astype(np.float32)).cuda()
    n_pool = 64
    hosts = [wl.expert(g, H, F, c["fmt"], c["gs"]) for _ in range(8)]
    dev = [tuple(coli.tensor_upload(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in hosts[e % 8])
           for e in range(n_pool)]
    table = coli.ExpertTable(dev + [dev[e % n_pool] for e in range(E - n_pool)])
    xs = torch.randn(steps, 1, H, device="cuda")
    ids = torch.empty((1, K), dtype=torch.int32, device="cuda")
    w = torch.empty((1, K), device="cuda")
    y = torch.empty((1, H), device="cuda")
    st = torch.cuda.Stream()

    def timed(fn):
        with torch.cuda.stream(st):
            for i in range(3):
                fn(i)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            for i in range(steps):
                fn(i)
        graph.replay()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(st):
            a.record(st)
            graph.replay()
            b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3 / steps

    t_router = timed(lambda i: coli.moe_router(xs[i], router, K, ids, w, bias=bias, norm_topk=True, stream=st))
    t_layer = timed(lambda i: (coli.moe_router(xs[i], router, K, ids, w, bias=bias, norm_topk=True, stream=st),
                               coli.moe_block(xs[i], table, ids, w, y, stream=st)))
    coli.sync_check()
    rb = E * H * 4
    xh = xs[0].cpu().numpy()
    bh = bias.cpu().numpy()
    cpu = oracle_time(lambda: _orc().moe_topk(_orc().matmul(0, 0, E, H, Wr, None, xh), K, bias=bh, norm_topk=True),
                      rb / 1e9, "GB/s", "one token: f32 router logits and the biased top-8")
    return {"router_us": t_router * 1e6, "router_GB/s": rb / t_router / 1e9, "cpu_baseline": cpu,
            "router_plus_expert_block_us": t_layer * 1e6,
            "note": "S=1, f32 router 256x6144, top-8 of sigmoid+bias with norm_topk; expert block over a "
                    "64-expert resident pool (L2 sees part of it: the block time here is not the headline)"}


def bench_host(coli, torch, peaks, l2_bytes, steps=100):
    """Host-resident weights (coli_tensor_upload_host) read zero-copy over the
    CPU-GPU link: (a) the link's copy bandwidth, pinned host -> HBM (torch copy),
    as the reference; (b) a 2048x6144 int4 g64 matvec with its weights in host
    memory, rotated over copies exceeding 4x L2; (c) the decode expert block
    (H=6144, F=2048, int4 g64, S=1, K=8) with k of the 8 routed experts in host
    memory and the rest in HBM, a fresh routing per call."""
    out = {}
    nb = 1 << 29
    hsrc = torch.empty(nb, dtype=torch.uint8, pin_memory=True)
    ddst = torch.empty(nb, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        ddst.copy_(hsrc, non_blocking=True)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(4):
        ddst.copy_(hsrc, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    link = 4 * nb / (a.elapsed_time(b) / 1e3) / 1e9
    out["h2d_copy_GB/s"] = link
    del hsrc, ddst

    c = wl.GEMV_SWEEP
    O, I = c["O"], c["I"]
    g = wl.rng(c["seed"] + 50)
    m = wl.random_matrix(g, 4, O, I, 64)
    ncopy = max(2, math.ceil(4 * l2_bytes / m.nbytes))
    Ws = [coli.tensor_upload_host(m.fmt, m.gs, O, I, m.data, m.scales) for _ in range(ncopy)]
    x = torch.randn(1, I, device="cuda")
    y = torch.empty(1, O, device="cuda")
    t = _time_graph(torch, lambda i: coli.matmul(Ws[i % ncopy], x, y), max(100, 2 * ncopy))
    coli.sync_check()
    out["matvec_host_fmt4_g64_S1"] = {"us": t * 1e6, "GB/s": m.nbytes / t / 1e9,
                                      "frac_of_copy": m.nbytes / t / 1e9 / link, "copies": ncopy}
    del Ws

    d = wl.MOE_DECODE
    H, F, K = d["H"], d["F"], d["K"]
    g = wl.rng(d["seed"] + 200)
    hosts = [wl.expert(g, H, F, d["fmt"], d["gs"]) for _ in range(8)]
    n_dev, n_host = 64, 16
    dev = [tuple(coli.tensor_upload(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in hosts[e % 8])
           for e in range(n_dev)]
    hst = [tuple(coli.tensor_upload_host(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in hosts[e % 8])
           for e in range(n_host)]
    table = coli.ExpertTable(dev + hst)
    xs = torch.randn(steps, 1, H, device="cuda")
    w = torch.full((1, K), 1.0 / K, device="cuda")
    yb = torch.empty(1, H, device="cuda")
    per_expert = wl.expert_bytes(H, F, d["fmt"], d["gs"])
    res = {}
    for k in (0, 1, 2, 8):
        ids = np.empty((steps, 1, K), np.int32)
        for i in range(steps):
            dv = [(i * 7 + j) % n_dev for j in range(K - k)]
            hv = [n_dev + (i * 3 + j) % n_host for j in range(k)]
            ids[i, 0] = dv + hv
        idd = torch.from_numpy(ids).cuda()
        t = _time_graph(torch, lambda i: coli.moe_block(xs[i], table, idd[i], w, yb), steps)
        coli.sync_check()
        res[f"k{k}"] = {"us": t * 1e6, "host_bytes": k * per_expert, "hbm_bytes": (K - k) * per_expert,
                        "host_GB/s_if_link_bound": k * per_expert / t / 1e9}
    out["decode_block_k_of_8_in_host_memory"] = res
    return out


def bench_absorb(coli, torch, peaks, l2_bytes):
    """kv_b absorption products at an MLA decode shape: kv_b of 128 heads x
    (128 key + 128 value rows) x 512 latent inputs, int4 g64; per token the
    transposed product over each head's key rows and the forward product over
    its value rows, S = 1, rotated over copies exceeding 4x L2."""
    n_heads, per_head, n_rows, I = 128, 256, 128, 512
    g = wl.rng(4321)
    m = wl.random_matrix(g, 4, n_heads * per_head, I, 64)
    ncopy = max(2, math.ceil(4 * l2_bytes / m.nbytes))
    Ws = [coli.tensor_upload(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for _ in range(ncopy)]
    half = m.nbytes / 2   # each product touches half of the rows
    xt = torch.randn(1, n_heads, n_rows, device="cuda")
    yt = torch.empty(1, n_heads, I, device="cuda")
    xf = torch.randn(1, n_heads, I, device="cuda")
    yf = torch.empty(1, n_heads, n_rows, device="cuda")
    n = max(200, 2 * ncopy)
    t_t = _time_graph(torch, lambda i: coli.matmul_rows_t(Ws[i % ncopy], 0, per_head, n_rows, n_heads, xt, yt), n)
    t_f = _time_graph(torch, lambda i: coli.matmul_rows(Ws[i % ncopy], n_rows, per_head, n_rows, n_heads, xf, yf), n)
    coli.sync_check()
    res = {}
    for name, t in (("key_rows_transposed", t_t), ("value_rows_forward", t_f)):
        res[name] = {"us": t * 1e6, "GB/s": half / t / 1e9, "frac_hbm": half / t / 1e9 / peaks["hbm_gbs"]}
    res["note"] = (f"kv_b {n_heads}x{per_head} rows x {I} inputs, int4 g64 ({m.nbytes / 1e6:.1f} MB, "
                   f"{ncopy} copies); each product reads half of it")
    return res


def bench_decode_formats(coli, torch, peaks, steps=200, only=None):
    """The decode expert block (H=6144, F=2048, S=1, top-8 of 256 resident
    experts, a fresh softmax top-8 routing per call) for every expert format:
    f32, int8, int4 per-row, int2, int4 g64 (the headline's), int4 g128, int3
    g64 and FP8 E4M3 with 128x128 block scales.  The 256 experts are distinct device copies
    of 8 generated ones, so every pool is far larger than L2 (the smallest,
    int2, is 2.5 GB)."""
    d = wl.MOE_DECODE
    H, F, K, E = d["H"], d["F"], d["K"], d["E"]
    out = {}
    cases = (("f32_fmt0", 0, 0), ("int8_fmt1", 1, 0), ("int4_fmt2", 2, 0), ("int2_fmt3", 3, 0),
             ("int4_fmt4_g64", 4, 64), ("int4_fmt4_g128", 4, 128), ("int3_fmt5_g64", 5, 64), ("fp8_fmt7_b128", 7, 0))
    for name, fmt, gs in cases:
        if only and name != only:
            continue
        g = wl.rng(d["seed"] + 300 + fmt + gs)
        hosts = [wl.expert(g, H, F, fmt, gs) for _ in range(8)]
        dev = [tuple(coli.tensor_upload(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in hosts[e % 8])
               for e in range(E)]
        table = coli.ExpertTable(dev)
        ids_h, w_h = wl.routing_topk_softmax(g, steps, E, K)
        ids = torch.from_numpy(ids_h).cuda()
        w = torch.from_numpy(w_h).cuda()
        xs_h = wl.activations(g, steps, H)
        xs = torch.from_numpy(xs_h).cuda().view(steps, 1, H)
        y = torch.empty(1, H, device="cuda")
        t = _time_graph(torch, lambda i: coli.moe_block(xs[i], table, ids[i: i + 1], w[i: i + 1], y), steps)
        coli.sync_check()
        eb = wl.expert_bytes(H, F, fmt, gs)
        nbytes = K * eb + 2 * 4 * H + 8 * K
        cpu = None
        if CPU_TIMING["on"]:
            mats = [tuple(_omat(m) for m in hosts[e % 8]) for e in ids_h[0]]
            cpu = oracle_time(lambda: _orc().moe_block(H, F, mats, xs_h[:1], np.arange(K, dtype=np.int32)[None],
                                                       w_h[:1]), nbytes / 1e9, "GB/s", "one token's block (8 experts)")
        out[name] = {"us": t * 1e6, "GB/s": nbytes / t / 1e9, "frac_hbm": nbytes / t / 1e9 / peaks["hbm_gbs"],
                     "pool_GB": E * eb / 1e9, "cpu_baseline": cpu}
        del dev, table, hosts
        torch.cuda.empty_cache()
    return out


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle, timed as it stands, on a bounded
    sample of the default workload: one routed (row, expert) slot per step."""
    if rank != 0:
        return 0
    from oracle import oracle as orc
    c = wl.MOE_DECODE
    g = wl.rng(c["seed"])
    H, F = c["H"], c["F"]
    experts = [wl.expert(g, H, F, c["fmt"], c["gs"]) for _ in range(4)]
    mats = [tuple(orc.Mat(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in e) for e in experts]
    ids, w = wl.routing_topk_softmax(g, 64, 4, 1)
    x = wl.activations(g, 64, H)
    per_step = wl.expert_bytes(H, F, c["fmt"], c["gs"]) + 2 * 4 * H + 8
    for i in range(args.warmup):
        orc.moe_block(H, F, mats, x[i % 64: i % 64 + 1], ids[i % 64: i % 64 + 1], w[i % 64: i % 64 + 1])
    t0 = time.perf_counter()
    for i in range(args.steps):
        orc.moe_block(H, F, mats, x[i % 64: i % 64 + 1], ids[i % 64: i % 64 + 1], w[i % 64: i % 64 + 1])
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt / 1e9
    cores = orc.threads()
    line = {"impl": "reference", "metric": "decode MoE-block HBM GB/s (algorithmic bytes / time)", "value": value,
            "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / max(args.steps, 1), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "moe_decode_block", "hidden": H, "intermediate": F, "experts": 256, "topk": 8,
                       "fmt": 4, "gs": 64, "S": 1},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": "one routed (row, expert) slot of the decode block per step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def time_steps(torch, wk, steps, stream):
    """Time exactly `steps` steps on the device.  The steps are captured once
    into a CUDA graph and the replay is bracketed by events on the launching
    stream, so the host's per-call cost is not inside the timed region (the
    per-call API path is what `e2e` measures).  Returns (seconds, mode)."""
    torch.cuda.synchronize()
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(steps):
                wk.step(1_000_000 + i, stream=stream)
        mode = "cuda-graph replay"
    except Exception as exc:  # capture unsupported: time the direct launches
        graph = None
        mode = f"direct launches ({type(exc).__name__})"
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(steps):
                wk.step(1_000_000 + i, stream=stream)
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3, mode


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--workload", default="moe_decode",
                    choices=("moe_decode", "moe_prefill", "gemv_sweep", "streaming", "router", "host", "absorb",
                             "decode_formats"),
                    help="moe_decode is the headline line; the others print their own line (for profiling)")
    ap.add_argument("--experts-prefill", type=int, default=None, help="resident experts of the prefill workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--cpu-entry-budget", type=float, default=0.4,
                    help="seconds of oracle timing per by_workload entry and thread count (after one call)")
    ap.add_argument("--experts", type=int, default=None, help="resident experts of the decode workload (default 256)")
    ap.add_argument("--quick", action="store_true", help="headline workload only (no by_workload sweep)")
    ap.add_argument("--decode-format", default=None,
                    help="--workload decode_formats: run only this case (e.g. int8_fmt1, fp8_fmt7_b128)")
    ap.add_argument("--stream-pool-gb", type=float, default=None,
                    help="--workload streaming: resident pool size (default 40 GB)")
    ap.add_argument("--stream-fmt", type=int, default=None, help="--workload streaming: only this format")
    ap.add_argument("--gemv-case", default=None,
                    help="--workload gemv_sweep: run only this case (e.g. sweep_fmt4_g64, fp8_fmt7_b128)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    CPU_TIMING["on"] = not args.no_cpu_baseline
    CPU_TIMING["budget"] = args.cpu_entry_budget
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        import torch
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    torch.cuda.set_device(local)
    import bit_weight_gemv_fmt1_gb300 as coli
    peaks = load_peaks()
    if args.workload != "moe_decode":
        if rank == 0:
            if args.workload == "moe_prefill":
                res = bench_prefill(coli, torch, peaks, steps=max(1, args.steps), n_experts=args.experts_prefill)
            elif args.workload == "gemv_sweep":
                l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
                res = bench_gemv(coli, torch, peaks, l2, only=args.gemv_case)
            elif args.workload == "router":
                res = bench_router(coli, torch, peaks)
            elif args.workload == "decode_formats":
                res = bench_decode_formats(coli, torch, peaks, only=args.decode_format)
            elif args.workload == "absorb":
                res = bench_absorb(coli, torch, peaks,
                                   torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
            elif args.workload == "host":
                res = bench_host(coli, torch, peaks,
                                 torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
            else:
                res = bench_streaming(coli, torch, peaks, pool_gb=args.stream_pool_gb, only_fmt=args.stream_fmt)
            print(json.dumps({"workload": args.workload, "result": res}), flush=True)
        return 0

    wk = DecodeBlock(coli, torch, seed_offset=rank, n_experts=args.experts)
    stream = torch.cuda.Stream()
    coli.reset_stats()
    for i in range(args.warmup):
        wk.step(i, stream=stream)
    torch.cuda.synchronize()
    coli.sync_check(stream)
    barrier(world)

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    s0 = coli.stats()
    t_wall0 = time.time()
    seconds, timing_mode = time_steps(torch, wk, args.steps, stream)
    t_wall1 = time.time()
    s1 = coli.stats()
    coli.sync_check(stream)
    time.sleep(0.15)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    units, seconds_max = aggregate(wk.bytes_per_step * args.steps, seconds, world)
    barrier(world)
    value = units / seconds_max / 1e9
    launches = int(s1["launches"] - s0["launches"])

    # end to end through the C ABI with host buffers (pinned), copies inside the timed region
    wk.e2e_setup()
    e2e_steps = args.steps
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(wk.s_cp):   # pipelined: time from the first copy to the last one
        wk.e2e_begin(0)
        for i in range(args.warmup):
            wk.e2e_step(i)
        wk.e2e_join(wk.s_cp)
        torch.cuda.synchronize()
        t0.record(wk.s_cp)
        wk.s_cmp.wait_event(t0)
        wk.e2e_begin(args.warmup)
        for i in range(args.warmup, args.warmup + e2e_steps):
            wk.e2e_step(i)
        wk.e2e_join(wk.s_cp)
        t1.record(wk.s_cp)
    torch.cuda.synchronize()
    e2e_s = t0.elapsed_time(t1) / 1e3
    e2e_units, e2e_max = aggregate(wk.bytes_per_step * e2e_steps, e2e_s, world)
    e2e_value = e2e_units / e2e_max / 1e9

    # roofline of the dominant kernel (the single decode launch of each step)
    avg_launch_s = seconds / args.steps / wk.launches_per_step
    achieved = wk.bytes_per_step / avg_launch_s / 1e9
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tr_path):
        traffic = json.load(open(tr_path)).get("moe_decode_mma_kernel")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, n, dt = wk.oracle_sample(args.cpu_budget)
        from oracle import oracle as orc
        prev = orc.set_threads(1)
        try:
            v1, n1, dt1 = wk.oracle_sample(min(3.0, args.cpu_budget))
        finally:
            orc.set_threads(prev)
        cpu = {"value": v, "unit": "GB/s", "cores": orc.threads(), "kind": "oracle",
               "sample": f"{n} whole decode steps (8 routed experts each) in {dt:.1f} s",
               "single_thread": v1, "single_thread_sample": f"{n1} whole decode steps in {dt1:.1f} s"}

    by_wl = None
    if rank == 0 and not args.quick:
        l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
        by_wl = {"gemv": bench_gemv(coli, torch, peaks, l2), "moe_prefill": bench_prefill(coli, torch, peaks),
                 "weight_streaming": bench_streaming(coli, torch, peaks), "router": bench_router(coli, torch, peaks),
                 "moe_decode_per_format": bench_decode_formats(coli, torch, peaks)}

    if rank == 0:
        line = {
            "metric": "decode MoE-block HBM GB/s (algorithmic bytes / time)",
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": seconds_max * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "moe_decode_block", "hidden": wk.H, "intermediate": wk.F, "experts": wk.E,
                       "topk": wk.K, "fmt": 4, "gs": 64, "S": 1, "global_batch": world,
                       "parallelism": f"replicas x{world}",
                       "l2": f"inputs larger than L2: {wk.E * wl.expert_bytes(wk.H, wk.F, 4, 64) / 1e9:.2f} GB expert pool, fresh top-{wk.K} "
                             "routing every step",
                       "bytes_per_step": wk.bytes_per_step},
            "hbm_frac_of_measured": value / peaks["hbm_gbs"],
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                         "peak_source": peaks["source"], "kernel": "moe_decode_mma_kernel<1, 0>",
                         "avg_launch_us": avg_launch_s * 1e6, "timing": timing_mode},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": wk.h2d, "d2h_bytes_per_step": wk.d2h},
            "gpu_launches": launches,
            "clocks": clocks,
            "by_workload": by_wl,
        }
        print(json.dumps(line), flush=True)
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
