#!/usr/bin/env python3
"""Benchmark: W1.58A8 ternary GEMV effective HBM GB/s and us per 2B-shaped decode layer.

One step = one pass of the decode hot path over a 2B-shaped decoder stack at batch 1:
30 distinct layers (521 MB of packed weights, > 4x the 126 MB L2, so the timed
region streams HBM without any flush), each layer running

    [RMSNorm+quant](x_attn) -> GEMV q|k|v (3840x2560) -> [quant](x_o) -> GEMV o (2560x2560)
    -> [RMSNorm+quant](x_ffn) -> GEMV gate|up (13824x2560) -> [quant](x_down) -> GEMV down (2560x6912)

with each bracketed quantisation fused into its GEMV launch (tw_quant_gemv, chained by
programmatic dependent launch); --separate runs them as their own kernels.  Attention
and the FFN activation are not part of the path: the o and down inputs are fresh
N(0,1) vectors per layer.  Weights are N(0,1) drawn on the GPU (seeded torch generator)
and absmean-ternarised once with tw_pack_ternary before timing (the conversion is
offline).  The launches of a step are captured in one CUDA graph.

value   = algorithmic bytes of all GEMVs in the step (packed weights + int8 activations
          + scales) / device time of the step, whole job (all ranks).
e2e     = the same metric with each step's inputs copied from pinned host memory and all its
          outputs copied back inside the timed region (one copy each way per step); the copies
          of neighbouring steps overlap the computation (two buffer sets, their own streams);
          e2e.serial is the same without the overlap.
roofline: the product kernel.  Average launch duration = the timed region's device time
          over its product launches (fused path: every launch of the step); otherwise a graph
          of the product calls alone, replayed like the timed region.  Algorithmic bytes (or
          integer ops, M > 16) per launch = the step's over its launches; peak = measured HBM
          copy rate (or bf16 tensor rate).  traffic = DRAM bytes per launch from the committed
          ncu summary when it was taken on the unchanged kernel, else null.
cpu_baseline / --impl reference: the CPU oracle (oracle/), as it stands, on the host.
Default workload only, as extra keys: us_per_layer_unfused (the same step with the
quantisations as separate kernels), small_case (K = N = 256, M = 1: microseconds per
call, latency-bound), read_stream (a read-only streaming rate, the third bandwidth
basis next to the nominal 8 TB/s and the measured copy rate) and five_trits_per_byte
(the 2B step and a 57344 x 8192 product in the 1.6-bit layout next to the 2-bit one) and
fused_epilogue (the 2B step with the residual add and the next RMSNorm's statistics fused
into the o and down launches).

Under torchrun (N > 1) every rank runs its own replica of the workload (weak scaling,
no data-path collective); rank 0 prints max-over-ranks time and the summed bytes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W1.58A8 GEMV effective HBM GB/s (% of B300 peak); us per 2B-shaped decode layer"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6400.0
LAYERS = 30
MODEL = "2B"
WORKLOAD = "2B-shaped decoder layer, batch 1 (hidden 2560, ffn 6912, 20/5 heads), 30 distinct layers"

# --workload: the default is the decode-layer configuration the metric is quoted on; the
# others are the batched-decode, 8B and 70B sweeps (each prints its own line).
# name: (model, layers, M, distinct packed layers generated (the rest are byte copies))
WORKLOADS = {
    "2b": ("2B", 30, 1, 30),
    "2b_m8": ("2B", 30, 8, 30), "2b_m64": ("2B", 30, 64, 30), "2b_m256": ("2B", 30, 256, 30),
    "8b_m1": ("8B", 32, 1, 4), "8b_m16": ("8B", 32, 16, 4),
    "70b_m1": ("70B", 80, 1, 1), "70b_m4": ("70B", 80, 4, 1), "70b_m16": ("70B", 80, 16, 1),
}
SHAPE_TEXT = {"2B": "hidden 2560, ffn 6912, 20/5 heads", "8B": "hidden 4096, ffn 14336, 32/8 heads",
              "70B": "hidden 8192, ffn 28672, 64/8 heads"}
GEMV_SOURCES = ["ternary_weight_quant_b300/csrc/tw_gemv_stream.cu", "ternary_weight_quant_b300/csrc/tw_common.cuh"]
TRAFFIC_FILES = {"2b": os.path.join(ROOT, "profiles", "gemv_decode_2b_layer_launches.md")}


# ------------------------------------------------------------------ distributed helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def combine_over_ranks(elapsed_s: float, units: float, world: int):
    """Max elapsed time and summed units over ranks (identity when world == 1)."""
    if world <= 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ shapes and bytes
def layer_plan(model=MODEL):
    import seeded_inputs as si
    s = si.fused_layer_shapes(model)
    # (name, N, K, prologue) in step order; prologue: "rms" = RMSNorm+quant, "quant" = quant only
    return [("qkv", *s["qkv"], "rms"), ("o", *s["o"], "quant"), ("gateup", *s["gateup"], "rms"),
            ("down", *s["down"], "quant")]


def gemv_bytes(N, K, M=1):
    """Algorithmic bytes of one GEMV launch: packed weights + int8 activations + scales."""
    return N * K // 4 + M * K + 4 + 4 * M


def t5_row_bytes(K):
    """Bytes per row of the five-trits-per-byte layout: 16 ceil(K / 80)."""
    return 16 * ((K + 79) // 80)


def gemv_bytes_t5(N, K, M=1):
    """Algorithmic bytes of one GEMV launch over five-trits-per-byte rows."""
    return N * t5_row_bytes(K) + M * K + 4 + 4 * M


def step_bytes(M=1, model=MODEL, layers=LAYERS):
    return layers * sum(gemv_bytes(N, K, M) for _, N, K, _ in layer_plan(model))


def step_ops(M, model=MODEL, layers=LAYERS):
    """Integer operations of one step (2 per weight and token)."""
    return layers * sum(2 * M * N * K for _, N, K, _ in layer_plan(model))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense bf16 TFLOP/s measured on this machine (the tensor path computes in bf16 operands)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured bf16 burst"
    return 1800.0, "fallback"


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch (read + write, averaged over a step's launches) from the committed
    ncu summary of this workload, if it was taken on the current kernel sources."""
    path = TRAFFIC_FILES.get(workload)
    if path is None or not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ": " in line:
                k, v = line[2:].split(": ", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_hash") != source_hash(GEMV_SOURCES):
        return None
    try:
        return float(fields["dram_bytes_per_launch_avg"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int, period_ms: int = 50):
        self.index, self.period = index, period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        import subprocess
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)  # let the first samples arrive before the timed work starts
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        for line in self.lines:
            f = [v.strip() for v in line.split(",")]
            if len(f) != len(self.FIELDS):
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for name, v in zip(self.NAMES, f[3:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle (baseline / reference arm)
def host_cpu() -> str:
    """The host CPU model and its logical core count, for the CPU-baseline description."""
    model = "unknown CPU"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return f"{model}, {os.cpu_count()} logical cores on the host"


def sample_rows(N: int, K: int, M: int, budget: float = 2e7) -> int:
    """Rows of an N x K matrix the CPU oracle multiplies in one pass of its bounded sample:
    about `budget` weight-token products per matrix (at least 16 rows, at most all)."""
    return int(max(16, min(N, budget // max(1, M * K))))


def host_oracle_layer(model: str, M: int, seed: int = 4242, outliers: bool = False):
    """One layer of seeded host inputs for the CPU oracle, with the GPU workload's shapes and
    recipe; per matrix only sample_rows() rows are drawn (the oracle's rate per byte is what is
    measured, and its time per row does not depend on which rows)."""
    import oracle
    import seeded_inputs as si
    g = si.cpu_generator(seed)
    L = []
    for name, N, K, pro in layer_plan(model):
        rows = sample_rows(N, K, M)
        packed, gamma = oracle.pack_ternary(si.weights(rows, K, gen=g))
        L.append(dict(name=name, N=N, K=K, pro=pro, rows=rows, packed=packed, gamma=gamma,
                      x=si.activations(M, K, gen=g, outliers=outliers),
                      g=si.rms_gain(K, seed=seed) if pro == "rms" else None))
    return L


def oracle_rate(L, M: int, seconds: float, openmp: bool):
    """The oracle's decode-layer sequence (RMSNorm/quantisation of the M tokens, then the
    integer product of each matrix) repeated for at least `seconds`.  Each product's time is
    scaled by N / rows to the full matrix; returns (GB/s of the metric's bytes, passes)."""
    import oracle
    import seeded_inputs as si
    t0 = time.perf_counter()
    full_time, full_bytes, passes = 0.0, 0, 0
    while True:
        for e in L:
            a = time.perf_counter()
            if e["pro"] == "rms":
                xq, sx, _ = oracle.rmsnorm_quant_act(e["x"], e["g"], si.RMS_EPS)
            else:
                xq, sx, _ = oracle.quant_act(e["x"])
            b = time.perf_counter()
            oracle.ternary_matmul(e["packed"], e["gamma"], xq, sx, openmp=openmp)
            c = time.perf_counter()
            full_time += (b - a) + (c - b) * e["N"] / e["rows"]
            full_bytes += gemv_bytes(e["N"], e["K"], M)
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            return full_bytes / full_time / 1e9, passes


def cpu_baseline_for(model: str, M: int, seconds_single: float, seconds_all: float, outliers: bool = False):
    """The oracle as a CPU baseline of one workload: single thread, then all host cores (the
    OpenMP build of its integer product).  `value` is the all-core rate."""
    import oracle
    L = host_oracle_layer(model, M, outliers=outliers)
    single, n1 = oracle_rate(L, M, seconds_single, openmp=False)
    cores = oracle.threads(openmp=True)
    allc, n2 = oracle_rate(L, M, seconds_all, openmp=True)
    rows = ", ".join(f"{e['name']} {e['rows']}/{e['N']}" for e in L)
    return {"value": allc, "unit": UNIT, "cores": cores, "kind": "oracle",
            "single_thread": {"value": single, "cores": 1, "passes": n1},
            "sample": (f"{n2} pass(es) all-core and {n1} single-thread over one {model}-shaped layer at "
                       f"M = {M} (quantisation + the four products); rows multiplied per matrix: {rows}, "
                       f"each product's time scaled by N / rows; {host_cpu()}")}


def cpu_small_case_us(reps: int = 2000):
    """The small configuration (K = N = 256, M = 1) on the oracle: microseconds per call
    (quantisation + integer product), single thread."""
    import oracle
    import seeded_inputs as si
    W, x = si.gemv_case(1, 256, 256, seed=0)
    p, g = oracle.pack_ternary(W)
    t0 = time.perf_counter()
    for _ in range(reps):
        xq, sx, _ = oracle.quant_act(x)
        oracle.ternary_matmul(p, g, xq, sx)
    return (time.perf_counter() - t0) / reps * 1e6


def run_reference(args):
    """The oracle (the plain CPU implementation of the same path) as the reference arm: each
    step is one bounded pass over a row sample of the default workload on all host cores."""
    import oracle
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    L = host_oracle_layer(MODEL, 1)
    for _ in range(args.warmup):
        oracle_rate(L, 1, 0.0, openmp=True)
    t0 = time.perf_counter()
    rates = [oracle_rate(L, 1, 0.0, openmp=True)[0] for _ in range(args.steps)]
    el = time.perf_counter() - t0
    value = statistics.median(rates)
    cores = oracle.threads(openmp=True)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic",
            "config": {"workload": WORKLOAD + "; oracle step = one pass over a row sample of one layer",
                       "M": 1},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": ("one pass per step over one 2B-shaped layer (quantisation + four "
                                        "products), rows sampled per matrix, product times scaled to the "
                                        "full matrix; all cores (OpenMP over output rows); " + host_cpu())},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ GPU workload
class DecodeStack:
    """Layers of packed weights, activations and outputs resident on the GPU.

    All activation inputs of a step live in one flat device buffer and all outputs in
    another, so the end-to-end measurement moves each direction in one copy.  The first
    `distinct` layers are drawn and packed from their own seeds; further layers are
    byte copies of them in their own memory (the stream is what is measured)."""

    def __init__(self, tw, layers: int, M: int = 1, seed: int = 1234, model: str = MODEL, distinct=None,
                 layout: str = "2bit"):
        import torch
        import seeded_inputs as si
        self.tw, self.M, self.layers, self.model, self.layout = tw, M, layers, model, layout
        self.plan = layer_plan(model)
        distinct = layers if distinct is None else distinct
        n_in = layers * sum(M * K for _, N, K, _ in self.plan)
        n_out = layers * sum(M * N for _, N, K, _ in self.plan)
        self.x_all = torch.empty(n_in, dtype=torch.float32, device="cuda")
        self.y_all = torch.empty(n_out, dtype=torch.float32, device="cuda")
        self.L = []
        maxNK = max(N * K for _, N, K, _ in self.plan)
        ws = torch.empty(tw.tw_pack_workspace_bytes(1, 4), dtype=torch.uint8, device="cuda")
        maxMK = max(M * K for _, N, K, _ in self.plan)
        self.gemm_ws = tw.gemm_workspace(M, max(K for _, N, K, _ in self.plan)) if M > 4 else None
        oi = oo = 0
        for l in range(layers):
            d = {}
            for i, (name, N, K, pro) in enumerate(self.plan):
                row_bytes = tw.tw_t5_row_bytes(K) if layout == "t5" else K // 4
                packed = torch.empty((N, row_bytes), dtype=torch.uint8, device="cuda")
                gamma = torch.empty(1, dtype=torch.float32, device="cuda")
                if l < distinct:
                    W = si.device_normal((N, K), seed=seed + 1000 * l + i)
                    if layout == "t5":
                        tw.tw_pack_ternary_t5(W, packed, gamma, ws)
                    else:
                        tw.tw_pack_ternary(W, packed, gamma, ws)
                    del W
                else:
                    src = self.L[l % distinct][name]
                    packed.copy_(src["packed"])
                    gamma.copy_(src["gamma"])
                x = self.x_all[oi:oi + M * K].view(M, K)
                oi += M * K
                x.copy_(si.device_normal((M, K), seed=seed + 1000 * l + 100 + i))
                y = self.y_all[oo:oo + M * N].view(M, N)
                oo += M * N
                g = (1.0 + 0.1 * si.device_normal((K,), seed=seed + 1000 * l + 200 + i)) if pro == "rms" else None
                d[name] = dict(packed=packed, gamma=gamma, x=x, g=g, N=N, K=K, pro=pro, y=y,
                               x_q=torch.empty((M, K), dtype=torch.int8, device="cuda"),
                               s_x=torch.empty(M, dtype=torch.float32, device="cuda"),
                               x_sum=torch.empty(M, dtype=torch.int32, device="cuda"))
            self.L.append(d)
        del maxNK, maxMK
        self._fused_ok = {}
        torch.cuda.synchronize()

    def bind(self, x_all, y_all):
        """Point every GEMV's activation and output views at other flat buffers of the same
        sizes (the pipelined end-to-end loop alternates two sets)."""
        oi = oo = 0
        for d in self.L:
            for name, N, K, pro in self.plan:
                e = d[name]
                e["x"] = x_all[oi:oi + self.M * K].view(self.M, K)
                oi += self.M * K
                e["y"] = y_all[oo:oo + self.M * N].view(self.M, N)
                oo += self.M * N
        self.x_all, self.y_all = x_all, y_all

    def launches_per_step(self, fused=True):
        """Kernel launches of one step: 1 per GEMV when fused; otherwise the quantisation
        plus the GEMV (M <= 16) or plus the activation widening and the GEMM (M > 16)."""
        n = 0
        for name, N, K, pro in self.plan:
            if fused and self._fused_ok.get((N, K), True):
                n += 1
            else:
                n += 2 if self.M <= 16 else 3
        return self.layers * n

    def fused_ok(self, e):
        """Whether the fused quantisation + GEMV kernel takes this shape (decided once)."""
        if self.layout == "t5":
            return False
        key = (e["N"], e["K"])
        if key not in self._fused_ok:
            import seeded_inputs as si
            try:
                self.tw.tw_quant_gemv(e["x"], e["packed"], e["gamma"], e["y"], g=e["g"], eps=si.RMS_EPS)
                self._fused_ok[key] = True
            except self.tw.TWError as err:
                if err.status != self.tw.TW_ERR_UNSUPPORTED:
                    raise
                self._fused_ok[key] = False
        return self._fused_ok[key]

    def enqueue(self, events=None, fused=True, product_only=False):
        """Enqueue one step on the current stream (optionally with events around each GEMV).

        fused: one tw_quant_gemv launch per GEMV (quantisation fused in, programmatic
        dependent launch); otherwise tw_rmsnorm_quant_act / tw_quant_act + tw_ternary_gemv.
        product_only: leave the separate quantisation kernels out (their outputs from an
        earlier step stay in place), so that the product calls can be timed on their own."""
        import seeded_inputs as si
        tw = self.tw
        for d in self.L:
            for name, N, K, pro in self.plan:
                e = d[name]
                fz = fused and self.fused_ok(e)
                if not fz and not product_only:
                    if pro == "rms":
                        tw.tw_rmsnorm_quant_act(e["x"], e["g"], si.RMS_EPS, e["x_q"], e["s_x"], e["x_sum"])
                    else:
                        tw.tw_quant_act(e["x"], e["x_q"], e["s_x"], e["x_sum"])
                if events is not None:
                    a, b = events_new(), events_new()
                    a.record()
                if self.layout == "t5":
                    tw.tw_ternary_gemv_t5(e["packed"], e["gamma"], e["x_q"], e["s_x"], e["y"])
                elif fz:
                    tw.tw_quant_gemv(e["x"], e["packed"], e["gamma"], e["y"], g=e["g"], eps=si.RMS_EPS)
                else:
                    tw.tw_ternary_matmul(e["packed"], e["gamma"], e["x_q"], e["s_x"], e["y"], e["x_sum"],
                                         workspace=self.gemm_ws)
                if events is not None:
                    b.record()
                    events.append((name, a, b))


def events_new():
    import torch
    return torch.cuda.Event(enable_timing=True)


def gpu_sleep(ms: float):
    """Keep the current stream busy for about `ms` (torch's bounded spin kernel; ~2 GHz clock)."""
    import torch
    torch.cuda._sleep(int(ms * 2.0e6))


def capture(stack, fused, product_only=False):
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        stack.enqueue(fused=fused, product_only=product_only)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        stack.enqueue(fused=fused, product_only=product_only)
    return graph


def timed_replays(graph, steps, world):
    """Seconds for `steps` replays of `graph`, CUDA events on the replaying stream."""
    import torch
    start, stop = events_new(), events_new()
    barrier(world)
    torch.cuda.synchronize()
    start.record()
    for _ in range(steps):
        graph.replay()
    stop.record()
    torch.cuda.synchronize()
    return start.elapsed_time(stop) / 1e3


def small_case_latency(tw, reps: int = 200):
    """K = N = 256, M = 1 (the small configuration): fused quantisation + GEMV, `reps` calls
    chained in one CUDA graph; latency-bound, so reported as microseconds per call."""
    import torch
    import seeded_inputs as si
    W = si.device_normal((256, 256), seed=0)
    packed, gamma = tw.pack(W)
    x = si.device_normal((1, 256), seed=1)
    y = torch.empty((1, 256), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tw.tw_quant_gemv(x, packed, gamma, y)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            tw.tw_quant_gemv(x, packed, gamma, y)
    for _ in range(3):
        g.replay()
    el = timed_replays(g, 5, 1)
    return {"shape": "256x256, M = 1, fused quantisation", "us_per_call": el / (5 * reps) * 1e6,
            "calls_per_graph": reps}


def read_stream_rate(gib: float = 2.0):
    """A read-only streaming rate (torch.amax over a 2 GiB fp32 buffer, CUDA events): a
    third bandwidth basis next to the nominal figure and the measured copy rate."""
    import torch
    buf = torch.ones(int(gib * (1 << 30)) // 4, dtype=torch.float32, device="cuda")
    for _ in range(2):
        torch.amax(buf)
    a, b = events_new(), events_new()
    a.record()
    for _ in range(5):
        torch.amax(buf)
    b.record()
    torch.cuda.synchronize()
    gbs = 5 * buf.numel() * 4 / (a.elapsed_time(b) / 1e3) / 1e9
    del buf
    return {"GB/s": gbs, "how": "torch.amax over a 2 GiB fp32 buffer, 5 passes"}


def measure(tw, workload: str, steps: int, warmup: int, world: int, separate: bool = False, clocks=None,
            e2e_steps: int = 500):
    """GPU measurement of one workload: its decode-layer stack captured in one CUDA graph and
    replayed `steps` times (CUDA events on the replaying stream); the roofline of the product
    kernel; the same metric end to end (inputs from and outputs to pinned host memory inside
    the timed region).  Returns (result dict, stack, graph, fused)."""
    import torch
    model, layers, M, distinct = WORKLOADS[workload]
    # one token: quantisation fused into the GEMV launch; 2-4 tokens: separate kernels, which
    # measured faster (70B at 4 tokens: 241.6 against 275.4 us per layer; the fused prologue
    # quantises its tokens one after another)
    fused = (not separate) and M == 1
    stack = DecodeStack(tw, layers, M=M, model=model, distinct=distinct)
    plan = layer_plan(model)
    bytes_per_step = step_bytes(M, model, layers)
    ops_per_step = step_ops(M, model, layers)
    graph = capture(stack, fused)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: `steps` graph replays
    start, stop = events_new(), events_new()
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    if clocks is not None:
        clocks.__enter__()
    start.record()
    for _ in range(steps):
        graph.replay()
    stop.record()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.__exit__(None, None, None)
    t_wall = time.perf_counter() - t_wall0
    barrier(world)
    elapsed = start.elapsed_time(stop) / 1e3
    elapsed_max, total_bytes = combine_over_ranks(elapsed, bytes_per_step * steps, world)
    value = total_bytes / elapsed_max / 1e9
    ms_per_step = elapsed_max / steps * 1e3

    # ---- roofline of the product kernel.  Fused: every launch of the step is the product
    # kernel, so its average launch duration is the timed region over its launches.  Otherwise
    # a second graph holds only the product calls (the quantised inputs stay from earlier
    # steps) and is replayed as many times as the timed region, timed the same way.
    peak_hbm, peak_kind = measured_peaks()
    prod_calls_per_step = layers * len(plan)
    whole_step = fused and all(stack.fused_ok(stack.L[0][n]) for n, _, _, _ in plan)
    if whole_step:
        prod_elapsed = elapsed
    else:
        pgraph = capture(stack, fused, product_only=True)
        for _ in range(warmup):
            pgraph.replay()
        prod_elapsed = timed_replays(pgraph, steps, world)
        del pgraph
    avg_launch_s = prod_elapsed / (steps * prod_calls_per_step)
    if M <= 16:
        algo_per_call = bytes_per_step / prod_calls_per_step
        achieved, peak, unit, bound = algo_per_call / avg_launch_s / 1e9, peak_hbm, "GB/s", "hbm"
    else:
        algo_per_call = ops_per_step / prod_calls_per_step
        peak, pk = measured_tensor_peak()
        achieved, unit, bound, peak_kind = algo_per_call / avg_launch_s / 1e12, "TFLOP/s", "tensor", pk
    # the product kernels the library's dispatch takes for this workload's shapes
    if fused:
        kern = {"2B": "tw::gemv_decode_kernel (one token, quantisation fused)",
                "8B": "tw::gemv_decode_kernel (q|k|v, o) / gemv_stream_kernel (gate|up, down; one token, "
                      "quantisation fused)",
                "70B": "tw::gemv_stream_kernel (one token, quantisation fused)"}.get(model, "tw::gemv_decode_kernel")
    elif M <= 4:
        kern = "tw::gemv_stream_kernel / mma::gemv_mma_kernel / gemv_dp4a_kernel (by shape)"
    elif M <= 16:
        kern = "tw::mma::gemv_mma_kernel (mma.sync) / gemm kernels (by shape)"
    else:
        kern = "tw::gemm::gemm_tok_kernel / gemm_tma_kernel (tcgen05)"

    # ---- e2e: every step's inputs from pinned host memory and its outputs back to pinned host
    # memory inside the timed region (one copy each way per step).  Serial: copy in, step,
    # copy out, one after another.  Pipelined (the reported e2e): two sets of device buffers
    # and two graphs; the upload of step t + 1 and the download of step t - 1 run on their own
    # streams while step t computes, ordered by events (a buffer is refilled only after the
    # step that read it, and overwritten only after its outputs were downloaded).
    h_in = stack.x_all.cpu().pin_memory()
    h_out = torch.empty(stack.y_all.shape, dtype=torch.float32).pin_memory()
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size()
    n_e2e = max(1, min(steps, e2e_steps))

    def e2e_step():
        stack.x_all.copy_(h_in, non_blocking=True)
        graph.replay()
        h_out.copy_(stack.y_all, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = events_new(), events_new()
    e0.record()
    for _ in range(n_e2e):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    serial_el, serial_bytes = combine_over_ranks(e0.elapsed_time(e1) / 1e3, bytes_per_step * n_e2e, world)

    xs_ = [stack.x_all, torch.empty_like(stack.x_all)]
    ys_ = [stack.y_all, torch.empty_like(stack.y_all)]
    stack.bind(xs_[1], ys_[1])
    graph_b = capture(stack, fused)
    stack.bind(xs_[0], ys_[0])
    graphs = [graph, graph_b]
    h_ins = [h_in, h_in.clone().pin_memory()]
    h_outs = [h_out, torch.empty_like(h_out).pin_memory()]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def pipelined(n):
        ev = lambda: torch.cuda.Event()
        ev_in, ev_comp, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        start, stop = events_new(), events_new()
        start.record(comp)
        s_in.wait_event(start)
        with torch.cuda.stream(s_in):
            xs_[0].copy_(h_ins[0], non_blocking=True)
            ev_in[0].record(s_in)
        for t in range(n):
            b = t % 2
            comp.wait_event(ev_in[b])
            if t >= 2:
                comp.wait_event(ev_out[b])  # the outputs of step t - 2 have been downloaded
            graphs[b].replay()
            ev_comp[b].record(comp)
            if t + 1 < n:
                nb = 1 - b
                with torch.cuda.stream(s_in):
                    if t >= 1:
                        s_in.wait_event(ev_comp[nb])  # step t - 1 has read its inputs
                    xs_[nb].copy_(h_ins[nb], non_blocking=True)
                    ev_in[nb].record(s_in)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b])
                h_outs[b].copy_(ys_[b], non_blocking=True)
                ev_out[b].record(s_out)
        comp.wait_event(ev_out[0])
        comp.wait_event(ev_out[1])
        stop.record(comp)
        return start, stop

    pipelined(3)
    torch.cuda.synchronize()
    barrier(world)
    p0, p1 = pipelined(n_e2e)
    torch.cuda.synchronize()
    e2e_el, e2e_bytes = combine_over_ranks(p0.elapsed_time(p1) / 1e3, bytes_per_step * n_e2e, world)
    del graph_b

    res = {"value": value, "unit": UNIT, "ms_per_step": ms_per_step,
           "us_per_layer": ms_per_step * 1e3 / layers, "M": M, "layers": layers,
           "bytes_per_step": bytes_per_step, "int_ops_per_step": ops_per_step,
           "launches_per_step": stack.launches_per_step(fused),
           "quantisation": "fused into the GEMV launch" if fused else "separate kernels",
           "TFLOP/s": ops_per_step * steps * world / elapsed_max / 1e12,
           "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                        "frac": achieved / peak, "kernel": kern, "peak_source": peak_kind,
                        "algorithmic_per_launch": algo_per_call, "avg_launch_us": avg_launch_s * 1e6,
                        "timing": (("timed region / product launches" if whole_step else
                                    "graph of the product calls only, replayed like the timed region")
                                   + "; launches overlap under programmatic dependent launch, so this is "
                                     "step time / launches, not one kernel's duration")},
           "e2e": {"value": e2e_bytes / e2e_el / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h, "steps": n_e2e,
                   "how": "pipelined: two buffer sets, uploads and downloads on their own streams overlap "
                          "the neighbouring steps' computation; every step's inputs and outputs cross",
                   "serial": {"value": serial_bytes / serial_el / 1e9, "unit": UNIT,
                              "how": "copy in, step, copy out, one after another"}},
           "wall_s_timed": t_wall, "elapsed_s": elapsed_max}
    return res, stack, graph, fused


def per_shape_isolated(stack, fused, M, plan):
    """Each product call on its own: events around each call of extra steps enqueued behind
    a short GPU sleep (host launch overhead hidden; no overlap with the next call)."""
    import torch
    shapes = {name: (N, K) for name, N, K, _ in plan}
    per_launch = {}
    for rep in range(3):
        evs = []
        gpu_sleep(30.0)
        stack.enqueue(events=evs, fused=fused)
        torch.cuda.synchronize()
        if rep == 0:
            continue
        for name, a, b in evs:
            per_launch.setdefault(name, []).append(a.elapsed_time(b) / 1e3)
    return {n: {"bytes": gemv_bytes(*shapes[n], M), "us_median": statistics.median(v) * 1e6,
                "GB/s": gemv_bytes(*shapes[n], M) / statistics.median(v) / 1e9,
                "TFLOP/s": 2 * M * shapes[n][0] * shapes[n][1] / statistics.median(v) / 1e12}
            for n, v in per_launch.items()}


def epilogue_chain(tw, steps: int, warmup: int):
    """The 2B decode step (30 layers, one token) with the fused epilogues: q|k|v and gate|up
    quantise from the partial statistics the o and down launches left, which add their
    output to the residual stream in their epilogue.  Per layer: q|k|v (RMSNorm from finished
    statistics), o (quantisation of its synthetic input, GEMV, residual add, statistics of
    the next RMSNorm), gate|up (as q|k|v), down (as o).  One residual buffer, updated in
    place; one CUDA graph per step, timed like the main line."""
    import torch
    import seeded_inputs as si
    stack = DecodeStack(tw, LAYERS, M=1)
    hid = layer_plan(MODEL)[1][1]  # o: N = hidden
    h = si.device_normal((hid,), seed=77)
    ws = tw.epilogue_workspace()
    gains = [1.0 + 0.1 * si.device_normal((hid,), seed=900 + i) for i in range(2 * LAYERS)]

    def enqueue():
        for l, d in enumerate(stack.L):
            g_attn, g_ffn = gains[2 * l], gains[2 * l + 1]
            g_attn_next = gains[(2 * l + 2) % (2 * LAYERS)]
            e = d["qkv"]
            tw.tw_quant_gemv_stats(h, g_attn, ws, e["packed"], e["gamma"], e["y"], eps=si.RMS_EPS)
            e = d["o"]
            tw.tw_quant_gemv_residual(e["x"], e["packed"], e["gamma"], h, h, g_ffn, ws, eps=si.RMS_EPS, y=e["y"])
            e = d["gateup"]
            tw.tw_quant_gemv_stats(h, g_ffn, ws, e["packed"], e["gamma"], e["y"], eps=si.RMS_EPS)
            e = d["down"]
            tw.tw_quant_gemv_residual(e["x"], e["packed"], e["gamma"], h, h, g_attn_next, ws, eps=si.RMS_EPS,
                                      y=e["y"])

    def enqueue_unfused():
        # the same dataflow without the epilogue: RMSNorm over h in the q|k|v and gate|up
        # launches, the residual adds as separate (library) kernels after o and down
        h2 = h.view(1, -1)
        for l, d in enumerate(stack.L):
            g_attn, g_ffn = gains[2 * l], gains[2 * l + 1]
            e = d["qkv"]
            tw.tw_quant_gemv(h2, e["packed"], e["gamma"], e["y"], g=g_attn, eps=si.RMS_EPS)
            e = d["o"]
            tw.tw_quant_gemv(e["x"], e["packed"], e["gamma"], e["y"])
            h2.add_(e["y"])
            e = d["gateup"]
            tw.tw_quant_gemv(h2, e["packed"], e["gamma"], e["y"], g=g_ffn, eps=si.RMS_EPS)
            e = d["down"]
            tw.tw_quant_gemv(e["x"], e["packed"], e["gamma"], e["y"])
            h2.add_(e["y"])

    def timed(fn):
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            fn()
        torch.cuda.current_stream().wait_stream(st)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        for _ in range(warmup):
            graph.replay()
        el = timed_replays(graph, steps, 1)
        del graph
        return el

    # statistics for the very first q|k|v: one down-projection residual call
    e = stack.L[-1]["down"]
    tw.tw_quant_gemv_residual(e["x"], e["packed"], e["gamma"], h, h, gains[0], ws, y=e["y"])
    el = timed(enqueue)
    status = tw.tw_device_status()
    el_unfused = timed(enqueue_unfused)
    nbytes = step_bytes(1)
    del stack
    torch.cuda.empty_cache()
    return {"us_per_layer": el / steps / LAYERS * 1e6, "GB/s": nbytes * steps / el / 1e9,
            "bytes_per_step": nbytes, "launches_per_step": 4 * LAYERS, "device_status": status,
            "chain": "qkv (RMSNorm from finished statistics) -> o (+ residual, next statistics) -> gate|up "
                     "(finished statistics) -> down (+ residual, next statistics)",
            "us_per_layer_residual_unfused": el_unfused / steps / LAYERS * 1e6,
            "unfused": "the same dataflow: RMSNorm + quantisation fused into each GEMV launch, the two residual "
                       "adds as separate torch kernels (6 launches per layer)"}


def t5_comparison(tw, steps: int, warmup: int, copies: int = 4, reps: int = 5):
    """The five-trits-per-byte layout next to the 2-bit one: the 2B decode step (30 layers,
    quantisation as its own kernel before each product, one CUDA graph) in both layouts,
    and each layout's product alone on a large matrix (the 70B gate|up, 57344 x 8192, four
    copies so the stream leaves L2).  Weights per second is the comparable figure: the
    five-trit layout moves 20 % fewer bytes for the same weights."""
    import torch
    import seeded_inputs as si
    out = {}
    for layout in ("2bit", "t5"):
        stack = DecodeStack(tw, LAYERS, M=1, layout=layout)
        graph = capture(stack, fused=False)
        for _ in range(warmup):
            graph.replay()
        el = timed_replays(graph, steps, 1)
        plan = layer_plan(MODEL)
        nbytes = LAYERS * sum((gemv_bytes_t5 if layout == "t5" else gemv_bytes)(N, K) for _, N, K, _ in plan)
        weights = LAYERS * sum(N * K for _, N, K, _ in plan)
        out[f"2b_step_{layout}"] = {"us_per_layer": el / steps / LAYERS * 1e6,
                                    "GB/s": nbytes * steps / el / 1e9,
                                    "Gweights/s": weights * steps / el / 1e9,
                                    "bytes_per_step": nbytes, "launches_per_step": stack.launches_per_step(False)}
        del graph, stack
        torch.cuda.empty_cache()
    N, K = 57344, 8192
    ws = torch.empty(tw.tw_pack_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    x = si.device_normal((1, K), seed=5)
    xq, sx, xs = tw.quantize(x)
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    for layout in ("2bit", "t5"):
        packs = []
        for c in range(copies):
            W = si.device_normal((N, K), seed=300 + c)
            packs.append(tw.pack_t5(W) if layout == "t5" else tw.pack(W))
            del W

        def one_pass():
            for p, g in packs:
                if layout == "t5":
                    tw.tw_ternary_gemv_t5(p, g, xq, sx, y)
                else:
                    tw.tw_ternary_gemv(p, g, xq, sx, y, xs)

        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            one_pass()
        torch.cuda.current_stream().wait_stream(st)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one_pass()
        for _ in range(3):
            graph.replay()
        el = timed_replays(graph, reps, 1)
        us = el / (reps * copies) * 1e6
        nbytes = (gemv_bytes_t5 if layout == "t5" else gemv_bytes)(N, K)
        out[f"gemv_{N}x{K}_{layout}"] = {"us_per_launch": us, "GB/s": nbytes / us / 1e3,
                                          "Gweights/s": N * K / us / 1e3}
        del graph, packs
        torch.cuda.empty_cache()
    return out


# The other configurations, measured in the default run (each line's own roofline and CPU
# baseline): small steps, since each workload's graph is replayed back to back.
OTHER_WORKLOADS = ["2b_m8", "2b_m64", "2b_m256", "8b_m1", "8b_m16", "70b_m1", "70b_m4", "70b_m16"]


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    import ternary_weight_quant_b300 as tw

    model, layers, M, distinct = WORKLOADS[args.workload]
    plan = layer_plan(model)
    clocks = ClockSampler(local)
    res, stack, graph, fused = measure(tw, args.workload, args.steps, args.warmup, world, args.separate,
                                       clocks=clocks)
    per_shape = per_shape_isolated(stack, fused, M, plan)
    value = res["value"]
    peak_hbm, _ = measured_peaks()

    # ---- default workload only: the unfused variant of the same step, the smallest case's
    # latency per call, a read-only streaming rate as a third bandwidth basis, and every other
    # configuration with its own roofline and CPU baseline
    extra = {}
    default = args.workload == "2b" and not args.separate and not args.no_extras
    if default:
        ugraph = capture(stack, fused=False)
        for _ in range(args.warmup):
            ugraph.replay()
        u_el = timed_replays(ugraph, args.steps, world)
        extra["us_per_layer_unfused"] = u_el / args.steps / layers * 1e6
        extra["launches_per_step_unfused"] = stack.launches_per_step(False)
        del ugraph
    del graph, stack
    torch.cuda.empty_cache()
    if default:
        extra["small_case"] = small_case_latency(tw)
        extra["read_stream"] = read_stream_rate()
        extra["five_trits_per_byte"] = t5_comparison(tw, min(args.steps, 200), args.warmup)
        extra["fused_epilogue"] = epilogue_chain(tw, args.steps, args.warmup)
    cpu_ok = rank == 0 and world == 1 and not args.no_cpu_baseline
    if default and cpu_ok:
        extra["small_case"]["cpu_oracle_us_per_call_single_thread"] = cpu_small_case_us()
    if default and not args.no_workloads:  # (--no-extras leaves `default` false)
        wl = {}
        for name in OTHER_WORKLOADS:
            r, st, gr, _ = measure(tw, name, args.workload_steps, 3, world)
            del st, gr
            torch.cuda.empty_cache()
            wmodel, wlayers, wM, wdistinct = WORKLOADS[name]
            r["workload"] = (f"{wmodel}-shaped decoder layer, batch {wM} ({SHAPE_TEXT[wmodel]}), {wlayers} layers "
                             f"({wdistinct} drawn, the rest byte copies in their own memory)"
                             + ("; activations N(0,1) with 1 % outliers x20" if wmodel == "2B" else ""))
            if cpu_ok:
                r["cpu_baseline"] = cpu_baseline_for(wmodel, wM, args.cpu_seconds_workload,
                                                     args.cpu_seconds_workload, outliers=(wmodel == "2B"))
            wl[name] = r
        extra["workloads"] = wl

    # ---- CPU baseline: the oracle on the host, bounded sample (rank 0, N = 1)
    cpu = None
    if cpu_ok:
        cpu = cpu_baseline_for(model, M, args.cpu_seconds, args.cpu_seconds / 2,
                               outliers=(model == "2B" and M > 1))

    if rank == 0:
        workload = (WORKLOAD if args.workload == "2b" else
                    f"{model}-shaped decoder layer, batch {M} ({SHAPE_TEXT[model]}), {layers} layers "
                    f"({distinct} drawn, the rest byte copies in their own memory)")
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
            "config": {"workload": workload, "M": M, "layers": layers,
                       "bytes_per_step": res["bytes_per_step"], "int_ops_per_step": res["int_ops_per_step"],
                       "launches_per_step": res["launches_per_step"],
                       "quantisation": res["quantisation"],
                       "graph": "one CUDA graph per step",
                       "l2": f"working set {res['bytes_per_step'] / 1e6:.0f} MB of packed weights, > 4x the "
                             "126 MB L2; no flush needed",
                       "parallelism": f"replicas x{world}"},
            "us_per_layer": res["us_per_layer"],
            "TFLOP/s": res["TFLOP/s"],
            "pct_of_nominal_8TBs": 100.0 * value / world / NOMINAL_HBM_GBS,
            "pct_of_measured_copy": 100.0 * value / world / peak_hbm,
            **({"pct_of_measured_read": 100.0 * value / world / extra["read_stream"]["GB/s"]}
               if "read_stream" in extra else {}),
            **extra,
            "roofline": {**res["roofline"],
                         "traffic": recorded_traffic(args.workload) if fused else None,
                         "per_shape_isolated": per_shape},
            "cpu_baseline": cpu,
            "e2e": res["e2e"],
            "gpu_launches": res["launches_per_step"] * args.steps,
            "clocks": clocks.summary(),
            "wall_s_timed": res["wall_s_timed"],
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_kernel_case(args):
    """Kernels in isolation (for timing sweeps and small ncu captures; not the contract line).

    --kernel-case {gemv,t5,fused,fused_rms,residual,stats,quant,rms_quant,gemm,gemm_nows,matmul}
    (a comma list) on --shape NxK at --M tokens (a comma list), over --copies distinct weight
    tensors (so the stream leaves L2); one pass over them is captured in a CUDA graph and
    replayed --reps times (device time per launch, host launch cost excluded).  One JSON line
    per (case, M).  residual and stats take one token."""
    import torch
    import seeded_inputs as si
    torch.cuda.set_device(0)
    import ternary_weight_quant_b300 as tw
    N, K = (int(v) for v in args.shape.lower().split("x"))
    ws = torch.empty(tw.tw_pack_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    cases = args.kernel_case.split(",")
    packs, packs5 = [], []
    epi_ws = tw.epilogue_workspace() if any(k in ("residual", "stats") for k in cases) else None
    for c in range(args.copies):
        W = si.device_normal((N, K), seed=77 + c)
        if any(k != "t5" for k in cases):
            p = torch.empty((N, K // 4), dtype=torch.uint8, device="cuda")
            g = torch.empty(1, dtype=torch.float32, device="cuda")
            tw.tw_pack_ternary(W, p, g, ws)
            packs.append((p, g))
        if "t5" in cases:
            packs5.append(tw.pack_t5(W))
        del W
    gain = 1.0 + 0.1 * si.device_normal((K,), seed=6)
    for M in (int(v) for v in str(args.M).split(",")):
        x = si.device_normal((M, K), seed=5)
        xq, sx, xs = tw.quantize(x)
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        gws = tw.gemm_workspace(M, K)
        if epi_ws is not None:
            # residual case: the residual stream has N elements; stats case: x has K elements, and
            # the partial statistics come from one residual call over K outputs first
            hN = si.device_normal((N,), seed=11)
            hK = si.device_normal((K,), seed=12)
            gN = 1.0 + 0.1 * si.device_normal((N,), seed=13)
            pKK = tw.pack(si.device_normal((K, K), seed=14))
            xK = si.device_normal((1, K), seed=15)
            tw.tw_quant_gemv_residual(xK, pKK[0], pKK[1], hK, hK, gain, epi_ws)
        for k in cases:

            def launch(p, g):
                if k == "residual":
                    tw.tw_quant_gemv_residual(x, p, g, hN, hN, gN, epi_ws, y=y)
                elif k == "stats":
                    tw.tw_quant_gemv_stats(hK, gain, epi_ws, p, g, y)
                elif k == "t5":
                    tw.tw_ternary_gemv_t5(p, g, xq, sx, y)
                elif k == "gemv":
                    tw.tw_ternary_gemv(p, g, xq, sx, y, xs)
                elif k in ("fused", "fused_rms"):
                    tw.tw_quant_gemv(x, p, g, y, g=gain if k == "fused_rms" else None)
                elif k == "quant":
                    tw.tw_quant_act(x, xq, sx, xs)
                elif k == "rms_quant":
                    tw.tw_rmsnorm_quant_act(x, gain, 1e-6, xq, sx, xs)
                elif k == "gemm":
                    tw.tw_ternary_gemm(p, g, xq, sx, y, workspace=gws)
                elif k == "gemm_nows":
                    tw.tw_ternary_gemm(p, g, xq, sx, y)
                elif k == "matmul":
                    tw.tw_ternary_matmul(p, g, xq, sx, y, xs, workspace=gws)
                else:
                    raise SystemExit(f"unknown kernel case {k}")

            def one_pass():
                for p, g in (packs5 if k == "t5" else packs):
                    launch(p, g)

            try:
                # one pass over the copies captured in a CUDA graph, so host launch cost does not show
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(s):
                    one_pass()  # warm-up (and lazy initialisation) outside the capture
                torch.cuda.current_stream().wait_stream(s)
                torch.cuda.synchronize()
            except tw.TWError as e:
                print(json.dumps({"kernel_case": k, "N": N, "K": K, "M": M, "unsupported": str(e)}))
                continue
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                one_pass()
            for _ in range(3):
                graph.replay()
            torch.cuda.synchronize()
            a, b = events_new(), events_new()
            a.record()
            for _ in range(args.reps):
                graph.replay()
            b.record()
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / (args.copies * args.reps)
            nbytes = gemv_bytes_t5(N, K, M) if k == "t5" else gemv_bytes(N, K, M)
            print(json.dumps({"kernel_case": k, "N": N, "K": K, "M": M, "us_per_launch": us,
                              "GB/s": nbytes / us / 1e3, "Gweights/s": N * K / us / 1e3,
                              "TFLOP/s": 2 * M * N * K / us / 1e6}),
                  flush=True)
            del graph
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--separate", action="store_true", help="quantisation as separate kernels")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="2b",
                    help="2b (the default decode-layer configuration), 2b_m8/m64/m256, 8b_m1/m16, 70b_m1/m4/m16")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="single-thread seconds of the CPU baseline (all cores: half of it)")
    ap.add_argument("--cpu-seconds-workload", type=float, default=2.0,
                    help="seconds of each CPU baseline of the other configurations (single and all-core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="default run: leave out the other configurations")
    ap.add_argument("--workload-steps", type=int, default=10, help="timed steps of each other configuration")
    ap.add_argument("--no-extras", action="store_true",
                    help="default workload: skip the unfused step, small case, read stream, five-trit and "
                         "epilogue measurements (and the other configurations)")
    ap.add_argument("--kernel-case", default=None,
                    help="time one kernel alone: gemv, t5, fused, fused_rms, residual, stats, quant, rms_quant, gemm, "
                         "gemm_nows or matmul")
    ap.add_argument("--shape", default="13824x2560", help="NxK for --kernel-case")
    ap.add_argument("--M", default="1", help="tokens for --kernel-case (a comma list)")
    ap.add_argument("--copies", type=int, default=8, help="distinct weight tensors for --kernel-case")
    ap.add_argument("--reps", type=int, default=3, help="passes over the copies for --kernel-case")
    args = ap.parse_args()
    if args.kernel_case:
        return run_kernel_case(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
