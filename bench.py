"""Benchmark of the GB300 GPTQ linear layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

One step is one gptq_gemm call (the whole per-call hot path: activation permute, packed-weight
stream, dequant, MMA, reduction, y store) on the Llama-3-70B gate_proj layer (K=8192, N=28672,
4-bit, group 128, act-order, asymmetric zeros, fp16) at M=1, the largest M=1 configuration.
Successive steps use successive weight sets of an 8-layer resident stack, so the working set
(977 MB) is larger than L2 and no step reads weights another step left in L2.  Inputs are
synthetic and seeded.

value  = algorithmic bytes moved per call (packed weights + scales + packed zeros + perm + x + y)
         divided by the time per call, summed over ranks (one replica per GPU).  The time per call
         is the median over repeated replays of a CUDA graph of `steps` calls, replayed until at
         least 200 ms have been timed.
e2e    = the same metric through the public API with host buffers: pinned x copied to the
         device, gptq_gemm, y copied back, every step (the copies on two side streams, overlapping
         the neighbouring steps' GEMMs).
Also reported (rank 0): the Llama-3-8B decode layer at M=1 (decode_m1) and the prefill layer at
M=4096 (prefill_m4096) as top-level keys, more M values and formats under detail, and the oracle
timed on the host cores (cpu_baseline).

--impl reference times the CPU oracle (the only reference this build has: the pages publish
no runnable code) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "llama3-70b-gate-8192x28672-b4g128-descact"
DECODE = "llama3-8b-decode-4096x14336-b4g128-sym"
PREFILL = "prefill-8192x28672-b4g128"
METRIC = "GPTQ W4A16 GEMM µs/call, HBM GB/s (M=1), TFLOP/s (M=4096), % roofline"
LAYERS = 8
MIN_TIMED_S = 0.2
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def b_alg(spec, M: int) -> int:
    """Algorithmic bytes of one call: what the method has to move."""
    K, N, b, G = spec.K, spec.N, spec.bits, spec.G
    return K * N * b // 8 + 2 * G * N + G * N * b // 8 + (4 * K if spec.desc_act else 0) + 2 * M * K + 2 * M * N


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def code_sha256(text: str) -> str:
    """SHA-256 of a source with its comments removed and whitespace collapsed: edits to comments do
    not change the kernel the counters were taken on."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()


def traffic_record(kernel_file: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel on this workload, if the
    kernel's code is unchanged since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(f"{kernel_file}:{workload}", {})
        src = open(os.path.join(ROOT, "weight_only_quantized_gb300", "csrc", kernel_file)).read()
        if rec.get("code_sha256") == code_sha256(src):
            return rec
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,utilization.gpu,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.path = index, None, None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 8:
                    rows.append(f)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        busy = [r for r in rows if r[3] not in ("0", "[N/A]")] or rows
        mhz = [float(r[1]) for r in busy if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": reasons, "samples": len(busy)}


def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, v: float) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- oracle arm
def oracle_sample_rate(spec, M: int, seconds: float, cols_per_call: int):
    """Oracle GB/s on column samples of the workload: bytes scaled by the sampled fraction."""
    import numpy as np

    import oracle
    from weight_only_quantized_gb300 import synth
    ck = synth.make_checkpoint(spec, seed=0)
    x = synth.make_x(M, spec.K, spec.dtype, seed=1)
    cols_per_call = min(cols_per_call, spec.N)
    rng = np.random.default_rng(0)
    calls, t_total = 0, 0.0
    while t_total < seconds or calls == 0:
        cols = np.sort(rng.choice(spec.N, cols_per_call, replace=False)).astype(np.int32)
        t0 = time.perf_counter()
        oracle.linear(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, spec.bits, spec.group_size, spec.dtype, x,
                      None, cols)
        t_total += time.perf_counter() - t0
        calls += 1
    frac = cols_per_call / spec.N
    gbs = b_alg(spec, M) * frac * calls / t_total / 1e9
    return gbs, calls, t_total, oracle.num_threads(), f"{calls} oracle calls on {cols_per_call} of {spec.N} output columns (all K, M={M}), {t_total:.1f} s"


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    from weight_only_quantized_gb300 import synth
    spec, _ = synth.workload(WORKLOAD)
    M = 1
    # each step: one oracle call on a fixed-size column sample
    cols = 512
    import numpy as np
    import oracle
    ck = synth.make_checkpoint(spec, seed=0)
    x = synth.make_x(M, spec.K, spec.dtype, seed=1)
    rng = np.random.default_rng(0)
    for _ in range(max(0, args.warmup - 1)):
        c = np.sort(rng.choice(spec.N, cols, replace=False)).astype(np.int32)
        oracle.linear(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, spec.bits, spec.group_size, spec.dtype, x, None, c)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        c = np.sort(rng.choice(spec.N, cols, replace=False)).astype(np.int32)
        oracle.linear(ck.qweight, ck.qzeros, ck.scales, ck.g_idx, spec.bits, spec.group_size, spec.dtype, x, None, c)
    dt = time.perf_counter() - t0
    frac = cols / spec.N
    value = b_alg(spec, M) * frac * args.steps / dt / 1e9
    sample = f"each step: oracle on {cols} of {spec.N} output columns, all K, M={M}; bytes scaled by {frac:.4f}"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "K": spec.K, "N": spec.N, "bits": spec.bits,
                       "group_size": spec.group_size, "act_order": spec.desc_act,
                       "parallelism": "rank 0 only (host cores)"},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- native arm
def make_layers(spec, count, seed0=0, distinct=False):
    """`count` resident handles of the layer: repacks of one seeded checkpoint (distinct=False; the
    handles are separate device copies, so each call streams its own weights from HBM) or of
    `count` checkpoints with successive seeds."""
    import torch
    from weight_only_quantized_gb300 import gptq, synth
    hs, cks = [], []
    dev = None
    for i in range(count):
        if distinct or i == 0:
            ck = synth.make_checkpoint(spec, seed=seed0 + i)
            dev = [t.cuda() if t is not None else None for t in (ck.qweight, ck.qzeros, ck.scales, ck.g_idx)]
            cks.append(ck)
        hs.append(gptq.gptq_repack(dev[0], dev[1], dev[2], dev[3], spec.bits, spec.group_size))
    del dev
    torch.cuda.synchronize()
    return hs, cks


def time_calls(hs, xs, ys, M, steps, warmup, graph=True, min_total_s=MIN_TIMED_S, min_reps=5):
    """Per-call device time (s) of `steps` calls rotating over the handles.

    graph=True: the `steps` calls are captured once into a CUDA graph (how a decode step is
    deployed); the graph is replayed until at least `min_total_s` of replays (and at least five)
    have been timed, each replay bracketed by CUDA events on the replay stream, and the median
    replay time / steps is returned.  graph=False: eager launches from the host, events around the
    loop, repeated the same way.  (min_total_s = 0, min_reps = 1: exactly `steps` timed calls.)"""
    import torch
    from weight_only_quantized_gb300 import gptq
    n = len(hs)
    st = torch.cuda.current_stream()
    for i in range(warmup):
        gptq.gptq_gemm(hs[i % n], xs[i % len(xs)], ys[i % len(ys)], M, st)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g = None
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(steps):
                gptq.gptq_gemm(hs[i % n], xs[i % len(xs)], ys[i % len(ys)], M)
        torch.cuda.synchronize()
        g.replay()                      # untimed replay: graph upload and first-touch effects
        torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    times, total = [], 0.0
    while total < min_total_s or len(times) < min_reps:
        t0.record(st)
        if graph:
            g.replay()
        else:
            for i in range(steps):
                gptq.gptq_gemm(hs[i % n], xs[i % len(xs)], ys[i % len(ys)], M, st)
        t1.record(st)
        torch.cuda.synchronize()
        dt = t0.elapsed_time(t1) / 1e3
        times.append(dt / steps)
        total += dt
    del g
    return statistics.median(times)


def layer_line(spec, M, t, hbm, tf_burst, tf_sus):
    """One (layer, M) result: time, GB/s, TFLOP/s and the roofline fraction (burst and sustained
    bf16 peaks for tensor-bound cases)."""
    B, F = b_alg(spec, M), 2.0 * M * spec.N * spec.K
    roof = max(B / (hbm * 1e9), F / (tf_burst * 1e12))
    r = {"us": round(t * 1e6, 2), "GB/s": round(B / t / 1e9, 1), "TFLOP/s": round(F / t / 1e12, 2),
         "roofline_frac": round(roof / t, 4),
         "bound": "hbm" if B / (hbm * 1e9) >= F / (tf_burst * 1e12) else "tensor"}
    if r["bound"] == "tensor":
        r["roofline_frac_sustained"] = round(max(B / (hbm * 1e9), F / (tf_sus * 1e12)) / t, 4)
    return r


def run_native(args, ws, rank, local):
    import torch
    from weight_only_quantized_gb300 import gptq, synth
    hbm, tf_burst, tf_sus, peak_kind = peaks()
    spec, _ = synth.workload(WORKLOAD)
    M = 1
    dt = torch.float16 if spec.dtype == "fp16" else torch.bfloat16
    hs, _ = make_layers(spec, LAYERS)
    xs = [synth.make_x(M, spec.K, spec.dtype, seed=100 + i).cuda() for i in range(LAYERS)]
    ys = [torch.empty(M, spec.N, dtype=dt, device="cuda") for _ in range(LAYERS)]
    launches_per_call = gptq.gptq_gemm_launches(hs[0], M)
    plan = gptq.gptq_gemm_plan(hs[0], M)

    def measure():
        barrier(ws)
        torch.cuda.synchronize()
        total = time_calls(hs, xs, ys, M, args.steps, args.warmup, graph=True)
        barrier(ws)
        eager = time_calls(hs, xs, ys, M, args.steps, args.warmup, graph=False)
        barrier(ws)
        return max_over_ranks(ws, total), max_over_ranks(ws, eager)

    def measure_e2e():
        # End to end through the public API with host buffers, every step: pinned x copied in,
        # gptq_gemm, y copied back.  The copies run on two side streams, so step i + 1's x copy and
        # step i - 1's y copy overlap step i's GEMM (a serving loop's double buffering); events order
        # each buffer's reuse.  The timed region runs from before the first copy in to after the last
        # copy out.
        xh = [synth.make_x(M, spec.K, spec.dtype, seed=100 + i).pin_memory() for i in range(LAYERS)]
        yh = [torch.empty(M, spec.N, dtype=dt).pin_memory() for _ in range(LAYERS)]
        st = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(LAYERS)]
        ev_k = [torch.cuda.Event() for _ in range(LAYERS)]
        ev_out = [torch.cuda.Event() for _ in range(LAYERS)]

        def run(steps):
            run_on(st, steps)

        def run_on(sc, steps):
            for i in range(steps):
                j = i % LAYERS
                if i >= LAYERS:
                    s_in.wait_event(ev_k[j])            # the GEMM that read x[j] is done
                with torch.cuda.stream(s_in):
                    xs[j].copy_(xh[j], non_blocking=True)
                ev_in[j].record(s_in)
                sc.wait_event(ev_in[j])
                if i >= LAYERS:
                    sc.wait_event(ev_out[j])            # y[j] of the earlier step has been copied out
                gptq.gptq_gemm(hs[j], xs[j], ys[j], M, sc)
                ev_k[j].record(sc)
                s_out.wait_event(ev_k[j])
                with torch.cuda.stream(s_out):
                    yh[j].copy_(ys[j], non_blocking=True)
                ev_out[j].record(s_out)
            for j in range(min(steps, LAYERS)):
                sc.wait_event(ev_out[j])

        run(args.warmup)
        torch.cuda.synchronize()
        # the `steps` steps on the three streams captured once into a CUDA graph (the host enqueue of
        # ~10 calls a step would otherwise bound the loop), replayed like the device-timed value
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(st)
        with torch.cuda.graph(g, stream=cap):
            st_cap = torch.cuda.current_stream()
            fork = torch.cuda.Event()
            fork.record(st_cap)
            s_in.wait_event(fork)
            s_out.wait_event(fork)
            run_on(st_cap, args.steps)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times, tot = [], 0.0
        while tot < MIN_TIMED_S or len(times) < 5:
            e0.record(st)
            g.replay()
            e1.record(st)
            torch.cuda.synchronize()
            d = e0.elapsed_time(e1) / 1e3
            times.append(d / args.steps)
            tot += d
        del g
        return max_over_ranks(ws, statistics.median(times))

    with ClockSampler(local) as clk:
        total, eager = measure()
        e2e_t = measure_e2e()
        barrier(ws)
        extra = {} if (args.no_extra or rank != 0) else extra_workloads(args, hbm, tf_burst, peak_kind, tf_sus)
    clocks = clk.summary()
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"} & set(clocks["reasons"])
    if bad and not args._remeasured:
        args._remeasured = True
        with ClockSampler(local) as clk:
            total, eager = measure()
        clocks = clk.summary()

    B = b_alg(spec, M)
    value = B * ws / total / 1e9
    achieved = B / total / 1e9
    traffic = traffic_record("gemm_small.cu", WORKLOAD)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total * 1e3, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": spec.dtype, "data": "synthetic",
        "us_per_call": round(total * 1e6, 3),
    }
    # the other two headline configurations, small and at the top of the line
    for key in ("decode_m1", "prefill_m4096"):
        if key in extra:
            line[key] = extra.pop(key)
    line.update({
        "config": {"workload": WORKLOAD, "M": M, "K": spec.K, "N": spec.N, "bits": spec.bits,
                   "group_size": spec.group_size, "act_order": spec.desc_act, "zero": "asymmetric",
                   "act_dtype": spec.dtype, "layers_rotated": LAYERS,
                   "l2": f"inputs larger than L2: {LAYERS} resident weight sets ({LAYERS * B / 1e6:.0f} MB) "
                         f"rotated per step", "parallelism": f"replicas x{ws}", "bytes_per_call": B,
                   "kernel_plan": {"path": "small-M" if plan.path == gptq.PATH_SMALL_M else "large-M",
                                   "launches": plan.launches, "grid": plan.grid,
                                   "consumer_warps": plan.consumer_warps,
                                   "act_order_in_kernel": plan.act_order_in_kernel, "stages": plan.stages}},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                     "traffic": traffic["dram_bytes_per_launch"] if traffic else None,
                     "kernel": "k_gemm_small (small-M: persistent TMA-fed weight stream, mma.sync swap-AB)",
                     "timing": "CUDA events around each replay of a graph of the timed calls; median over "
                               f"replays totalling >= {MIN_TIMED_S * 1e3:.0f} ms"},
        "eager_us_per_call": round(eager * 1e6, 3),
        "e2e": {"value": round(B * ws / e2e_t / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": 2 * M * spec.K,
                "d2h_bytes_per_step": 2 * M * spec.N, "us_per_step": round(e2e_t * 1e6, 3),
                "how": "pinned x in, gptq_gemm, y out every step; copies on two side streams overlap the "
                       "neighbouring steps' GEMMs; the steps replayed as one CUDA graph"},
        "gpu_launches": launches_per_call * args.steps,
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
    })
    if rank == 0 and not args.no_cpu_baseline:
        gbs, calls, secs, cores, sample = oracle_sample_rate(spec, M, args.cpu_seconds, 2048)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
        # the same oracle on one host core (a separate figure; the line's value is the all-core one)
        import oracle
        oracle.set_num_threads(1)
        g1, _, _, _, s1 = oracle_sample_rate(spec, M, args.cpu_seconds / 2, 256)
        oracle.set_num_threads(cores)
        line["cpu_baseline"]["one_core"] = {"value": round(g1, 4), "unit": "GB/s", "sample": s1}
    if extra:
        line["detail"] = extra
    if rank == 0:
        print(json.dumps(line), flush=True)
    for h in hs:
        h.close()
    return 0


def repack_times():
    """Load-time repack (checkpoint -> runtime layout) per layer, timed apart from the GEMM: host wall
    clock around each repack call (it ends with a stream synchronize), median of three."""
    import torch
    from weight_only_quantized_gb300 import gptq, synth
    out = {}
    for name in ("llama3-8b-decode-4096x14336-b4g128-sym", "llama3-70b-gate-8192x28672-b4g128-descact"):
        spec, _ = synth.workload(name)
        ck = synth.make_checkpoint(spec, seed=3)
        d = [t.cuda() if t is not None else None for t in (ck.qweight, ck.qzeros, ck.scales, ck.g_idx)]
        ts = []
        for _ in range(4):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            h = gptq.gptq_repack(d[0], d[1], d[2], d[3], spec.bits, spec.group_size)
            torch.cuda.synchronize()
            ts.append(time.perf_counter() - t0)
            h.close()
        ts = sorted(ts[1:])
        out[name] = {"ms": round(ts[1] * 1e3, 3), "weight_MB": round(spec.K * spec.N * spec.bits / 8 / 1e6, 1)}
        del d
    return out


def extra_workloads(args, hbm, tf_burst, peak_kind, tf_sus):
    """Rank 0: the decode layer (M = 1 as a headline key, then 8 and 16), the gate layer's other M,
    the prefill layer (M = 4096 as a headline key, then 512 and 2048), AWQ and FP8 layers, the
    K = N = 4096 format sweep, and the load-time repack."""
    import torch
    from weight_only_quantized_gb300 import gptq, synth
    out = {}
    steps = max(20, min(args.steps, 200))

    def one(spec, Ms, layers):
        hs, _ = make_layers(spec, layers, seed0=1000)
        for h in hs:
            gptq.gptq_reserve(h, max(Ms))
        dt = torch.float16 if spec.dtype == "fp16" else torch.bfloat16
        res = {}
        for M in Ms:
            xs = [synth.make_x(M, spec.K, spec.dtype, seed=M + i).cuda() for i in range(min(layers, 4))]
            ys = [torch.empty(M, spec.N, dtype=dt, device="cuda") for _ in range(min(layers, 4))]
            n = steps if M <= 64 else max(5, steps // 10)
            res[f"M={M}"] = layer_line(spec, M, time_calls(hs, xs, ys, M, n, 3, graph=True), hbm, tf_burst, tf_sus)
            del xs, ys
        for h in hs:
            h.close()
        torch.cuda.empty_cache()
        return res

    s2, _ = synth.workload(DECODE)
    r2 = one(s2, [1, 8, 16], 16)
    out["decode_m1"] = dict(r2.pop("M=1"), workload=DECODE)
    out[DECODE] = r2
    s3, m3 = synth.workload(WORKLOAD)
    out[WORKLOAD] = one(s3, [m for m in m3 if m != 1], 8)
    s4, m4 = synth.workload(PREFILL)
    r4 = one(s4, [4096] if args.quick_prefill else [4096] + [m for m in m4 if m != 4096], 1)
    out["prefill_m4096"] = dict(r4.pop("M=4096"), workload=PREFILL)
    tr = traffic_record("gemm_large.cu", PREFILL)
    # DRAM bytes of one launch from the committed ncu capture (while the kernel code is unchanged)
    out["prefill_m4096"]["traffic"] = tr["dram_bytes_per_launch"] if tr else None
    out[PREFILL] = r4
    out["awq-4096x14336-b4g128-fp16"] = awq_layer(hbm, tf_burst)
    out["fp8-4096x14336-block128-bf16"] = fp8_layer(hbm, tf_burst)
    if not args.no_sweep:
        out["format-sweep-4096x4096"] = format_sweep(hbm, tf_burst)
    out["repack"] = repack_times()
    out["peaks"] = {"hbm_gbs": hbm, "bf16_tflops": tf_burst, "bf16_tflops_sustained": tf_sus, "kind": peak_kind}
    return out


def awq_layer(hbm, tf_burst):
    """An AutoAWQ GEMM checkpoint of the decode layer's shape (K = 4096, N = 14336, 4-bit, group
    128, fp16, asymmetric zeros) through gptq_repack_awq, at M = 1, 16 and 512; 16 handles
    rotated so every call streams its weights from HBM."""
    import torch
    from weight_only_quantized_gb300 import gptq, synth
    K, N, gs = 4096, 14336, 128
    spec = synth.LayerSpec(K, N, 4, gs, False, False, "fp16")     # for the byte count only
    ck = synth.make_awq_checkpoint(K, N, gs, "fp16", seed=5)
    dev = [ck.qweight.cuda(), ck.qzeros.cuda(), ck.scales.cuda()]
    hs = [gptq.gptq_repack_awq(dev[0], dev[1], dev[2], gs) for _ in range(LAYERS)]
    torch.cuda.synchronize()
    r = {"layers_rotated": LAYERS}
    for M in (1, 16, 512):
        xs = [synth.make_x(M, K, "fp16", seed=M + i).cuda() for i in range(4)]
        ys = [torch.empty(M, N, dtype=torch.float16, device="cuda") for _ in range(4)]
        t = time_calls(hs, xs, ys, M, 200 if M <= 64 else 50, 3, graph=True)
        B, F = b_alg(spec, M), 2.0 * M * N * K
        roof = max(B / (hbm * 1e9), F / (tf_burst * 1e12))
        r[f"M={M}"] = {"us": round(t * 1e6, 2), "GB/s": round(B / t / 1e9, 1), "TFLOP/s": round(F / t / 1e12, 2),
                       "roofline_frac": round(roof / t, 4),
                       "bound": "hbm" if B / (hbm * 1e9) >= F / (tf_burst * 1e12) else "tensor"}
        del xs, ys
    for h in hs:
        h.close()
    del hs, dev
    torch.cuda.empty_cache()
    return r


def fp8_layer(hbm, tf_burst):
    """An FP8 block-scaled layer of the decode layer's shape (K = 4096, N = 14336, e4m3 weights, one
    float32 factor per 128 x 128 block, bf16 x and y) through gptq_repack_fp8 at M = 1, 16 and 512;
    16 handles rotated (940 MB of weights) so every call streams from HBM.  Bytes per call: the
    weight bytes, the factors, x and y."""
    import torch
    from weight_only_quantized_gb300 import gptq, synth
    K, N = 4096, 14336
    ck = synth.make_fp8_checkpoint(K, N, "bf16", seed=6)
    w, s = ck.weight.cuda(), ck.scale_inv.cuda()
    hs = [gptq.gptq_repack_fp8(w, s, torch.bfloat16) for _ in range(LAYERS)]
    del w, s
    torch.cuda.synchronize()
    r = {"layers_rotated": LAYERS}
    for M in (1, 16, 512):
        xs = [synth.make_x(M, K, "bf16", seed=M + i).cuda() for i in range(4)]
        ys = [torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
        t = time_calls(hs, xs, ys, M, 200 if M <= 64 else 50, 3, graph=True)
        B = N * K + 4 * (-(-N // 128)) * (-(-K // 128)) + 2 * M * K + 2 * M * N
        F = 2.0 * M * N * K
        roof = max(B / (hbm * 1e9), F / (tf_burst * 1e12))
        r[f"M={M}"] = {"us": round(t * 1e6, 2), "GB/s": round(B / t / 1e9, 1), "TFLOP/s": round(F / t / 1e12, 2),
                       "roofline_frac": round(roof / t, 4),
                       "bound": "hbm" if B / (hbm * 1e9) >= F / (tf_burst * 1e12) else "tensor"}
        del xs, ys
    for h in hs:
        h.close()
    del hs
    torch.cuda.empty_cache()
    return r


def format_sweep(hbm, tf_burst):
    """K = N = 4096 at bits 2/3/8 (group 128) and bits 4 at groups -1/32/64, M = 1/32/256.

    One seeded checkpoint per format, repacked into as many handles as it takes for the rotated
    weights to cover three L2 sizes, so every call streams its weights from HBM."""
    import torch
    from weight_only_quantized_gb300 import gptq, synth
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    res = {}
    for spec in synth.format_sweep():
        name = f"b{spec.bits}g{spec.group_size}{'-descact' if spec.desc_act else ''}"
        B1 = b_alg(spec, 1)
        nl = max(4, min(128, -(-3 * l2 // B1)))
        ck = synth.make_checkpoint(spec, seed=7)
        dev = [t.cuda() if t is not None else None for t in (ck.qweight, ck.qzeros, ck.scales, ck.g_idx)]
        hs = [gptq.gptq_repack(dev[0], dev[1], dev[2], dev[3], spec.bits, spec.group_size) for _ in range(nl)]
        for h in hs:
            gptq.gptq_reserve(h, max(synth.SWEEP_M))
        torch.cuda.synchronize()
        r = {"layers_rotated": nl}
        for M in synth.SWEEP_M:
            xs = [synth.make_x(M, spec.K, spec.dtype, seed=M + i).cuda() for i in range(4)]
            ys = [torch.empty(M, spec.N, dtype=torch.float16, device="cuda") for _ in range(4)]
            n = 200 if M <= 64 else 50
            t = time_calls(hs, xs, ys, M, n, 3, graph=True)
            B, F = b_alg(spec, M), 2.0 * M * spec.N * spec.K
            roof = max(B / (hbm * 1e9), F / (tf_burst * 1e12))
            r[f"M={M}"] = {"us": round(t * 1e6, 2), "GB/s": round(B / t / 1e9, 1), "TFLOP/s": round(F / t / 1e12, 2),
                           "roofline_frac": round(roof / t, 4),
                           "bound": "hbm" if B / (hbm * 1e9) >= F / (tf_burst * 1e12) else "tensor"}
            del xs, ys
        for h in hs:
            h.close()
        del hs, dev
        torch.cuda.empty_cache()
        res[name] = r
    return res


PROFILE_LAYERS = {"decode": DECODE, "gate": WORKLOAD, "prefill": PREFILL}


def run_profile(args):
    """One layer, one weight set, `steps` eager calls at M = --profile-m: a small, fixed launch
    sequence for ncu captures (repack kernels first, then warm-up and timed gptq_gemm launches)."""
    import torch
    from weight_only_quantized_gb300 import gptq, synth
    spec, _ = synth.workload(PROFILE_LAYERS[args.profile_layer])
    M = args.profile_m
    hs, _ = make_layers(spec, 1)
    gptq.gptq_reserve(hs[0], M)
    dt = torch.float16 if spec.dtype == "fp16" else torch.bfloat16
    xs = [synth.make_x(M, spec.K, spec.dtype, seed=3).cuda()]
    ys = [torch.empty(M, spec.N, dtype=dt, device="cuda")]
    t = time_calls(hs, xs, ys, M, args.steps, args.warmup, graph=False, min_total_s=0.0, min_reps=1)
    B, F = b_alg(spec, M), 2.0 * M * spec.N * spec.K
    print(json.dumps({"profile_layer": args.profile_layer, "M": M, "us_per_call": round(t * 1e6, 2),
                      "GB/s": round(B / t / 1e9, 1), "TFLOP/s": round(F / t / 1e12, 2),
                      "launches_per_call": gptq.gptq_gemm_launches(hs[0], M)}), flush=True)
    hs[0].close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-extra", action="store_true", help="skip the other layers and M values")
    ap.add_argument("--no-sweep", action="store_true", help="skip the K = N = 4096 format sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--quick-prefill", action="store_true", help="prefill at M=4096 only")
    ap.add_argument("--profile-layer", choices=["decode", "gate", "prefill"], default=None,
                    help="profiling mode: time only this layer at --profile-m (one weight set) and print one line")
    ap.add_argument("--profile-m", type=int, default=1)
    args = ap.parse_args()
    args._remeasured = False
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        return run_reference(args, ws, rank)
    ws, rank, local = dist_setup()
    if args.profile_layer:
        return run_profile(args)
    try:
        return run_native(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
