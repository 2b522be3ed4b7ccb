"""Benchmark of the 4-bit decode GEMVs on GB300.

One step is one call of every GEMV entry point on its workload:
  q4_gemv 256x1024, fused_rmsnorm_q4k_gemv 3584x3584, fused_gateup_q4k_gemv 2x18944x3584,
  q4_gemv_batched 14336x4096 at M = 1, 2, 4 and 8, and moe_q4_gemv (64 experts x 1408x2048, 8 tokens x top-8).
The metric is effective weight bandwidth: the weight bytes each call must read (for MoE, the distinct selected
experts' bytes) divided by device time. Steps replay CUDA graphs over two replica sets of all weights, so each
call reads weights that were last touched about 650 MB of traffic earlier (the L2 holds 129 MB). Per-call times
(`per_call`) come from graphs of one call type back to back over weight copies of at least 3x the L2, with the
spread of five batches, a launch-inclusive single-call time and the pure-read instrument of the same bytes.

Prints one JSON line (rank 0). ``--impl reference`` times the plain-C fp64 oracle instead (host cores).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

L2_BYTES = 129 * 2**20
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
# The one metric both arms report: `value` is the suite's weight bytes over its time (the reference arm's time is
# its host time for the same bytes); `per_call` holds each call's GB/s, fraction of the HBM peak and us.
METRIC = "effective weight GB/s per GEMV call and % of GB300 HBM peak; \u00b5s/call"

KERNEL_SOURCES = ["device_common.cuh", "launch.h", "q4_dense.cuh", "kernels_q4.cu", "kernels_q4_v2_4.cu",
                  "kernels_q4_v5_8.cu", "kernels_q4_v9_16.cu", "kernels_q4k.cu", "kernels_q4k_rows.cu",
                  "kernels_q4k_batched.cu", "kernels_moe.cu", "kernels_router.cu", "q4_xr.cuh"]


# ------------------------------------------------------------------------------------------------
# workload definition (shared by both arms)
# ------------------------------------------------------------------------------------------------

def q4_bytes(N, K):
    return N * K // 2 + N * (K // 32) * 2


def q4k_bytes(N, K):
    return N * (K // 256) * 144


def make_inputs(seed=0):
    c1 = synth.make_q4_gemv(seed, 256, 1024)
    c2 = synth.make_fused_rmsnorm(seed + 1, 3584, 3584)
    c3 = synth.make_gateup(seed + 2, 18944, 3584)
    c4 = synth.make_q4_gemv(seed + 3, 14336, 4096, M=8)
    c5 = synth.make_moe(seed + 4, 64, 1408, 2048, 8, 8)
    return c1, c2, c3, c4, c5


def call_table(c5_ids):
    """(name, weight bytes, key) of each call of a step, in launch order."""
    uniq = len(np.unique(c5_ids))
    return [
        ("q4_gemv 256x1024", q4_bytes(256, 1024), "q4_gemv_256x1024"),
        ("fused_rmsnorm_q4k_gemv 3584x3584", q4k_bytes(3584, 3584), "rmsnorm_q4k_3584x3584"),
        ("fused_gateup_q4k_gemv 2x18944x3584", 2 * q4k_bytes(18944, 3584), "gateup_q4k_2x18944x3584"),
        ("q4_gemv_batched 14336x4096 M=1", q4_bytes(14336, 4096), "q4_batched_14336x4096_m1"),
        ("q4_gemv_batched 14336x4096 M=2", q4_bytes(14336, 4096), "q4_batched_14336x4096_m2"),
        ("q4_gemv_batched 14336x4096 M=4", q4_bytes(14336, 4096), "q4_batched_14336x4096_m4"),
        ("q4_gemv_batched 14336x4096 M=8", q4_bytes(14336, 4096), "q4_batched_14336x4096_m8"),
        (f"moe_q4_gemv e64 1408x2048 t8k8 ({uniq} experts)", 2 * uniq * q4_bytes(1408, 2048), "moe_q4_e64_t8k8"),
    ]


def call_fmas(c5_ids):
    """fp32 FMAs of each call of a step (M per weight and vector; MoE: every token's slot, gate and up)."""
    T, topk = np.asarray(c5_ids).shape
    return [256 * 1024, 3584 * 3584, 2 * 18944 * 3584] + [M * 14336 * 4096 for M in (1, 2, 4, 8)] + \
        [T * topk * 2 * 1408 * 2048]


WORKLOAD_NAME = ("decode GEMV suite: Q4 256x1024; RMSNorm+Q4_K 3584x3584; gate+up Q4_K 2x18944x3584; "
                 "Q4 14336x4096 at M=1,2,4,8; MoE Q4 64x(1408x2048) gate+up, 8 tokens top-8")


def measured_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "quantized_decode_gemv_q4_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, or None when absent or stale."""
    try:
        with open(TRAFFIC_FILE) as f:
            lines = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    except OSError:
        return None
    cur = kernel_source_hash()
    for parts in lines:
        if len(parts) >= 3 and parts[0] == kernel_key and parts[2] == cur:
            return float(parts[1])
    return None


# ------------------------------------------------------------------------------------------------
# clocks
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        try:
            sm = [float(r[1]) for r in rows]
            smax = max(float(r[2]) for r in rows)
            power = [float(r[3]) for r in rows]
        except ValueError:
            return None
        # samples under load: power well above the idle floor
        floor = min(power)
        load = [s for s, p in zip(sm, power) if p > floor + 0.25 * (max(power) - floor)] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": smax, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------------------------
# multi-rank plumbing
# ------------------------------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def aggregate(per_rank_seconds: float, bytes_per_step: float, steps: int, world: int):
    """Whole-job throughput: every rank runs the same step (independent replicas), timing is the slowest rank."""
    t = max_over_ranks(per_rank_seconds, world)
    return world * bytes_per_step * steps / t / 1e9, t


# ------------------------------------------------------------------------------------------------
# CPU oracle leg
# ------------------------------------------------------------------------------------------------

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def row_chunks(n: int, parts: int):
    """[lo, hi) ranges that split n rows into at most `parts` nearly equal chunks."""
    step = -(-n // max(1, parts))
    return [(lo, min(n, lo + step)) for lo in range(0, n, step)]


def oracle_step(o, inputs, frac=1.0, pool=None, parts=1):
    """The step's work on the host oracle, on the first `frac` of each matrix's rows. Returns weight bytes.

    With a thread pool, every call's rows are split into `parts` chunks that the pool runs at once (the oracle's
    C functions release the interpreter lock, and a row's result depends only on that row and the inputs)."""
    c1, c2, c3, c4, c5 = inputs
    done = 0

    def rows(n):
        return max(1, int(round(n * frac)))

    def run(fn, n):
        if pool is None:
            return [fn(0, n)]
        return list(pool.map(lambda r: fn(*r), row_chunks(n, parts)))

    n = rows(256)
    run(lambda lo, hi: o.q4_gemv(c1["qs"][lo:hi], c1["d"][lo:hi], c1["x"][0]), n)
    done += q4_bytes(n, 1024)
    n = rows(3584)
    run(lambda lo, hi: o.fused_rmsnorm_q4k_gemv(c2["w"][lo:hi], c2["x"], c2["gamma"], c2["eps"]), n)
    done += q4k_bytes(n, 3584)
    n = rows(18944)
    run(lambda lo, hi: o.fused_gateup_q4k_gemv(c3["w_gate"][lo:hi], c3["w_up"][lo:hi], c3["x"], c3["gamma"],
                                               c3["eps"]), n)
    done += 2 * q4k_bytes(n, 3584)
    n = rows(14336)
    for M in (1, 2, 4, 8):
        run(lambda lo, hi, M=M: o.q4_gemv_batched(c4["qs"][lo:hi], c4["d"][lo:hi], c4["x"][:M]), n)
        done += q4_bytes(n, 4096)
    n = rows(1408)

    def per_expert(a, lo, hi):
        return np.ascontiguousarray(a.reshape(64, 1408, *a.shape[1:])[:, lo:hi].reshape(64 * (hi - lo), *a.shape[1:]))

    run(lambda lo, hi: o.moe_q4_gemv(per_expert(c5["qs_gate"], lo, hi), per_expert(c5["d_gate"], lo, hi),
                                     per_expert(c5["qs_up"], lo, hi), per_expert(c5["d_up"], lo, hi), c5["x"],
                                     c5["ids"], 64), n)
    done += 2 * len(np.unique(c5["ids"])) * q4_bytes(n, 2048)
    return done


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle

    from concurrent.futures import ThreadPoolExecutor

    o = oracle.default()
    inputs = make_inputs()
    cores = host_cores()
    with ThreadPoolExecutor(cores) as pool:
        t0 = time.perf_counter()
        oracle_step(o, inputs, 1.0 / 64, pool, cores)
        t_full = (time.perf_counter() - t0) * 64
        frac = min(1.0 / 4, max(1.0 / 4096, 90.0 / ((args.steps + args.warmup) * t_full)))
        for _ in range(args.warmup):
            oracle_step(o, inputs, frac, pool, cores)
        t0 = time.perf_counter()
        done = 0
        for _ in range(args.steps):
            done += oracle_step(o, inputs, frac, pool, cores)
        dt = time.perf_counter() - t0
    value = done / dt / 1e9
    sample = (f"each step: the suite on the first {frac:.5f} of every matrix's rows (MoE: of every expert's rows), "
              f"each call's rows split over {cores} threads; the fraction is sized so that warm-up plus timed steps "
              f"take about 90 s, at most a quarter of the rows ({(args.steps + args.warmup) * dt / args.steps:.1f} s "
              "here)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)", "config": {"workload": WORKLOAD_NAME, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------------
# GPU leg
# ------------------------------------------------------------------------------------------------

class Suite:
    """Device copies of the suite's weights (several replica sets) and its per-step inputs/outputs."""

    def __init__(self, inputs, replicas: int, dev):
        import torch

        cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
        c1, c2, c3, c4, c5 = inputs
        self.inputs = inputs
        self.sets = []
        for _ in range(replicas):
            self.sets.append(dict(
                c1=(cu(c1["qs"]), cu(c1["d"])), c2=cu(c2["w"]), c3=(cu(c3["w_gate"]), cu(c3["w_up"])),
                c4=[(cu(c4["qs"]), cu(c4["d"])) for _ in range(4)],  # one copy per batch width: each call cold
                c5=(cu(c5["qs_gate"]), cu(c5["d_gate"]), cu(c5["qs_up"]), cu(c5["d_up"]))))
        # Per-step activations and outputs, each set packed into one device buffer (256-byte aligned views) so
        # that a step's inputs arrive by one copy and its outputs leave by one copy.
        self.in_buf, (self.x1, self.x2, self.g2, self.x3, self.g3, self.X4, self.x5, self.ids5) = packed(
            [c1["x"][0], c2["x"], c2["gamma"], c3["x"], c3["gamma"], c4["x"], c5["x"], c5["ids"]], dev)
        f32 = np.float32
        self.out_buf, outs = packed([np.zeros(256, f32), np.zeros(3584, f32), np.zeros(18944, f32),
                                     np.zeros(18944, f32)] + [np.zeros((M, 14336), f32) for M in (1, 2, 4, 8)] +
                                    [np.zeros((8, 8, 1408), f32), np.zeros((8, 8, 1408), f32)], dev)
        self.y1, self.y2, self.y3g, self.y3u = outs[:4]
        self.Y4 = outs[4:8]
        self.y5g, self.y5u = outs[8:]

    def calls(self, s, stream=None):
        """The step's calls on replica set s, as closures in launch order (on `stream`, else the current one)."""
        import quantized_decode_gemv_q4_gb300 as q4

        w = self.sets[s]
        c2eps = float(self.inputs[1]["eps"])
        c3eps = float(self.inputs[2]["eps"])
        st = stream
        out = [
            lambda: q4.q4_gemv(self.y1, w["c1"][0], w["c1"][1], self.x1, stream=st),
            lambda: q4.fused_rmsnorm_q4k_gemv(self.y2, w["c2"], self.x2, self.g2, c2eps, stream=st),
            lambda: q4.fused_gateup_q4k_gemv(self.y3g, self.y3u, w["c3"][0], w["c3"][1], self.x3, self.g3, c3eps,
                                             stream=st),
        ]
        for i, M in enumerate((1, 2, 4, 8)):
            out.append(lambda i=i, M=M: q4.q4_gemv_batched(self.Y4[i], w["c4"][i][0], w["c4"][i][1], self.X4[:M],
                                                           stream=st))
        out.append(lambda: q4.moe_q4_gemv(self.y5g, self.y5u, *w["c5"], self.x5, self.ids5, 64, stream=st))
        return out


def packed(arrays, dev):
    """One device byte buffer holding the given host arrays at 256-byte aligned offsets, and typed views of it
    (in order) that start out holding the arrays' values."""
    import torch

    offs, n = [], 0
    for a in arrays:
        offs.append(n)
        n += (a.nbytes + 255) // 256 * 256
    host = np.zeros(n, np.uint8)
    for a, o in zip(arrays, offs):
        host[o:o + a.nbytes] = np.ascontiguousarray(a).view(np.uint8).ravel()
    buf = torch.from_numpy(host).to(dev)
    tdt = {np.dtype(np.float32): torch.float32, np.dtype(np.int32): torch.int32}
    views = [buf[o:o + a.nbytes].view(tdt[a.dtype]).view(a.shape) for a, o in zip(arrays, offs)]
    return buf, views


def capture(fns, stream):
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for fn in fns:
            fn()
    return g


def run_gpu(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import quantized_decode_gemv_q4_gb300 as q4

    q4.load()
    # Launch overlap: each call's first weight copies overlap the previous call's tail (the weights are never
    # written inside the step; every kernel waits for its predecessor before touching inputs or outputs).
    q4.q4_set_launch_overlap(True)
    inputs = make_inputs()
    table = call_table(inputs[4]["ids"])
    step_bytes = sum(t[1] for t in table)
    replicas = 2
    suite = Suite(inputs, replicas, dev)
    stream = torch.cuda.Stream(device=dev)

    # warm every call once eagerly (plans, attributes), then capture one graph per replica set
    with torch.cuda.stream(stream):
        for s in range(replicas):
            for fn in suite.calls(s):
                fn()
    torch.cuda.synchronize()
    graphs = [capture(suite.calls(s), stream) for s in range(replicas)]
    n_calls = len(table)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % replicas].replay()
    torch.cuda.synchronize()

    # ---- headline: K steps, device-timed ----------------------------------------------------------
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            start.record()
            for i in range(args.steps):
                graphs[i % replicas].replay()
            end.record()
        torch.cuda.synchronize()
    barrier(world)
    secs = start.elapsed_time(end) / 1e3
    value, tmax = aggregate(secs, step_bytes, args.steps, world)
    clocks = clk.summary()

    # context: the same steps with launch overlap off (graphs captured again)
    q4.q4_set_launch_overlap(False)
    plain = [capture(suite.calls(s), stream) for s in range(replicas)]
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup // 4)):
            plain[i % replicas].replay()
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record()
        for i in range(args.steps):
            plain[i % replicas].replay()
        end.record()
    torch.cuda.synchronize()
    barrier(world)
    value_plain, _ = aggregate(start.elapsed_time(end) / 1e3, step_bytes, args.steps, world)
    del plain
    q4.q4_set_launch_overlap(True)

    # ---- per-call device time: each call type alone, back to back over weight copies of >= 3x the L2 ------
    peak, peak_kind = measured_peaks()
    fma = measure_fma_ceiling(stream, call_fmas(inputs[4]["ids"])[6])
    per_call = measure_per_call(suite, inputs, table, stream, peak, fma["fmas_per_us"])
    kt_us = np.array([pc["us"] for pc in per_call])
    dom = int(np.argmax(kt_us))
    traffic = committed_traffic(table[dom][2])
    achieved = table[dom][1] / kt_us[dom] / 1e3
    roofline = {"bound": "hbm", "kernel": table[dom][0], "achieved": round(achieved, 1), "peak": peak,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
                "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "algorithmic_bytes": table[dom][1], "us_per_launch": round(float(kt_us[dom]), 3)}

    # ---- the NEXT rows (router, SwiGLU forms, wider batches, launch chain), timed the same way ------
    next_rows = measure_next_rows(suite, inputs, stream, replicas, peak, fma["fmas_per_us"])
    fma["fmas_per_us"] = round(fma["fmas_per_us"], 1)
    next_rows["fma_ceiling"] = fma

    # ---- end to end through the Python API with host buffers ---------------------------------------
    e2e = run_e2e(suite, inputs, stream, max(20, min(args.steps // 20, 400)), table)

    # ---- CPU baseline (oracle, host cores) -----------------------------------------------------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inputs)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tmax / args.steps * 1e3, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 (4-bit weights, fp32 inputs and accumulation)",
            "data": "synthetic (seeded generators; no trained weights)",
            "config": {"workload": WORKLOAD_NAME, "weight_bytes_per_step": step_bytes,
                       "l2": "inputs larger than L2: the step rotates 2 replica sets of all weights (846 MB), each "
                             "call reads weights last touched ~650 MB of traffic earlier; per_call and next_rows "
                             "rotate each call over weight copies of >= 3x the L2 (rotation_bytes)",
                       "graph": "one CUDA graph per step",
                       "launch_overlap": "on (programmatic dependent launch: each call's first weight copies "
                                         "overlap the previous call's tail)",
                       "value_without_launch_overlap": round(value_plain, 1),
                       "parallelism": f"replicas x{world}"},
            "per_call": per_call, "next_rows": next_rows, "roofline": roofline, "gpu_launches": args.steps * n_calls,
            "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def cold_copies(tensors, nbytes):
    """Device copies of a weight set, enough that their bytes (`nbytes` read per call) reach 3x the L2: calls
    rotated over them read weights no earlier call left in the L2. Each copy is a slice of one allocation per
    tensor (contiguous, 256-byte aligned when the tensor's size is)."""
    import torch

    k = max(2, int(np.ceil(3 * L2_BYTES / nbytes)))
    stacks = []
    for t in tensors:
        s = torch.empty((k,) + tuple(t.shape), dtype=t.dtype, device=t.device)
        s.copy_(t.unsqueeze(0).expand_as(s))
        stacks.append(s)
    return [tuple(s[i] for s in stacks) for i in range(k)], k


def _graph_us(fns, stream, reps=None, tries=5):
    """Per-launch device time of a CUDA graph of `reps` calls (fns rotated; default: each once, at least 16):
    one replay discarded, then the best of `tries` timed replays and the spread (worst / best)."""
    import torch

    reps = reps or max(16, len(fns))
    g = capture([fns[i % len(fns)] for i in range(reps)], stream)
    with torch.cuda.stream(stream):
        g.replay()
    times = []
    for _ in range(tries):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record()
            g.replay()
            b.record()
        b.synchronize()
        times.append(a.elapsed_time(b) / reps * 1e3)
    del g
    return min(times), max(times) / min(times)


def _single_us(fn, stream, n=21):
    """Launch-inclusive time of one call (events around one eager call, idle device before it): median of n."""
    import torch

    ts = []
    for _ in range(n):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record()
            fn()
            b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    return float(np.median(ts))


def _entry(name, nbytes, us, spread, k, peak, fmas=None, fma_rate=None, **extra):
    """One timed call. With its FMA count and the measured FMA rate (FMAs per us, from the FMA-ceiling
    instrument), the two floors beside it: the weight bytes at the HBM peak and the FMAs at the FMA ceiling,
    and which of them is the binding roof."""
    e = {"call": name, "us": round(us, 3), "weight_GBps": round(nbytes / us / 1e3, 1),
         "frac_of_hbm_peak": round(nbytes / us / 1e3 / peak, 4), "spread": round(spread, 3),
         "rotation_bytes": int(k * nbytes), "copies": k}
    if fmas is not None and fma_rate:
        hbm_floor, fma_floor = nbytes / peak / 1e3, fmas / fma_rate
        e.update({"hbm_floor_us": round(hbm_floor, 3), "fma_floor_us": round(fma_floor, 3),
                  "bound": "hbm" if hbm_floor >= fma_floor else "fma",
                  "frac_of_binding_roof": round(max(hbm_floor, fma_floor) / us, 4)})
    e.update(extra)
    return e


def measure_fma_ceiling(stream, fmas):
    """The FMA-ceiling instrument at `fmas` FMAs (one launch per call, back to back in a graph): its us, the FMAs
    it ran and the FMA rate in FMAs per us."""
    import torch

    import quantized_decode_gemv_q4_gb300 as q4

    sink = torch.empty(1024, device=torch.device("cuda", torch.cuda.current_device()))
    done = q4.q4_fma_ceiling(sink, fmas, stream=stream)
    us, sp = _graph_us([lambda: q4.q4_fma_ceiling(sink, fmas, stream=stream)], stream)
    return {"us": round(us, 3), "spread": round(sp, 3), "fmas": done, "fmas_per_us": done / us,
            "fp32_TFLOPs": round(2 * done / us / 1e6, 2),
            "what": "fp32x2 FMA chains on one 512-thread CTA per SM, no loads; the M=8 call's FMA count"}


def measure_per_call(suite, inputs, table, stream, peak, fma_rate=None):
    """Each suite call alone, back to back in one CUDA graph over weight copies whose bytes reach 3x the L2, so
    every call streams its weights from HBM; the pure-read instrument of the same bytes beside it."""
    import torch

    import quantized_decode_gemv_q4_gb300 as q4

    w = suite.sets[0]
    c2eps = float(inputs[1]["eps"])
    c3eps = float(inputs[2]["eps"])
    fmas = call_fmas(inputs[4]["ids"])
    out = []

    def one(j, fns, k, pure=None, pure_per_call=1):
        us, spread = _graph_us(fns, stream)
        single = _single_us(fns[0], stream)
        extra = {"single_call_us": round(single, 3)}
        if pure is not None:
            pus, pspread = _graph_us(pure, stream)
            pus *= pure_per_call  # instrument launches that read the call's bytes
            extra["pure_read_us"] = round(pus, 3)
            extra["pure_read_frac_of_hbm_peak"] = round(table[j][1] / pus / 1e3 / peak, 4)
            extra["kernel_over_pure_read"] = round(us / pus, 3)
        out.append(_entry(table[j][0], table[j][1], us, spread, k, peak, fmas=fmas[j], fma_rate=fma_rate, **extra))

    cp, k = cold_copies(w["c1"], table[0][1])
    one(0, [lambda c=c: q4.q4_gemv(suite.y1, c[0], c[1], suite.x1, stream=stream) for c in cp], k,
        pure=[lambda c=c: q4.q4_pure_read(suite.y1, c[0], c[1], stream=stream) for c in cp])
    del cp
    cp, k = cold_copies((w["c2"],), table[1][1])
    one(1, [lambda c=c: q4.fused_rmsnorm_q4k_gemv(suite.y2, c[0], suite.x2, suite.g2, c2eps, stream=stream)
            for c in cp], k,
        pure=[lambda c=c: q4.q4k_pure_read(suite.y2, c[0], stream=stream) for c in cp])
    del cp
    cp, k = cold_copies(w["c3"], table[2][1])
    one(2, [lambda c=c: q4.fused_gateup_q4k_gemv(suite.y3g, suite.y3u, c[0], c[1], suite.x3, suite.g3, c3eps,
                                                 stream=stream) for c in cp], k,
        pure=[lambda m=m: q4.q4k_pure_read(suite.y3g, m, stream=stream) for c in cp for m in c], pure_per_call=2)
    del cp
    cp, k = cold_copies(w["c4"][0], table[3][1])
    for i, M in enumerate((1, 2, 4, 8)):
        one(3 + i, [lambda c=c, i=i, M=M: q4.q4_gemv_batched(suite.Y4[i], c[0], c[1], suite.X4[:M], stream=stream)
                    for c in cp], k,
            pure=[lambda c=c: q4.q4_pure_read(suite.Y4[3][0], c[0], c[1], stream=stream) for c in cp] if M == 1 else None)
    del cp
    cp, k = cold_copies(w["c5"], table[7][1])
    one(7, [lambda c=c: q4.moe_q4_gemv(suite.y5g, suite.y5u, *c, suite.x5, suite.ids5, 64, stream=stream)
            for c in cp], k,
        pure=[lambda c=c: q4.moe_q4_pure_read(suite.y5g, suite.y5u, *c, suite.ids5, 64, stream=stream) for c in cp])
    del cp
    torch.cuda.empty_cache()
    return out


def measure_next_rows(suite, inputs, stream, replicas, peak, fma_rate=None):
    """The router, the SwiGLU forms, the wider batches and a dependent router -> MoE-SwiGLU chain, each over
    weight copies of >= 3x the L2 like the suite's calls."""
    import torch

    import quantized_decode_gemv_q4_gb300 as q4

    dev = suite.x1.device
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    rng = np.random.default_rng(7)
    E, K, T, topk = 64, 2048, 8, 8
    rq, rd = synth.q4_weights(rng, E, K)
    rq, rd = cu(rq), cu(rd)
    ids = torch.empty(T, topk, dtype=torch.int32, device=dev)
    wts = torch.empty(T, topk, device=dev)
    ysw = torch.empty(18944, device=dev)
    ymo = torch.empty(T, topk, 1408, device=dev)
    c3eps = float(inputs[2]["eps"])
    out = {}
    rb = q4_bytes(E, K)
    cp, k = cold_copies((rq, rd), rb)
    us, sp = _graph_us([lambda c=c: q4.moe_router_q4(ids, wts, c[0], c[1], suite.x5, topk, True, stream=stream)
                        for c in cp], stream)
    out["moe_router_q4 e64 k2048 t8 top8"] = {"us": round(us, 3), "spread": round(sp, 3), "copies": k,
                                              "note": "74 KB of router weights: launch-latency bound"}
    del cp
    gb = 2 * q4k_bytes(18944, 3584)
    cp, k = cold_copies(suite.sets[0]["c3"], gb)
    us, sp = _graph_us([lambda c=c: q4.fused_gateup_swiglu_q4k_gemv(ysw, c[0], c[1], suite.x3, suite.g3, c3eps,
                                                                    stream=stream) for c in cp], stream)
    out["fused_gateup_swiglu_q4k_gemv 2x18944x3584"] = _entry("", gb, us, sp, k, peak)
    # unfused batched Q4_K on the gate and up matrices of the same copies (12 matrices of 38 MB rotated)
    kb = q4k_bytes(18944, 3584)
    Xk = torch.from_numpy(np.ascontiguousarray(synth.activations(rng, 8, 3584))).to(dev)
    mats = [m for c in cp for m in c]
    for M in (1, 8):
        Yk = torch.empty(M, 18944, device=dev)
        us, sp = _graph_us([lambda m=m: q4.q4k_gemv_batched(Yk, m, Xk[:M], stream=stream) for m in mats], stream)
        out[f"q4k_gemv_batched 18944x3584 M={M}"] = _entry("", kb, us, sp, len(mats) // 2, peak,
                                                           fmas=M * 18944 * 3584, fma_rate=fma_rate)
    del cp, mats
    uniq = len(np.unique(inputs[4]["ids"]))
    mb = 2 * uniq * q4_bytes(1408, 2048)
    cp, k = cold_copies(suite.sets[0]["c5"], mb)
    us, sp = _graph_us([lambda c=c: q4.moe_q4_swiglu_gemv(ymo, *c, suite.x5, suite.ids5, 64, stream=stream)
                        for c in cp], stream)
    out[f"moe_q4_swiglu_gemv e64 1408x2048 t8k8 ({uniq} experts)"] = _entry("", mb, us, sp, k, peak)
    # dependent chain: the router's ids drive the MoE call on the device
    chain = []
    for ov in (True, False):
        q4.q4_set_launch_overlap(ov)
        fns = []
        for c in cp:
            fns.append(lambda: q4.moe_router_q4(ids, wts, rq, rd, suite.x5, topk, True, stream=stream))
            fns.append(lambda c=c: q4.moe_q4_swiglu_gemv(ymo, *c, suite.x5, ids, 64, stream=stream))
        chain.append(_graph_us(fns, stream)[0] * 2)
    q4.q4_set_launch_overlap(True)
    out["chain router -> moe_q4_swiglu_gemv (us per pair)"] = {"with_launch_overlap": round(chain[0], 3),
                                                               "without": round(chain[1], 3)}
    del cp
    qs16, d16 = synth.q4_weights(rng, 14336, 2048)
    b16 = q4_bytes(14336, 2048)
    cp, k = cold_copies((cu(qs16), cu(d16)), b16)
    X16 = torch.from_numpy(np.ascontiguousarray(synth.activations(rng, 16, 2048))).to(dev)
    Y16 = torch.empty(16, 14336, device=dev)
    us, sp = _graph_us([lambda c=c: q4.q4_gemv_batched(Y16, c[0], c[1], X16, stream=stream) for c in cp], stream)
    out["q4_gemv_batched 14336x2048 M=16"] = _entry("", b16, us, sp, k, peak, fmas=16 * 14336 * 2048,
                                                    fma_rate=fma_rate,
                                                    fp32_TFLOPs=round(16 * 2 * 14336 * 2048 / us / 1e6, 2))
    del cp
    for v in out.values():
        v.pop("call", None)
    torch.cuda.empty_cache()
    return out


def run_e2e(suite, inputs, stream, steps, table):
    """Each step: copy the step's activations (and expert ids) from pinned host memory in one copy, make the
    eight calls through the Python binding, read every output back to pinned host memory in one copy, wait."""
    import torch

    import quantized_decode_gemv_q4_gb300 as q4

    # the step's activations and ids in pinned host memory, laid out like the suite's packed input buffer
    h_in = suite.in_buf.cpu().pin_memory()
    h_out = torch.empty(suite.out_buf.shape, dtype=suite.out_buf.dtype).pin_memory()
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size()
    step_bytes = sum(t[1] for t in table)
    calls = [suite.calls(s, stream) for s in range(len(suite.sets))]

    def step(i):
        with torch.cuda.stream(stream):
            suite.in_buf.copy_(h_in, non_blocking=True)
            for fn in calls[i % len(calls)]:
                fn()
            h_out.copy_(suite.out_buf, non_blocking=True)
        stream.synchronize()

    for i in range(5):
        step(i)
    t0 = time.perf_counter()
    for i in range(steps):
        step(i)
    dt = time.perf_counter() - t0
    assert q4.q4_device_faults() == 0
    return {"value": round(step_bytes * steps / dt / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(dt / steps * 1e3, 4),
            "path": "python binding, eager launches, one pinned host copy in and one out, one host sync per step"}


def cpu_baseline(inputs):
    """The oracle on the host: on all cores (each call's rows split over one thread per core), with the
    single-threaded pass beside it. Each leg runs about 10 s of host work on a row sample of every matrix."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    o = oracle.default()

    def leg(pool, parts):
        t0 = time.perf_counter()
        oracle_step(o, inputs, 1.0 / 64, pool, parts)
        t_full = (time.perf_counter() - t0) * 64
        frac = min(1.0, 10.0 / t_full)  # aim at about 10 s of host work: a row sample, or whole passes
        passes = 1
        if frac == 1.0:  # time one whole pass, then repeat it to about 10 s
            t0 = time.perf_counter()
            oracle_step(o, inputs, 1.0, pool, parts)
            passes = max(1, int(round(10.0 / (time.perf_counter() - t0))))
        t0 = time.perf_counter()
        done = sum(oracle_step(o, inputs, frac, pool, parts) for _ in range(passes))
        dt = time.perf_counter() - t0
        return done / dt / 1e9, frac, dt, passes

    cores = host_cores()
    with ThreadPoolExecutor(cores) as pool:
        v_all, f_all, t_all, n_all = leg(pool, cores)
    v_one, f_one, t_one, n_one = leg(None, 1)
    return {"value": round(v_all, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_all} pass(es) of the suite over the first {f_all:.3f} of every matrix's rows (MoE: of "
                      f"every expert's rows), each call's rows split over {cores} threads; {t_all:.1f} s fp64",
            "single_thread": {"value": round(v_one, 4), "cores": 1,
                              "sample": f"{n_one} pass(es) over the first {f_one:.3f} of every matrix's rows, one "
                                        f"thread; {t_one:.1f} s"}}


CASES = ["c1", "c2", "c3", "c4m1", "c4m2", "c4m4", "c4m8", "c5", "pure_q4", "pure_q4k", "pure_moe", "router",
         "c3_swiglu", "c5_swiglu", "q4k_batched_m1", "q4k_batched_m8", "c4m16", "fma"]


def run_case(args):
    """A few plain calls of one workload (for profilers): no graphs, no timing, one replica."""
    import torch

    import quantized_decode_gemv_q4_gb300 as q4

    torch.cuda.set_device(0)
    inputs = make_inputs()
    suite = Suite(inputs, 1, torch.device("cuda", 0))
    fns = suite.calls(0)
    w = suite.sets[0]
    dev = suite.x1.device
    rng = np.random.default_rng(7)

    def on_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def router():  # 64 experts x 2048, the MoE tokens, top-8
        rq, rd = synth.q4_weights(rng, 64, 2048)
        rq, rd = on_dev(rq), on_dev(rd)
        ids = torch.empty(8, 8, dtype=torch.int32, device=dev)
        wts = torch.empty(8, 8, device=dev)
        return lambda: q4.moe_router_q4(ids, wts, rq, rd, suite.x5, 8, True)

    def q4k_batched(M):  # the gate matrix of the gate+up workload at M vectors
        X = on_dev(synth.activations(rng, M, 3584))
        Y = torch.empty(M, 18944, device=dev)
        return lambda: q4.q4k_gemv_batched(Y, w["c3"][0], X)

    def c4m16():  # 14336 x 2048 at 16 vectors
        qs, d = synth.q4_weights(rng, 14336, 2048)
        qs, d = on_dev(qs), on_dev(d)
        X = on_dev(synth.activations(rng, 16, 2048))
        Y = torch.empty(16, 14336, device=dev)
        return lambda: q4.q4_gemv_batched(Y, qs, d, X)

    def fma():  # the FMA-ceiling instrument at the M=8 call's FMA count
        sink = torch.empty(1024, device=dev)
        return lambda: q4.q4_fma_ceiling(sink, 8 * 14336 * 4096)

    ysw = torch.empty(18944, device=dev)
    ymo = torch.empty(8, 8, 1408, device=dev)
    c3eps = float(inputs[2]["eps"])
    makers = {"c1": lambda: fns[0], "c2": lambda: fns[1], "c3": lambda: fns[2], "c4m1": lambda: fns[3],
              "c4m2": lambda: fns[4], "c4m4": lambda: fns[5], "c4m8": lambda: fns[6], "c5": lambda: fns[7],
              "pure_q4": lambda: lambda: q4.q4_pure_read(suite.Y4[3][0], w["c4"][0][0], w["c4"][0][1]),
              "pure_q4k": lambda: lambda: q4.q4k_pure_read(suite.y3g, w["c3"][0]),
              "pure_moe": lambda: lambda: q4.moe_q4_pure_read(suite.y5g, suite.y5u, *w["c5"], suite.ids5, 64),
              "router": router,
              "c3_swiglu": lambda: lambda: q4.fused_gateup_swiglu_q4k_gemv(ysw, w["c3"][0], w["c3"][1], suite.x3,
                                                                            suite.g3, c3eps),
              "c5_swiglu": lambda: lambda: q4.moe_q4_swiglu_gemv(ymo, *w["c5"], suite.x5, suite.ids5, 64),
              "q4k_batched_m1": lambda: q4k_batched(1), "q4k_batched_m8": lambda: q4k_batched(8),
              "c4m16": c4m16, "fma": fma}
    pick = makers[args.case]()
    for _ in range(args.iters):
        pick()
    torch.cuda.synchronize()
    assert q4.q4_device_faults() == 0
    print(f"case {args.case}: {args.iters} calls ok", flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=CASES, help="run a few calls of one workload (for profilers) and exit")
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args(argv)
    if args.case:
        return run_case(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
