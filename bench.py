"""Benchmark: Q4_0 matmul effective weight GB/s on Qwen2.5-7B decode linears.

Workload (one "step"): the 28-layer stack of Qwen2.5-7B linear shapes
(q/o 3584x3584, k/v 512x3584, gate/up 18944x3584, down 3584x18944 as N x K),
all stored as Q4_0 (3.67 GB of packed weights, far larger than L2), each
multiplied by M activation rows for every M in {1, 2, 3, 4, 5, 8}: 6 x 196
q4mm_forward calls.  Weights are N(0, 0.02^2) and activations N(0, 1), seeded
(synthetic; no checkpoint).  value = weight bytes streamed per step / step time.

Per step, for each M and each linear type, the 28 calls of that type are one
CUDA graph replay bracketed by CUDA events on the launching stream; those
events give each kernel's average launch duration for the roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle (fp64, OpenMP on the host cores) on a
bounded sample of the same workload.  Under torchrun each rank runs its own
replica of the workload (the path does not shard: replicas only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M_SWEEP = (1, 2, 3, 4, 5, 8)
TYPES = ("q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj")
# calls per layer: the projections that share their input go in one grouped call
GROUPS = (("qkv", ("q_proj", "k_proj", "v_proj")), ("o", ("o_proj",)),
          ("gate_up", ("gate_proj", "up_proj")), ("down", ("down_proj",)))
METRIC = "Q4 matmul effective weight GB/s and token-rows/s vs M (1-256); % of HBM peak"
WORKLOAD = "qwen2.5-7b decode linears, Q4_0, 28-layer stack (q,k,v,o,gate,up,down), M sweep 1,2,3,4,5,8"
BLOCK_BYTES_PER_WEIGHT = 18.0 / 32.0

# DRAM traffic of the dominant kernel from one ncu capture, per launch, with the
# hash of the kernel source it was taken on (null once the kernel changes).
TRAFFIC = {
    "source_hash": "a66b813a87e0b4b9",
    "grouped": True,
    "m_sweep": [1, 2, 3, 4, 5, 8],
    # dram__bytes_read.sum + dram__bytes_write.sum, mean of the step's 96 mma_kernel launches
    "bytes_per_launch": 32947672,
    "capture": "ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum "
               "--clock-control none -k regex:\"mma_kernel|xpre_kernel\" -s 120 -c 120 python bench.py "
               "--layers 4 --steps 2 --warmup 3 --no-cpu-baseline --no-configs (one step: 4 layers x 4 calls "
               "x 6 M, 96 mma_kernel launches and 24 activation pre-conversion passes)",
}


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# the sources the streaming kernel (mma_kernel) is compiled from
TRAFFIC_SOURCES = ("bit_quantized_matmul_gb300/csrc/q4mm_mma.cu",
                   "bit_quantized_matmul_gb300/csrc/q4mm_epilogue.cuh",
                   "bit_quantized_matmul_gb300/csrc/q4mm_internal.h",
                   "include/q4mm.h")


def _kernel_source_hash():
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", "q4mm_clocks_%d_%d.csv" % (os.getpid(), index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for name, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def _dist():
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local = _env_int("LOCAL_RANK", 0)
    return world, rank, local


def max_over_ranks(ms, world, device=None):
    """The timed region's duration (ms) of the slowest rank: one MAX
    all-reduce over the process group when there are several ranks."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(step_bytes, world, ms_per_step):
    """Whole-job throughput: every rank (an independent replica) streams
    step_bytes per step, in the slowest rank's time."""
    return step_bytes * world / (ms_per_step * 1e-3) / 1e9


# ----------------------------------------------------------------------------- CPU oracle arm

def cpu_oracle_sample(layers=1, Ms=M_SWEEP):
    """Time the oracle (as it stands) on `layers` layers of the stack at each M."""
    import numpy as np

    import oracle
    import synthetic

    work = []
    for layer in range(layers):
        for t_i, name in enumerate(TYPES):
            N, K = synthetic.QWEN7B_LINEARS[name]
            w = synthetic.normal(synthetic.weight_seed(100 + layer, t_i), (N, K), sigma=0.02)
            work.append((name, N, K, oracle.quantize(w)))
    xs = {(M, K): synthetic.normal(synthetic.act_seed(1, M) + K, (M, K))
          for M in Ms for K in (3584, 18944)}
    t0 = time.perf_counter()
    wbytes = 0.0
    rows = 0
    for M in Ms:
        for name, N, K, blocks in work:
            oracle.matmul(blocks, xs[(M, K)])
            wbytes += N * K * BLOCK_BYTES_PER_WEIGHT
        rows += M
    dt = time.perf_counter() - t0
    return {"value": wbytes / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": dt, "rows_per_s": rows / dt,
            "sample": "%d layer(s) of the 7 Qwen2.5-7B linears at M in %s (fp64 oracle, OpenMP over "
                      "(m,n)), weights quantized beforehand" % (layers, list(Ms))}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    # each step: one layer of the stack at every M of the sweep (~1-3 s on 16 cores)
    import oracle  # noqa: F401

    samples = []
    for i in range(args.warmup + args.steps):
        r = cpu_oracle_sample(layers=1)
        if i >= args.warmup:
            samples.append(r)
    value = statistics.median(s["value"] for s in samples)
    secs = sum(s["seconds"] for s in samples)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / len(samples),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "layers_per_step": 1,
                                        "note": "bounded sample: one layer of the stack per step"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": samples[0]["cores"],
                         "kind": "oracle", "sample": samples[0]["sample"]},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

def build_stack(q4, torch, dev, layers):
    """Quantize the 28-layer stack on the device (seeded host draws)."""
    import synthetic

    stack = {name: [] for name in TYPES}
    for layer in range(layers):
        for t_i, name in enumerate(TYPES):
            N, K = synthetic.QWEN7B_LINEARS[name]
            w = synthetic.normal(synthetic.weight_seed(1000 + layer, t_i), (N, K), sigma=0.02)
            wd = torch.from_numpy(w).to(dev)
            stack[name].append(q4.q4_quantize(wd))
            del wd
    torch.cuda.synchronize(dev)
    return stack


def run_gpu(args):
    import numpy as np
    import torch

    import bit_quantized_matmul_gb300 as q4
    import synthetic

    msw = tuple(args.m_sweep)
    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    layers = args.layers
    stack = build_stack(q4, torch, dev, layers)
    stream = torch.cuda.Stream(dev)

    # activations: x for K=3584 inputs and K=18944 (down_proj) per M
    xs = {}
    for M in msw:
        for K in (3584, 18944):
            xs[(M, K)] = torch.from_numpy(synthetic.normal(synthetic.act_seed(1, M) + K, (M, K))).to(dev)
    ys = {}
    for M in msw:
        for name in TYPES:
            N, _ = synthetic.QWEN7B_LINEARS[name]
            ys[(M, name)] = torch.empty((M, N), dtype=torch.float32, device=dev)
    groups = tuple((n, (n,)) for n in TYPES) if args.separate else GROUPS
    flags = q4.Q4MM_BATCH_INVARIANT if args.batch_invariant else 0

    def issue(M, gname):
        names = dict(groups)[gname]
        K = synthetic.QWEN7B_LINEARS[names[0]][1]
        x = xs[(M, K)]
        for layer in range(layers):
            if len(names) == 1:
                q4.q4mm_forward_ex(stack[names[0]][layer], x, flags, y=ys[(M, names[0])], stream=stream)
            else:
                q4.q4mm_forward_group([stack[n][layer] for n in names], x,
                                      ys=[ys[(M, n)] for n in names], flags=flags, stream=stream)

    # warm the library (scratch allocation) before capture
    with torch.cuda.stream(stream):
        for M in msw:
            for gname, _ in groups:
                issue(M, gname)
    torch.cuda.synchronize(dev)

    def issue_stack(M):
        # the whole stack in layer order: q/k/v, o, gate/up, down of layer 0, then layer 1, ...
        for layer in range(layers):
            for gname, names in groups:
                K = synthetic.QWEN7B_LINEARS[names[0]][1]
                x = xs[(M, K)]
                if len(names) == 1:
                    q4.q4mm_forward_ex(stack[names[0]][layer], x, flags, y=ys[(M, names[0])], stream=stream)
                else:
                    q4.q4mm_forward_group([stack[n][layer] for n in names], x,
                                          ys=[ys[(M, n)] for n in names], flags=flags, stream=stream)

    # one CUDA graph per M holds the whole stack; per-call graphs (the
    # `layers` calls of one kind) give the per-call breakdown
    graphs = {}
    for M in msw:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            issue_stack(M)
        graphs[M] = g
        for gname, _ in groups:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                issue(M, gname)
            graphs[(M, gname)] = g
    torch.cuda.synchronize(dev)

    launches = {}
    launches_per_step = 0
    for M in msw:
        for gname, names in groups:
            if len(names) > 1:
                # one launch (pair) covers the group on either path
                grp = flags or (q4.Q4MM_FORCE_MMA if M < q4.q4mm_get_group_m_threshold() else 0)
                _, l, _ = q4.q4mm_plan_info(stack[names[0]][0], M, grp)
            else:
                _, l, _ = q4.q4mm_plan_info(stack[names[0]][0], M, flags)
            launches[(M, gname)] = l
            launches_per_step += l * layers

    wbytes = {name: synthetic.QWEN7B_LINEARS[name][0] * synthetic.QWEN7B_LINEARS[name][1]
              * BLOCK_BYTES_PER_WEIGHT for name in TYPES}
    step_wbytes = sum(wbytes[n] * layers for n in TYPES) * len(msw)

    def algo_bytes(M, gname):
        """Bytes a call must move: packed weights once, x once, y once."""
        names = dict(groups)[gname]
        K = synthetic.QWEN7B_LINEARS[names[0]][1]
        return sum(wbytes[n] + 4.0 * M * synthetic.QWEN7B_LINEARS[n][0] for n in names) + 4.0 * M * K

    ev = {}

    def step(record):
        for M in msw:
            if record:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                graphs[M].replay()
                b.record(stream)
                ev.setdefault(M, []).append((a, b))
            else:
                graphs[M].replay()

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step(False)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    sampler = ClockSampler(local)
    sampler.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(args.steps):
            step(True)
        t1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_per_step = ms / args.steps
    value = whole_job_gbs(step_wbytes, world, ms_per_step)

    # per-M durations over the timed region: each graph replay is the whole
    # stack at one M, bracketed by events on the launching stream
    per_stack = {M: sum(a.elapsed_time(b) for a, b in pairs) / len(pairs) for M, pairs in ev.items()}  # ms
    # per-call breakdown (outside the timed region): the per-kind graphs
    per = {}
    with torch.cuda.stream(stream):
        for M in msw:
            for gname, _ in groups:
                graphs[(M, gname)].replay()
                times = []
                for _ in range(5):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    graphs[(M, gname)].replay()
                    b.record(stream)
                    b.synchronize()
                    times.append(a.elapsed_time(b))
                per[(M, gname)] = statistics.median(times) / layers  # ms per call
    peak, peak_kind = _peaks()
    # roofline over every launch of the step (one kernel function serves them all):
    # algorithmic bytes of all calls / event-timed duration of the stack graphs
    tot_bytes = sum(algo_bytes(M, g) for M in msw for g, _ in groups) * layers
    tot_ms = sum(per_stack[M] for M in msw)
    n_calls = len(msw) * len(groups)
    achieved = tot_bytes / (tot_ms * 1e-3) / 1e9
    traffic = None
    if TRAFFIC and TRAFFIC.get("source_hash") == _kernel_source_hash() and \
            TRAFFIC.get("grouped") == (not args.separate) and not args.batch_invariant and \
            TRAFFIC.get("m_sweep", list(M_SWEEP)) == list(msw):
        traffic = TRAFFIC.get("bytes_per_launch")
    per_m = {}
    for M in msw:
        t = per_stack[M]
        b = sum(wbytes[n] * layers for n in TYPES)
        per_m[str(M)] = {
            "weight_gbs": b / (t * 1e-3) / 1e9,
            "token_rows_per_s": M / (t * 1e-3),
            "frac_of_measured_hbm": b / (t * 1e-3) / 1e9 / peak,
            "call_us": {g: per[(M, g)] * 1e3 for g, _ in groups},
        }

    # ---- end to end through the C ABI: pinned host x in, every output out ----
    e2e = e2e_c_abi(q4, torch, dev, stack, msw, layers, args.steps, stream, world, flags)
    e2e_value = whole_job_gbs(step_wbytes, world, e2e["ms_per_step"])

    configs = None
    if not args.no_configs:
        configs = extra_configs(q4, torch, dev, stack, stream, args, rank == 0 and world == 1)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(layers=1, Ms=msw)
        cpu = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}

    if world > 1:
        torch.distributed.barrier()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD if msw == M_SWEEP else
                       WORKLOAD.replace("M sweep 1,2,3,4,5,8", "M sweep " + ",".join(map(str, msw))),
                       "layers": layers, "M_sweep": list(msw),
                       "weights": "Q4_0 (18 B per 32 weights), N(0,0.02^2)", "activations": "fp32 N(0,1)",
                       "l2": "inputs larger than L2 (%.2f GB packed weight stack, streamed once per M)"
                             % (sum(wbytes[n] * layers for n in TYPES) / 1e9),
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "calls_per_layer": [g for g, _ in groups],
                       "graphs": "one CUDA graph per M holding the whole stack in layer order (programmatic "
                                 "dependent launch between consecutive calls); call_us from per-kind graphs",
                       "mode": "batch-invariant" if args.batch_invariant else "default",
                       "m_threshold": q4.q4mm_get_m_threshold(),
                       "group_m_threshold": q4.q4mm_get_group_m_threshold()},
            "token_rows_per_s": sum(msw) * world / (ms_per_step * 1e-3),
            "per_M": per_m,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind
                         if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "kernel": "q4mm kernels (mma_kernel below the M threshold, with the activation "
                                   "pre-conversion pass of row-group launches of 4-8 rows; xop_kernel + "
                                   "tc_kernel from the threshold), every "
                                   "call of one step (%d calls, %d kernel launches)"
                                   % (n_calls * layers, launches_per_step),
                         "algorithmic_bytes_per_call": tot_bytes / (n_calls * layers),
                         "algorithmic_bytes_rule": "0.5625*sum(N_i*K) + 4*M*K + 4*M*sum(N_i) per call"},
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": e2e["h2d"],
                    "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": e2e["ms_per_step"],
                    "calls_per_step": e2e["calls"],
                    "how": "every call of the step through the C ABI (q4mm_forward_group for q/k/v and "
                           "gate/up, q4mm_forward for o and down), x copied in from pinned host memory per M, "
                           "every output of every layer copied back to pinned host memory per M on a second "
                           "stream overlapping the next M's calls; the timed region ends after the last copy"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    for name in TYPES:
        for W in stack[name]:
            W.free()
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def _graph_us(torch, stream, issue, reps, calls, warm=3):
    """Median per-call time (us) of `issue` (which makes `calls` calls),
    captured once in a CUDA graph and replayed `reps` times."""
    with torch.cuda.stream(stream):
        issue()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        issue()
    times = []
    with torch.cuda.stream(stream):
        for r in range(warm + reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            if r >= warm:
                times.append(a.elapsed_time(b) * 1e3 / calls)
    del g
    return statistics.median(times)


def e2e_c_abi(q4, torch, dev, stack, msw, layers, steps, stream, world, flags=0):
    """The step end to end through the library's C ABI: per M, x is copied in
    from pinned host memory, every call is made through the C entry points
    (argument checks, path choice and launches inside the timed region), and
    the outputs of every layer and projection (one arena per M) are copied
    back to pinned host memory, on a second stream that overlaps the next M's
    calls.  Returns ms per step and the bytes moved."""
    import ctypes

    import synthetic

    lib = q4.raw_library()
    sh = ctypes.c_void_p(stream.cuda_stream)
    per_m = []
    h2d = d2h = 0
    calls = 0
    for M in msw:
        xh = {K: torch.from_numpy(synthetic.normal(synthetic.act_seed(1, M) + K, (M, K))).pin_memory()
              for K in (3584, 18944)}
        xd = {K: torch.empty((M, K), dtype=torch.float32, device=dev) for K in (3584, 18944)}
        per_layer = sum(synthetic.QWEN7B_LINEARS[n][0] for n in TYPES) * M
        arena = torch.empty(layers * per_layer, dtype=torch.float32, device=dev)
        arena_h = torch.empty(layers * per_layer, dtype=torch.float32).pin_memory()
        h2d += sum(v.numel() * 4 for v in xh.values())
        d2h += arena.numel() * 4
        ops = []
        off = 0
        for layer in range(layers):
            yp = {}
            for n in TYPES:
                yp[n] = arena.data_ptr() + off * 4
                off += synthetic.QWEN7B_LINEARS[n][0] * M
            for gname, names in GROUPS:
                K = synthetic.QWEN7B_LINEARS[names[0]][1]
                if len(names) == 1:
                    ops.append((lib.q4mm_forward_ex, (stack[names[0]][layer].handle, ctypes.c_void_p(xd[K].data_ptr()),
                                                      ctypes.c_void_p(yp[names[0]]), M, flags, sh)))
                else:
                    hw = (ctypes.c_void_p * len(names))(*[stack[n][layer].handle.value for n in names])
                    hy = (ctypes.c_void_p * len(names))(*[yp[n] for n in names])
                    ops.append((lib.q4mm_forward_group, (hw, len(names), ctypes.c_void_p(xd[K].data_ptr()), hy, M,
                                                         flags, sh)))
        calls += len(ops)
        per_m.append((xh, xd, arena, arena_h, ops))

    # the outputs of one M are copied back on a second stream while the next
    # M's calls run; an M's calls in the next step wait until its arena has
    # been copied out (the arena is rewritten)
    copy_stream = torch.cuda.Stream(dev)
    done = [torch.cuda.Event() for _ in per_m]    # an M's calls finished
    copied = [torch.cuda.Event() for _ in per_m]  # its arena copied back

    def step():
        for i, (xh, xd, arena, arena_h, ops) in enumerate(per_m):
            for K in (3584, 18944):
                xd[K].copy_(xh[K], non_blocking=True)
            stream.wait_event(copied[i])
            for fn, a in ops:
                st = fn(*a)
                if st != 0:
                    raise RuntimeError("C ABI call failed with status %d" % st)
            done[i].record(stream)
            copy_stream.wait_event(done[i])
            with torch.cuda.stream(copy_stream):
                arena_h.copy_(arena, non_blocking=True)
            copied[i].record(copy_stream)

    with torch.cuda.stream(stream):
        for _ in range(2):
            step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            step()
        for ev in copied:  # every copy of the last step is inside the timed region
            stream.wait_event(ev)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / steps
    return {"ms_per_step": ms, "h2d": h2d, "d2h": d2h, "calls": calls}


def _oracle_single_core():
    """The oracle on one host core: the 896 x 896 call at M = 1, 2, 4 and the
    gate projection (18944 x 3584) at M = 1, quantized beforehand."""
    import numpy as np

    import oracle
    import synthetic

    out = {}
    prev = oracle.set_threads(1)
    try:
        for (name, N, K, Ms) in (("896x896", 896, 896, (1, 2, 4)), ("gate_proj", 18944, 3584, (1,))):
            blocks = oracle.quantize(synthetic.normal(synthetic.weight_seed(1, 0), (N, K), sigma=0.02))
            for M in Ms:
                x = synthetic.normal(synthetic.act_seed(1, M), (M, K))
                t0 = time.perf_counter()
                oracle.matmul(blocks, x)
                dt = time.perf_counter() - t0
                out["%s@M=%d" % (name, M)] = {"s": dt, "weight_gbs": N * K * BLOCK_BYTES_PER_WEIGHT / dt / 1e9,
                                                "rows_per_s": M / dt}
    finally:
        oracle.set_threads(prev)
    return {"cores": 1, "kind": "oracle", "cases": out}


def extra_configs(q4, torch, dev, stack, stream, args, with_oracle):
    """Every configuration of the metric besides the headline step: the
    896 x 896 call, the M = 124 mixed step in default and batch-invariant mode,
    the LM-head greedy pick, and the M sweep on gate_proj and on the stack
    with the measured streaming / tensor-core crossover."""
    import synthetic

    peak, _ = _peaks()
    reps = max(5, min(args.steps, 20))
    out = {}

    # ---- 896 x 896, M = 1, 2, 4: 400 weight copies (180 MB, beyond L2) in one graph
    N = K = 896
    copies = 400
    Ws = [q4.q4_quantize(torch.from_numpy(synthetic.normal(synthetic.weight_seed(1, c), (N, K), sigma=0.02)).to(dev))
          for c in range(copies)]
    wb = N * K * BLOCK_BYTES_PER_WEIGHT
    c1 = {}
    for M in (1, 2, 4):
        x = torch.from_numpy(synthetic.normal(synthetic.act_seed(1, M), (M, K))).to(dev)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)

        def issue():
            for W in Ws:
                q4.q4mm_forward(W, x, y=y, stream=stream)
        us = _graph_us(torch, stream, issue, reps, copies)
        singles = []
        with torch.cuda.stream(stream):
            for r in range(23):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                q4.q4mm_forward(Ws[(7 * r) % copies], x, y=y, stream=stream)
                b.record(stream)
                b.synchronize()
                if r >= 3:
                    singles.append(a.elapsed_time(b) * 1e3)
        c1[str(M)] = {"us_per_call_graph": us, "us_single_launch": statistics.median(singles),
                      "weight_gbs": wb / us / 1e3, "frac_of_measured_hbm": wb / us / 1e3 / peak,
                      "token_rows_per_s": M / us * 1e6}
    for W in Ws:
        W.free()
    out["c1_896x896"] = {"workload": "Q4_0 896x896, %d weight copies in one CUDA graph (beyond L2); the single "
                                     "launch is one call between events" % copies, "per_M": c1}

    # ---- M = 124 mixed step (120 prefill + 4 verify rows) through gate/up/down
    L3 = min(8, len(stack["gate_proj"]))
    M = 124
    x1 = torch.from_numpy(synthetic.normal(synthetic.act_seed(3, M), (M, 3584))).to(dev)
    x2 = torch.from_numpy(synthetic.normal(synthetic.act_seed(3, M) + 1, (M, 18944))).to(dev)
    yg = torch.empty((M, 18944), device=dev)
    yu = torch.empty((M, 18944), device=dev)
    yd = torch.empty((M, 3584), device=dev)
    wb3 = sum(synthetic.QWEN7B_LINEARS[n][0] * synthetic.QWEN7B_LINEARS[n][1]
              for n in ("gate_proj", "up_proj", "down_proj")) * BLOCK_BYTES_PER_WEIGHT
    c3 = {}
    decode = {}
    inv_tc = q4.Q4MM_BATCH_INVARIANT | q4.Q4MM_FORCE_TC
    for mode, fl in (("default", 0), ("batch_invariant", q4.Q4MM_BATCH_INVARIANT),
                     ("batch_invariant_tc", inv_tc)):
        for rows, res in ((M, c3), (1, decode)):
            def issue():
                for l in range(L3):
                    q4.q4mm_forward_group([stack["gate_proj"][l], stack["up_proj"][l]], x1[:rows],
                                          ys=[yg[:rows], yu[:rows]], flags=fl, stream=stream)
                    q4.q4mm_forward_ex(stack["down_proj"][l], x2[:rows], fl, y=yd[:rows], stream=stream)
            us = _graph_us(torch, stream, issue, reps, L3)
            _, lg, _ = q4.q4mm_plan_info(stack["gate_proj"][0], rows, fl)
            _, ld, _ = q4.q4mm_plan_info(stack["down_proj"][0], rows, fl)
            res[mode] = {"us_per_layer": us, "weight_gbs": wb3 / us / 1e3, "token_rows_per_s": rows / us * 1e6,
                         "launches_gate_up_down": [lg, ld]}
    c3["batch_invariant_over_default"] = c3["batch_invariant"]["us_per_layer"] / c3["default"]["us_per_layer"]
    c3["batch_invariant_tc_over_default"] = \
        c3["batch_invariant_tc"]["us_per_layer"] / c3["default"]["us_per_layer"]
    out["c3_mixed_m124"] = {"workload": "M = 124 (120 prefill + 4 verify rows) through gate/up (one grouped call) "
                                        "and down, %d layers of the 7B stack in one CUDA graph; the same layers "
                                        "at M = 1 in each mode (decode_m1)" % L3,
                            "modes": c3, "decode_m1": decode,
                            "launches": "q4mm_plan_info of gate_proj and down_proj alone"}

    # ---- LM head, fused greedy pick
    out["c4_lm_head"] = lm_head_cases(q4, torch, dev, stream, reps)

    # ---- M sweep on gate_proj (28 copies) and on the stack (all layers), and the crossover
    sweep = (1, 2, 3, 4, 5, 6, 8, 16, 32, 64, 128, 256)
    Lg = len(stack["gate_proj"])
    gb = 18944 * 3584 * BLOCK_BYTES_PER_WEIGHT
    lb = sum(synthetic.QWEN7B_LINEARS[n][0] * synthetic.QWEN7B_LINEARS[n][1] for n in TYPES) * BLOCK_BYTES_PER_WEIGHT
    gate, stk = {}, {}
    for M in sweep:
        xa = torch.from_numpy(synthetic.normal(synthetic.act_seed(5, M), (M, 3584))).to(dev)
        xb = torch.from_numpy(synthetic.normal(synthetic.act_seed(5, M) + 1, (M, 18944))).to(dev)
        ys = {n: torch.empty((M, synthetic.QWEN7B_LINEARS[n][0]), device=dev) for n in TYPES}

        def issue_gate(fl=0):
            for l in range(Lg):
                q4.q4mm_forward_ex(stack["gate_proj"][l], xa, fl, y=ys["gate_proj"], stream=stream)
        us = _graph_us(torch, stream, issue_gate, reps, Lg)
        gate[str(M)] = {"us": us, "weight_gbs": gb / us / 1e3, "frac_of_measured_hbm": gb / us / 1e3 / peak,
                        "token_rows_per_s": M / us * 1e6, "path": q4.q4mm_select_path(stack["gate_proj"][0], M)}

        def issue_stack():
            for l in range(Lg):
                for gname, names in GROUPS:
                    x = xb if names[0] == "down_proj" else xa
                    if len(names) == 1:
                        q4.q4mm_forward(stack[names[0]][l], x, y=ys[names[0]], stream=stream)
                    else:
                        q4.q4mm_forward_group([stack[n][l] for n in names], x, ys=[ys[n] for n in names],
                                              stream=stream)
        us = _graph_us(torch, stream, issue_stack, max(3, reps // 2), Lg)
        stk[str(M)] = {"us_per_layer": us, "weight_gbs": lb / us / 1e3, "frac_of_measured_hbm": lb / us / 1e3 / peak,
                       "token_rows_per_s": M / us * 1e6}
    # both paths forced around the threshold, on gate_proj
    paths = {}
    for M in (8, 12, 16, 17, 20, 24, 32, 64):
        xa = torch.from_numpy(synthetic.normal(synthetic.act_seed(6, M), (M, 3584))).to(dev)
        yg = torch.empty((M, 18944), device=dev)

        def issue_forced(fl):
            for l in range(Lg):
                q4.q4mm_forward_ex(stack["gate_proj"][l], xa, fl, y=yg, stream=stream)
        paths[str(M)] = {"streaming_us": _graph_us(torch, stream, lambda: issue_forced(q4.Q4MM_FORCE_MMA), reps, Lg),
                         "tensor_core_us": _graph_us(torch, stream, lambda: issue_forced(q4.Q4MM_FORCE_TC), reps, Lg)}
    cross = None
    for M in (8, 12, 16, 17, 20, 24, 32, 64):
        if all(paths[str(m)]["tensor_core_us"] <= paths[str(m)]["streaming_us"]
               for m in (8, 12, 16, 17, 20, 24, 32, 64) if m >= M):
            cross = M
            break
    out["c5_m_sweep"] = {"workload": "M sweep on gate_proj 18944x3584 (%d copies) and on the %d-layer stack "
                                     "(grouped q/k/v and gate/up calls)" % (Lg, Lg),
                         "gate_proj": gate, "stack": stk, "gate_proj_both_paths": paths,
                         "measured_crossover_gate": cross, "m_threshold": q4.q4mm_get_m_threshold(),
                         "group_m_threshold": q4.q4mm_get_group_m_threshold()}
    # ---- the decoder layer with the gated step fused (gate/up -> h -> down), the
    # whole stack in one graph, against the seven linears with g and u written
    Lf = len(stack["gate_proj"])
    fused = {}
    for M in (1, 4, 8):
        xa = torch.from_numpy(synthetic.normal(synthetic.act_seed(8, M), (M, 3584))).to(dev)
        xb = torch.from_numpy(synthetic.normal(synthetic.act_seed(8, M) + 1, (M, 18944))).to(dev)
        ys = {n: torch.empty((M, synthetic.QWEN7B_LINEARS[n][0]), device=dev) for n in TYPES}
        h = torch.empty((M, 18944), device=dev)

        def issue_fused():
            for l in range(Lf):
                q4.q4mm_forward_group([stack[n][l] for n in ("q_proj", "k_proj", "v_proj")], xa,
                                      ys=[ys[n] for n in ("q_proj", "k_proj", "v_proj")], stream=stream)
                q4.q4mm_forward(stack["o_proj"][l], xa, y=ys["o_proj"], stream=stream)
                q4.q4mm_forward_gated(stack["gate_proj"][l], stack["up_proj"][l], xa, h=h, stream=stream)
                q4.q4mm_forward(stack["down_proj"][l], h, y=ys["down_proj"], stream=stream)

        def issue_plain():
            for l in range(Lf):
                q4.q4mm_forward_group([stack[n][l] for n in ("q_proj", "k_proj", "v_proj")], xa,
                                      ys=[ys[n] for n in ("q_proj", "k_proj", "v_proj")], stream=stream)
                q4.q4mm_forward(stack["o_proj"][l], xa, y=ys["o_proj"], stream=stream)
                q4.q4mm_forward_group([stack["gate_proj"][l], stack["up_proj"][l]], xa,
                                      ys=[ys["gate_proj"], ys["up_proj"]], stream=stream)
                q4.q4mm_forward(stack["down_proj"][l], xb, y=ys["down_proj"], stream=stream)
        uf = _graph_us(torch, stream, issue_fused, max(3, reps // 2), Lf)
        up = _graph_us(torch, stream, issue_plain, max(3, reps // 2), Lf)
        fused[str(M)] = {"fused_us_per_layer": uf, "seven_linears_us_per_layer": up,
                         "fused_weight_gbs": lb / uf / 1e3, "fused_frac_of_measured_hbm": lb / uf / 1e3 / peak,
                         "output_bytes_saved_per_layer": 4 * M * 18944}
    out["next2_fused_gated_layer"] = {"workload": "the %d-layer 7B stack in one CUDA graph per M, each layer q/k/v "
                                                  "(grouped), o, q4mm_forward_gated (gate, up -> h = SiLU(g)*u, "
                                                  "only h written), down(h); against the same layer with gate/up "
                                                  "as a grouped call writing g and u" % Lf, "per_M": fused}
    if with_oracle:
        out["oracle_single_core"] = _oracle_single_core()
    return out



def run_path_sweep(args):
    """Measure both kernel paths (CUDA-core streaming vs tensor-core) per M on
    the 7B shapes; the crossover is the library's M threshold."""
    import torch

    import bit_quantized_matmul_gb300 as q4
    import synthetic

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    layers = args.layers
    stack = build_stack(q4, torch, dev, layers)
    stream = torch.cuda.Stream(dev)
    sweep = (1, 2, 3, 4, 5, 6, 8, 16, 24, 32, 48, 64, 128, 256)
    paths = {"simt": q4.Q4MM_FORCE_SIMT, "mma": q4.Q4MM_FORCE_MMA, "tc": q4.Q4MM_FORCE_TC}
    out = {}
    groups_out = {}
    for M in sweep:
        xs = {K: torch.from_numpy(synthetic.normal(synthetic.act_seed(5, M) + K, (M, K))).to(dev)
              for K in (3584, 18944)}
        for name in ("q_proj", "k_proj", "gate_proj", "down_proj"):
            N, K = synthetic.QWEN7B_LINEARS[name]
            y = torch.empty((M, N), dtype=torch.float32, device=dev)
            for pname, flags in paths.items():
                def issue():
                    for W in stack[name]:
                        q4.q4mm_forward_ex(W, xs[K], flags, y=y, stream=stream)
                with torch.cuda.stream(stream):
                    issue()
                torch.cuda.synchronize(dev)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    issue()
                with torch.cuda.stream(stream):
                    for _ in range(3):
                        g.replay()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    for _ in range(5):
                        g.replay()
                    b.record(stream)
                torch.cuda.synchronize(dev)
                us = a.elapsed_time(b) * 1e3 / (5 * layers)
                wb = N * K * BLOCK_BYTES_PER_WEIGHT
                out.setdefault(name, {}).setdefault(str(M), {})[pname] = {
                    "us": us, "weight_gbs": wb / us / 1e3, "rows_per_s": M / us * 1e6}
                del g
        # grouped calls on the streaming path (one launch for the group); on
        # the tensor-core path a group is one call per weight
        for gname, names in GROUPS:
            if len(names) < 2:
                continue
            K = synthetic.QWEN7B_LINEARS[names[0]][1]
            ys = [torch.empty((M, synthetic.QWEN7B_LINEARS[n][0]), dtype=torch.float32, device=dev)
                  for n in names]

            def time_group(flags):
                def issue_group():
                    for li in range(layers):
                        q4.q4mm_forward_group([stack[n][li] for n in names], xs[K], ys=ys,
                                              flags=flags, stream=stream)
                with torch.cuda.stream(stream):
                    issue_group()
                torch.cuda.synchronize(dev)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    issue_group()
                with torch.cuda.stream(stream):
                    for _ in range(3):
                        g.replay()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    for _ in range(5):
                        g.replay()
                    b.record(stream)
                torch.cuda.synchronize(dev)
                return a.elapsed_time(b) * 1e3 / (5 * layers)

            # streaming: one launch per 16 rows over the group; tensor cores:
            # one launch pair over the group (the group threshold forced to 1)
            rec = {"mma_group_us": time_group(q4.Q4MM_FORCE_MMA)}
            old_thr = q4.q4mm_get_group_m_threshold()
            q4.q4mm_set_group_m_threshold(1)
            try:
                rec["tc_group_us"] = time_group(0)
            finally:
                q4.q4mm_set_group_m_threshold(old_thr)
            groups_out.setdefault(gname, {})[str(M)] = rec
    # threshold: smallest M of the sweep from which one decoder layer (q, o like
    # q_proj; k, v like k_proj; gate, up like gate_proj; down) takes no longer
    # on the tcgen05 path than on the streaming path, for every larger M too
    weight = {"q_proj": 2, "k_proj": 2, "gate_proj": 2, "down_proj": 1}

    def layer_us(M, path):
        return sum(c * out[n][str(M)][path]["us"] for n, c in weight.items())

    thr = None
    for i, M in enumerate(sweep):
        if all(layer_us(m, "tc") <= layer_us(m, "mma") for m in sweep[i:]):
            thr = M
            break
    # grouped calls: q/k/v and gate/up as one streaming launch each, against
    # one tensor-core call per weight (o and down are single calls either way)
    like = {"q_proj": "q_proj", "k_proj": "k_proj", "v_proj": "k_proj", "gate_proj": "gate_proj",
            "up_proj": "gate_proj"}
    for gname, names in GROUPS:
        if gname in groups_out:
            for M in sweep:  # for reference: the group's weights as separate tcgen05 calls
                groups_out[gname][str(M)]["tc_separate_us"] = sum(out[like[n]][str(M)]["tc"]["us"]
                                                                  for n in names)

    def group_layer(M, path):
        key = "tc_group_us" if path == "tc" else "mma_group_us"
        return sum(groups_out[g][str(M)][key] for g in groups_out)

    gthr = None
    for i, M in enumerate(sweep):
        if all(group_layer(m, "tc") <= group_layer(m, "mma") for m in sweep[i:]):
            gthr = M
            break
    # The crossover of "Row-by-Row GEMV to the Rescue": one decoder layer (the
    # seven linears as separate calls) at M = 1..8 under each path; ratio =
    # throughput of a path / throughput of the tensor-core GEMM path (the
    # pages' 134.3% / 109.2% / 90.7% at 3 / 4 / 5 requests compare their
    # row-by-row GEMV with their GEMM the same way, on Metal).
    cross = {}
    pflags = {"row_by_row": q4.Q4MM_ROW_BY_ROW, "simt_single_launch": q4.Q4MM_FORCE_SIMT,
              "mma_single_launch": q4.Q4MM_FORCE_MMA, "tensor_core_gemm": q4.Q4MM_FORCE_TC, "default": 0}
    for M in range(1, 9):
        xs = {K: torch.from_numpy(synthetic.normal(synthetic.act_seed(7, M) + K, (M, K))).to(dev)
              for K in (3584, 18944)}
        ys = {n: torch.empty((M, synthetic.QWEN7B_LINEARS[n][0]), device=dev) for n in TYPES}
        rec = {}
        for pname, fl in pflags.items():
            def issue_layer():
                for li in range(layers):
                    for n in TYPES:
                        K = synthetic.QWEN7B_LINEARS[n][1]
                        q4.q4mm_forward_ex(stack[n][li], xs[K], fl, y=ys[n], stream=stream)
            rec[pname + "_us_per_layer"] = _graph_us(torch, stream, issue_layer, 5, layers)
        for pname in pflags:
            rec[pname + "_vs_gemm"] = rec["tensor_core_gemm_us_per_layer"] / rec[pname + "_us_per_layer"]
        cross[str(M)] = rec
    print(json.dumps({"path_sweep": out, "measured_threshold": thr, "groups": groups_out,
                      "measured_group_threshold": gthr, "layers": layers, "sweep": list(sweep),
                      "row_by_row_crossover": cross}),
          flush=True)
    for name in TYPES:
        for W in stack[name]:
            W.free()
    return 0


def lm_head_cases(q4, torch, dev, stream, reps=10):
    """Fused greedy pick (q4mm_argmax through the C ABI) on the Qwen2.5-7B LM
    head, 152064 x 3584 Q4_0 (N(0, 0.02^2) weights, fp32 N(0,1) activations),
    at M = 1, 4, 16.  Two weight copies (612 MB, far beyond L2) alternate
    between the 20 calls of one CUDA graph; no logits are written."""
    import synthetic

    N, K = synthetic.LM_HEAD
    Ws = []
    for c in range(2):
        w = torch.from_numpy(synthetic.normal(synthetic.weight_seed(3, 10 + c), (N, K), sigma=0.02)).to(dev)
        Ws.append(q4.q4_quantize(w))
        del w
    wbytes = N * K * BLOCK_BYTES_PER_WEIGHT
    peak, kind = _peaks()
    lib = q4.raw_library()
    cases = {}
    for M in (1, 4, 16):
        x = torch.from_numpy(synthetic.normal(synthetic.act_seed(3, M), (M, K))).to(dev)
        idx = torch.empty((M,), dtype=torch.int32, device=dev)
        mx = torch.empty((M,), dtype=torch.float32, device=dev)
        calls = 20

        def issue():
            for r in range(calls):
                st = lib.q4mm_argmax(Ws[r % 2].handle, x.data_ptr(), idx.data_ptr(), mx.data_ptr(), M,
                                     stream.cuda_stream)
                assert st == q4.Q4_OK, st
        us = _graph_us(torch, stream, issue, reps, calls)
        path = q4.q4mm_plan_info(Ws[0], M)[0]
        cases[str(M)] = {"us_per_call": us, "weight_gbs": wbytes / (us * 1e-6) / 1e9,
                         "frac_of_measured_hbm": wbytes / (us * 1e-6) / 1e9 / peak,
                         "token_rows_per_s": M / (us * 1e-6), "path": int(path)}
    assert q4.q4_device_status() == q4.Q4_OK
    for W in Ws:
        W.free()
    return {"workload": "qwen2.5-7b LM head 152064x3584 Q4_0, M = 1, 4, 16, fused argmax (no logits written)",
            "l2": "two weight copies (612 MB) alternate", "per_M": cases, "peak_gbs": peak, "peak_source": kind}


def run_lm_head(args):
    """The LM-head greedy pick alone; prints one JSON line (GB/s of packed
    weight bytes)."""
    import torch

    import bit_quantized_matmul_gb300 as q4

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    c = lm_head_cases(q4, torch, dev, stream, max(5, args.steps))
    line = {"metric": "LM-head greedy pick (fused argmax) weight GB/s", "unit": "GB/s",
            "value": c["per_M"]["1"]["weight_gbs"], "n_gpus": 1, "higher_is_better": True, "dtype": "f32",
            "data": "synthetic", "config": {"workload": c["workload"], "l2": c["l2"]},
            "cases": c["per_M"], "peak_gbs": c["peak_gbs"], "peak_source": c["peak_source"]}
    print(json.dumps(line), flush=True)
    return 0


def run_kv_append(args):
    """KV-cache append of a Qwen2.5-0.5B-shaped cache (24 layers, 2 KV heads,
    head_dim 64, bf16): a 2,049-row prefill into one slot and a decode step of
    64 requests, with V as a transposed view.  Prints one JSON line; bytes
    moved = new rows read + the same bytes written."""
    import numpy as np
    import torch

    import bit_quantized_matmul_gb300 as q4

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    L, H, D, slots, cap = 24, 2, 64, 64, 4096
    kc = torch.zeros((L, slots, H, cap, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    stream = torch.cuda.Stream(dev)
    cases = {}
    for name, reqs, ctx in (("prefill_2049", [(0, 2049)], 0), ("decode_64x1", [(s, 1) for s in range(slots)], 2049)):
        total = sum(n for _, n in reqs)
        g = torch.Generator(device="cpu").manual_seed(0x4B58)
        k_new = torch.randn((L, total, H, D), generator=g).to(torch.bfloat16).to(dev)
        v_new = torch.randn((L, H, total, D), generator=g).to(torch.bfloat16).to(dev).transpose(1, 2)
        offsets = torch.tensor(np.concatenate([[0], np.cumsum([n for _, n in reqs])]), dtype=torch.int32,
                               device=dev)
        slot = torch.tensor([s for s, _ in reqs], dtype=torch.int32, device=dev)
        pos = torch.full((len(reqs),), ctx, dtype=torch.int32, device=dev)
        reps = 50
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                q4.q4_kv_append(kc, vc, k_new, v_new, offsets, slot, pos, stream=stream)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(reps):
                    q4.q4_kv_append(kc, vc, k_new, v_new, offsets, slot, pos, stream=stream)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = []
        for _ in range(max(1, args.steps)):
            with torch.cuda.stream(stream):
                e0.record(stream)
                graph.replay()
                e1.record(stream)
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1) * 1e3 / reps)
        us = statistics.median(times)
        row_bytes = 2 * L * H * D * 2  # K and V of one packed row, all layers
        moved = 2 * total * row_bytes
        cases[name] = {"us_per_append": us, "gbs": moved / (us * 1e-6) / 1e9, "bytes_moved": moved,
                       "rows": total, "context": ctx,
                       # a cache grown by concatenation re-copies every request's rows each step
                       "bytes_a_concatenating_cache_copies": sum(ctx + n for _, n in reqs) * row_bytes}
    assert q4.q4_device_status() == q4.Q4_OK
    peak, kind = _peaks()
    line = {"metric": "KV-cache append GB/s (new rows read + written)", "unit": "GB/s",
            "value": cases["prefill_2049"]["gbs"], "n_gpus": 1, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": "qwen2.5-0.5b KV cache (24 layers, 2 KV heads, head_dim 64, "
                                                         "bf16, V a transposed view), one launch per append",
                                            "l2": "new rows hot in L2, as the producing kernel leaves them"},
            "cases": cases, "peak_gbs": peak, "peak_source": kind,
            "frac_of_peak": cases["prefill_2049"]["gbs"] / peak}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=28)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config measurements (896x896, M=124 step, LM head, M sweep, "
                         "single-core oracle)")
    ap.add_argument("--m-sweep", type=lambda v: [int(t) for t in v.split(",")], default=list(M_SWEEP),
                    help="token-row counts of the step (default 1,2,3,4,5,8)")
    ap.add_argument("--separate", action="store_true",
                    help="one call per linear instead of grouping q/k/v and gate/up")
    ap.add_argument("--path-sweep", action="store_true",
                    help="time both kernel paths per M and print the measured M threshold")
    ap.add_argument("--batch-invariant", action="store_true",
                    help="run every call of the step in batch-invariant mode (Q4MM_BATCH_INVARIANT)")
    ap.add_argument("--lm-head", action="store_true",
                    help="time the fused greedy pick (q4mm_argmax) on the LM head instead of the step")
    ap.add_argument("--kv-append", action="store_true",
                    help="time the KV-cache append (q4_kv_append) instead of the matmul step")
    args = ap.parse_args()
    if args.kv_append:
        return run_kv_append(args)
    if args.lm_head:
        return run_lm_head(args)
    if args.path_sweep:
        return run_path_sweep(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
