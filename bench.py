#!/usr/bin/env python
"""Benchmark of the int4 group-128 weight-only decode path on one GB300.

Step (what one timed iteration is): one synthetic decode step -- 36 layers x
{fused qkv+gate+up 25,088x3072, o-proj 3072x3072, down 3072x8192} -- plus the
wide output head (65,536x3072) and the argmax over its logits, all int4
group-128 with fp16 scale/min, batch 1, replayed as one CUDA graph (the
rumik-oss-1 page, "Step 3": the whole step -- every projection plus the head --
captured as a single CUDA graph).  Every step streams 2.243 GB of weights, far above the 129 MB L2, so
no L2 flush is needed between steps.

Metric: achieved HBM GB/s of algorithmic bytes (weights + activations +
outputs) per step, plus decode-step microseconds at batch 1 and 8.  The step
is three launches: activation prep, the persistent tile kernel over all 109
matrices, argmax.  The dominant kernel's roofline is that tile kernel, timed
alone with CUDA events around each launch (activations prepared once before).
The fused 25,088x3072 GEMV is also timed as a single call over 8 rotating
weight copies (328 MB, so every launch reads DRAM).

`--impl reference` times the fp64 CPU oracle on the same workload (a bounded
sample of its matrices), in GB/s of the same algorithmic bytes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# one BLAS thread per process, set before numpy loads: the oracle baseline states the cores it uses,
# and its all-cores figure comes from one process per core
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

import synthetic  # noqa: E402

LAYERS = synthetic.LAYERS
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SRC = os.path.join(ROOT, "int4_weight_only_q4_gb300", "csrc", "q4_gemv.cu")
KERNEL_HDR = os.path.join(os.path.dirname(KERNEL_SRC), "q4_common.cuh")
FALLBACK_HBM_GBS = 6800.0


def algo_bytes(N: int, K: int, B: int) -> int:
    """Codes + fp16 scale and min + bf16 activations in + fp32 outputs."""
    return N * K // 2 + 4 * N * (K // 128) + 2 * B * K + 4 * B * N


def step_shapes():
    shapes = []
    for _ in range(LAYERS):
        for p in synthetic.LAYER_PROJS:
            N, K, _ = synthetic.SHAPES[p]
            shapes.append((N, K))
    N, K, _ = synthetic.SHAPES["head"]
    shapes.append((N, K))
    return shapes


def step_bytes(B: int) -> int:
    return sum(algo_bytes(N, K, B) for N, K in step_shapes()) + 4 * B  # + argmax indices


# ----------------------------------------------------------------------------- input generation
def _gen_packed(job):
    """Worker: one seeded matrix, packed by the library's host packer."""
    kind, layer, proj, seed = job
    sys.path.insert(0, ROOT)
    import synthetic as S
    from int4_weight_only_q4_gb300 import pack_host
    if kind == "layer":
        w, _ = S.decode_step_matrix(layer, proj, 1, seed)
    else:
        N, K, outl = S.SHAPES["head"]
        w, _ = S.weights(N, K, seed + 1000, outl)
    return pack_host(w, n_threads=2)


def step_jobs(seed: int):
    jobs = [("layer", l, p, seed) for l in range(LAYERS) for p in range(3)]
    jobs.append(("head", 0, 0, seed))
    return jobs


def step_activations(B: int, seed: int):
    """Activations of every matrix of the step, as bf16 bits [B, K]."""
    rng = np.random.default_rng(seed + 7919 * B)
    return [synthetic.f32_to_bf16_bits(rng.standard_normal((B, K), dtype=np.float32))
            for _, K in step_shapes()]


def generate_packed(seed: int, procs: int):
    ctx = mp.get_context("spawn")
    with ctx.Pool(procs) as pool:
        return pool.map(_gen_packed, step_jobs(seed), chunksize=1)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = max(smax, float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        loaded = [s for s in sm if s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- helpers
def measured_peak_gbs():
    try:
        d = json.load(open(PEAKS_FILE))
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def strip_comments(src: str) -> str:
    """C/C++/CUDA source without its comments and blank runs (string and character literals kept),
    so that the hash below changes with the code and not with its comments."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            i = src.find("*/", i + 2)
            i = n if i < 0 else i + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_src_sha() -> str:
    """Hash of the GEMV kernels' code (comments excluded): profiled counters stay valid until it
    changes."""
    h = hashlib.sha256()
    for f in (KERNEL_SRC, KERNEL_HDR):
        h.update(strip_comments(open(f, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if the kernel source is
    unchanged since it was taken; else None."""
    try:
        d = json.load(open(TRAFFIC_FILE))
    except (OSError, ValueError):
        return None
    if d.get("kernel_src_sha") != kernel_src_sha():
        return None
    return d.get("dram_bytes_per_launch", {}).get(kernel)


def dist_max(value: float, device=None) -> float:
    """Max of `value` over all ranks (the slowest rank sets the job's time); identity when not
    distributed.  gloo reduces a CPU tensor, nccl a tensor on `device`."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ----------------------------------------------------------------------------- the oracle arm
class OracleSampler:
    """Times the fp64 CPU oracle (dequantise-then-matvec) on a bounded sample of the step:
    row chunks of layer 0's three projections and of the head, in turn."""

    CHUNK = 512
    ROWS = 4096

    def __init__(self, B: int = 1, seed: int = 0, prepared=None, start: int = 0):
        import oracle
        self.oracle = oracle
        if prepared is None:
            ws = []
            for p in range(3):
                ws.append(np.ascontiguousarray(synthetic.decode_step_matrix(0, p, 1, seed)[0][:self.ROWS]))
            N, K, outl = synthetic.SHAPES["head"]
            ws.append(np.ascontiguousarray(synthetic.weights(N, K, seed + 1000, outl)[0][:self.ROWS]))
            # the oracle's own quantiser prepares its inputs (untimed): the first ROWS rows of each
            self.mats = [oracle.quantise_pack(w) for w in ws]
            del ws
            xs = step_activations(B, seed)
            self.xs = [xs[0], xs[1], xs[2], xs[-1]]
        else:
            self.mats, self.xs = prepared
        self.B = B
        # a worker of the all-cores run starts at its own row chunk and matrix
        self.pos = [(start * self.CHUNK) % self.ROWS] * 4
        self.m = start % 4

    def run(self, seconds: float):
        done, t_work, chunks = 0, 0.0, 0
        while t_work < seconds or chunks == 0:
            codes, sc, mn = self.mats[self.m]
            N, H = codes.shape
            K = 2 * H
            r0 = self.pos[self.m]
            rows = np.arange(r0, min(N, r0 + self.CHUNK))
            t0 = time.perf_counter()
            self.oracle.gemv_packed(codes, sc, mn, self.xs[self.m], rows=rows)
            t_work += time.perf_counter() - t0
            r = rows.size
            done += r * (K // 2 + 4 * (K // 128) + 4 * self.B) + 2 * self.B * K * r // N
            self.pos[self.m] = 0 if r0 + r >= N else r0 + r
            self.m = (self.m + 1) % len(self.mats)
            chunks += 1
        return done, t_work, chunks

    def describe(self, done, t_work, chunks):
        return (f"{chunks} chunks of {self.CHUNK} rows from the first {self.ROWS} rows of layer-0 "
                f"fused/o/down and the head, "
                f"fp64 dequantise + matvec, B={self.B}: {done / 1e6:.1f} MB algorithmic in {t_work:.2f} s")


def cpu_model() -> str:
    """The host CPU's model name (x86 /proc/cpuinfo "model name", else lscpu's "Model name")."""
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine() or "unknown"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


_SAMPLER = None


def _oracle_worker_init(prepared, B):
    global _SAMPLER
    _SAMPLER = (prepared, B)


def _oracle_worker(job):
    """One process of the all-cores oracle run: the oracle as it stands, one BLAS thread, on the same
    row-chunk sample, starting at its own chunk; returns (bytes, seconds of work, chunks)."""
    start, seconds = job
    prepared, B = _SAMPLER
    return OracleSampler(B, prepared=prepared, start=start).run(seconds)


def oracle_all_cores(sampler: "OracleSampler", seconds: float, procs: int):
    """The oracle on every host core at once: `procs` spawned processes, each timing the oracle on the
    sample for `seconds`; throughput = all processes' bytes / the wall time of the run."""
    ctx = mp.get_context("spawn")
    with ctx.Pool(procs, initializer=_oracle_worker_init, initargs=((sampler.mats, sampler.xs), sampler.B)) as pool:
        pool.map(_oracle_worker, [(i, 0.05) for i in range(procs)])      # start-up outside the timing
        t0 = time.perf_counter()
        res = pool.map(_oracle_worker, [(i, seconds) for i in range(procs)])
        wall = time.perf_counter() - t0
    done = sum(r[0] for r in res)
    chunks = sum(r[2] for r in res)
    return done, wall, chunks


def run_reference(args):
    ws, rank, _ = dist_setup()
    if rank != 0:
        return 0
    sampler = OracleSampler(1, args.seed)
    procs = host_cores()
    # each step times one bounded sample of the workload on every core; the whole run stays within
    # a few minutes
    budget = min(2.0, max(0.05, 120.0 / max(1, args.steps + args.warmup)))
    per_step, step_s, tot = [], [], [0, 0.0, 0]
    ctx = mp.get_context("spawn")
    with ctx.Pool(procs, initializer=_oracle_worker_init, initargs=((sampler.mats, sampler.xs), sampler.B)) as pool:
        pool.map(_oracle_worker, [(i, 0.05) for i in range(procs)])
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            res = pool.map(_oracle_worker, [(j + i * procs, budget) for j in range(procs)])
            wall = time.perf_counter() - t0
            done = sum(r[0] for r in res)
            if i >= args.warmup:
                per_step.append(done / wall / 1e9)
                step_s.append(wall)
                tot = [tot[0] + done, tot[1] + wall, tot[2] + sum(r[2] for r in res)]
    value = statistics.median(per_step) if per_step else None
    one = OracleSampler(1, args.seed, prepared=(sampler.mats, sampler.xs))
    d1, t1, c1 = one.run(min(5.0, 2 * budget))
    sample = (f"per step, on each of {procs} processes (one BLAS thread each), "
              f"{one.CHUNK}-row chunks from the first {one.ROWS} rows of layer-0 fused/o/down and the head, fp64 "
              f"dequantise + matvec, B=1; all steps: {tot[0] / 1e6:.1f} MB algorithmic in {tot[1]:.2f} s")
    line = {
        "impl": "reference", "metric": "int4 GEMV achieved HBM GB/s (decode step, B=1)", "value": value,
        "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.median(step_s), 3) if step_s else None,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(_config(1), step=("one bounded sample of the decode step's rows per step (the fp64 oracle "
                                         "is ~10^4x slower than the GPU path); ms_per_step is the sample's own "
                                         "wall time, value its throughput in the same algorithmic bytes")),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": procs, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": sample,
                         "one_core": {"value": round(d1 / t1 / 1e9, 4), "cores": 1, "sample": one.describe(d1, t1, c1)}},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def _config(B):
    return {"workload": "decode step: 36 x {fused qkv+gate+up 25088x3072, o-proj 3072x3072, down 3072x8192} "
                        "+ head 65536x3072 + argmax, int4 group-128 fp16 scale/min, one CUDA graph",
            "batch": B, "seed": 0,
            "l2": "inputs larger than L2 (2.24 GB of weights per step vs 129 MB L2); no flush",
            "parallelism": "replicas (one independent step per GPU)"}


# ----------------------------------------------------------------------------- our arm
def run_ours(args):
    world, rank, local = dist_setup()
    if args.gpus > 1 and world == 1:
        print(json.dumps({"error": "launch with torchrun for --gpus > 1"}))
        return 2
    # CPU work that needs no GPU first (spawned pool: no CUDA state to inherit)
    procs = max(1, min(16, (os.cpu_count() or 2)))
    t0 = time.time()
    packed = generate_packed(args.seed, procs)
    gen_s = time.time() - t0

    import torch
    import int4_weight_only_q4_gb300 as q4
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    shapes = step_shapes()
    mats = [q4.QuantizedMatrix.from_packed(*p, device=dev) for p in packed]
    head_i = len(mats) - 1

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    graphs = {}
    for B in (1, 8):
        xs = step_activations(B, args.seed)
        g = q4.DecodeStepGraph(mats, B, device=dev, with_argmax_of=head_i)
        for i, x in enumerate(xs):
            g.X[i].copy_(bf16(x))
        graphs[B] = (g, xs)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def time_graph(g, steps, warmup):
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(steps):
            g.replay()
        e.record()
        torch.cuda.synchronize()
        barrier()
        return s.elapsed_time(e) / steps  # ms

    g1, xs1 = graphs[1]
    with ClockSampler(dev.index) as clk:
        ms1 = time_graph(g1, args.steps, args.warmup)
        # keep the GPU busy long enough for the clock sampler to see the load
        t_end = time.time() + 1.0
        while time.time() < t_end:
            time_graph(g1, 200, 0)
    clocks = clk.summary()
    ms1 = dist_max(ms1, dev)
    ms8 = time_graph(graphs[8][0], max(20, args.steps // 4), max(3, args.warmup))
    sb1 = step_bytes(1)
    value = sb1 * world / (ms1 * 1e-3) / 1e9

    # decode step alone (108 projections, no head), batch 1 and 8: the metric's step time; the
    # same step as 108 dependency-safe launches (one per matrix) for comparison
    dec_us, chained_us = {}, {}
    for B in (1, 8):
        for indep, out in ((True, dec_us), (False, chained_us)):
            gd = q4.DecodeStepGraph(mats[:head_i], B, device=dev, independent=indep)
            for i, x in enumerate(graphs[B][1][:head_i]):
                gd.X[i].copy_(bf16(x))
            out[f"b{B}"] = round(1e3 * time_graph(gd, max(50, args.steps // 4), max(3, args.warmup)), 2)
            del gd

    # dominant kernel: the step's persistent tile kernel, events around every launch
    roof = step_roofline(q4, torch, mats, graphs[1][0], dev, args, ms1 * 1e3)
    # the fused 25,088x3072 projection: single calls, and sustained over the step's 36 copies
    fused_single = fused_single_call(q4, torch, mats[0], dev, args)
    fused_sus = fused_sustained(q4, torch, mats, dev, args)
    # the int8 output head with the argmax fused in
    head8 = int8_head(q4, torch, dev, args)
    samp = sampler_bench(q4, torch, dev, args)
    prefill = prefill_bench(q4, torch, mats, dev, args)
    attn = attention_bench(q4, torch, dev, args)

    # end to end through the public API with pinned host buffers
    e2e = end_to_end(q4, torch, g1, xs1, dev, max(10, args.steps // 20), barrier)

    peak, src = measured_peak_gbs()
    launches_per_step = 2 * ((len(mats) + 127) // 128) + 1  # prep + tile kernel per 128 matrices, argmax
    line = {
        "metric": "int4 GEMV achieved HBM GB/s (decode step, B=1)", "value": round(value, 1), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms1, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int4*bf16->f32",
        "data": "synthetic", "config": _config(1), "clocks": clocks,
        "frac_of_hbm_peak": round(value / world / peak, 4), "peak_source": src,
        "decode_step_us": dec_us, "decode_step_chained_launches_us": chained_us, "step_with_head_us": {"b1": round(ms1 * 1e3, 2), "b8": round(ms8 * 1e3, 2)},
        "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "roofline": roof, "fused_projection_sustained": fused_sus, "fused_gemv_single_call": fused_single,
        "int8_head_65536x3072": head8, "sampler_topk_gumbel": samp, "prefill_gemm": prefill,
        "flash_decoding_attention": attn,
        "gen_seconds": round(gen_s, 1),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sampler = OracleSampler(1, args.seed)
        done, t, c = sampler.run(args.cpu_seconds)
        procs = host_cores()
        da, ta, ca = oracle_all_cores(sampler, max(2.0, args.cpu_seconds / 2), procs)
        line["cpu_baseline"] = {"value": round(done / t / 1e9, 4), "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "cpu_model": cpu_model(), "sample": sampler.describe(done, t, c),
                                "all_cores": {"value": round(da / ta / 1e9, 4), "unit": "GB/s", "cores": procs,
                                              "sample": f"{procs} processes (one BLAS thread each) on the same "
                                                        f"sample: {ca} chunks, {da / 1e6:.1f} MB in {ta:.2f} s"}}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def graph_us(torch, enqueue, calls: int, replays: int, warmup: int = 3) -> float:
    """Microseconds per call of `enqueue(stream)`: `calls` calls captured in one CUDA graph (no host
    work between launches), replayed `replays` times between CUDA events on the replaying stream."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        enqueue(side)                      # first call outside capture (kernel attributes)
        side.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for _ in range(calls):
                enqueue(side)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return 1e3 * e0.elapsed_time(e1) / (replays * calls)


def step_roofline(q4, torch, mats, g, dev, args, step_us):
    """The step's tile kernel (all 109 matrices, B=1) alone: activations prepared once, then 10
    q4_step_stream launches per CUDA graph, timed over graph replays (the same launches the step
    graph holds, without its prep and argmax).  Beside it the read-only twin of the same launch
    (q4_step_stream_readonly: the same loads and stores, no arithmetic), the practical ceiling of
    the access pattern."""
    ws = q4.Workspace(q4.step_workspace_bytes([m.K for m in mats], 1))
    q4.step_prepare(mats, g.X, ws)
    torch.cuda.synchronize()
    reps = max(5, args.steps // 100)
    us = graph_us(torch, lambda st: q4.step_stream(mats, g.Y, 1, ws, stream=st), 10, reps)
    twin_us = graph_us(torch, lambda st: q4.step_stream_readonly(mats, g.Y, 1, ws, stream=st), 10, reps)
    bytes_launch = sum(algo_bytes(N, K, 1) for N, K in step_shapes())
    achieved = bytes_launch / (us * 1e-6) / 1e9
    twin = bytes_launch / (twin_us * 1e-6) / 1e9
    peak, src = measured_peak_gbs()
    return {"bound": "hbm", "kernel": "q4_tiles_ring_kernel (109 matrices of the step, B=1, one launch)",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic("q4_tiles_ring_kernel"), "algorithmic_bytes_per_launch": bytes_launch,
            "avg_launch_us": round(us, 2), "timing": f"10 launches per CUDA graph, {reps} replays",
            "kernel_within_step": bool(us <= step_us), "step_us": round(step_us, 2),
            "read_only_twin": {"kernel": "q4_tiles_ring_kernel<32, 4, 1, RO> (q4_step_stream_readonly)",
                               "avg_launch_us": round(twin_us, 2), "GB/s": round(twin, 1),
                               "frac_of_peak": round(twin / peak, 4)},
            "frac_of_twin": round(twin_us / us, 4),
            "peak_source": src}


def fused_single_call(q4, torch, W0, dev, args):
    """The fused 25,088x3072 projection as single q4_gemm_skinny calls (B=1 and B=8): 8 calls on 8
    rotating weight copies (328 MB, more than L2) captured in one CUDA graph, so that host launch
    cost stays out; microseconds per call = graph time / 8."""
    copies = [q4.QuantizedMatrix(W0.codes.clone(), W0.scales.clone(), W0.mins.clone(), W0.N, W0.K).build_tiled()
              for _ in range(8)]
    out = {}
    for B in (1, 8):
        x = torch.randn((B, W0.K), device=dev).to(torch.bfloat16)
        y = torch.empty((B, W0.N), dtype=torch.float32, device=dev)
        ws = q4.Workspace(q4.workspace_bytes(W0.N, W0.K, B), dev)
        side = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(side):
            for c in copies:
                q4.gemm_skinny(c, x, y, workspace=ws, stream=side)
            side.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for c in copies:
                    q4.gemm_skinny(c, x, y, workspace=ws, stream=side)
        for _ in range(5):
            g.replay()
        n = max(20, args.steps // 40)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / (n * len(copies))
        out[f"b{B}"] = {"us_per_call": round(us, 3), "GB/s": round(algo_bytes(W0.N, W0.K, B) / (us * 1e-6) / 1e9, 1)}
    peak, src = measured_peak_gbs()
    info = q4.plan(W0.N, W0.K)
    kname = {0: "q4_direct_kernel", 6: "q4_flat_kernel"}.get(info["kernel"], f"kernel {info['kernel']}")
    return {"kernel": f"{kname} (one launch per call, 8 calls per CUDA graph)", **out,
            "frac_b1": round(out["b1"]["GB/s"] / peak, 4), "peak": peak, "peak_source": src,
            "algorithmic_bytes_per_call_b1": algo_bytes(W0.N, W0.K, 1)}


def fused_sustained(q4, torch, mats, dev, args):
    """The step's 36 fused 25,088x3072 projections as one independent list (one tile-kernel launch),
    B=1: activations prepared once, 10 q4_step_stream launches per CUDA graph, timed over replays."""
    fused = [m for m in mats if (m.N, m.K) == (25088, 3072)]
    X = [torch.randn((1, m.K), device=dev).to(torch.bfloat16) for m in fused]
    Y = [torch.empty((1, m.N), device=dev) for m in fused]
    ws = q4.Workspace(q4.step_workspace_bytes([m.K for m in fused], 1), dev)
    q4.step_prepare(fused, X, ws)
    torch.cuda.synchronize()
    us = graph_us(torch, lambda st: q4.step_stream(fused, Y, 1, ws, stream=st), 10, max(5, args.steps // 100))
    byts = sum(algo_bytes(m.N, m.K, 1) for m in fused)
    achieved = byts / (us * 1e-6) / 1e9
    peak, src = measured_peak_gbs()
    return {"kernel": f"q4_tiles_ring_kernel ({len(fused)} fused 25088x3072 projections, B=1, one launch)",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "us_per_projection": round(us / len(fused), 3), "avg_launch_us": round(us, 2),
            "algorithmic_bytes_per_launch": byts, "peak_source": src}


def int8_head(q4, torch, dev, args):
    """The int8 output head (65,536 x 3072, per-row fp16 scales) with its argmax fused into the same
    launch: 8 calls on 8 rotating copies in one CUDA graph, microseconds per call, B=1 and B=8,
    logits + argmax and argmax only."""
    N, K, _ = synthetic.SHAPES["head"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed + 555)
    heads = []
    for i in range(8):  # seeded random codes and scales on the device (timing only)
        codes = torch.randint(-127, 128, (N, K), dtype=torch.int8, device=dev, generator=gen)
        sc = (torch.rand((N,), device=dev, generator=gen) * 1e-3 + 1e-4).half()
        heads.append(q4.Int8Head.from_device(codes, sc))
    out = {}
    for B in (1, 8):
        X = torch.randn((B, K), device=dev).to(torch.bfloat16)
        Y = torch.empty((B, N), device=dev)
        idx = torch.empty((B,), dtype=torch.int32, device=dev)
        ws = heads[0].workspace(B, dev)
        for logits in (True, False):
            side = torch.cuda.Stream(device=dev)
            with torch.cuda.stream(side):
                for H in heads:
                    H(X, Y, idx, logits=logits, workspace=ws, stream=side)
                side.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    for H in heads:
                        H(X, Y, idx, logits=logits, workspace=ws, stream=side)
            for _ in range(5):
                g.replay()
            n = max(20, args.steps // 40)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            us = 1e3 * e0.elapsed_time(e1) / (n * len(heads))
            byts = N * K + 2 * N + 2 * B * K + (4 * B * N if logits else 0) + 4 * B
            out[f"b{B}_{'logits_argmax' if logits else 'argmax_only'}"] = {
                "us_per_call": round(us, 3), "GB/s": round(byts / (us * 1e-6) / 1e9, 1)}
    peak, src = measured_peak_gbs()
    out["frac_b1_argmax_only"] = round(out["b1_argmax_only"]["GB/s"] / peak, 4)
    out["kernel"] = "q4_flat_kernel<16, 4, BT, true, true> + q8_argmax_final (8 calls per CUDA graph)"
    return out


def sampler_bench(q4, torch, dev, args):
    """Top-k (k = 50) Gumbel-max sampling over 65,536 logits per row (q4_sample_topk), B = 1 and 8:
    20 calls per CUDA graph, microseconds per call."""
    N = synthetic.SHAPES["head"][0]
    out = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed + 777)
    for B in (1, 8):
        Y = torch.randn((B, N), device=dev, generator=gen) * 3
        u = torch.rand((B, 50), device=dev, generator=gen).clamp_(1e-12, 1 - 1e-7)
        noise = -torch.log(-torch.log(u))
        tok = torch.empty((B,), dtype=torch.int32, device=dev)
        side = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(side):
            q4.sample_topk(Y, 50, 1.25, noise, token=tok, stream=side)
            side.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for _ in range(20):
                    q4.sample_topk(Y, 50, 1.25, noise, token=tok, stream=side)
        for _ in range(3):
            g.replay()
        n = max(10, args.steps // 100)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        out[f"b{B}_us_per_call"] = round(1e3 * e0.elapsed_time(e1) / (n * 20), 3)
    out["kernel"] = "q4_sample_cluster_kernel (a cluster of 8 CTAs per row; k = 50, N = 65,536)"
    return out


def prefill_bench(q4, torch, mats, dev, args):
    """The int4 prefill GEMM (q4_gemm_prefill) on the step's fused 25,088 x 3072 projection for
    prompts of 128 and 512 tokens: microseconds per call (5 per CUDA graph) and TFLOP/s."""
    W = next(m for m in mats if (m.N, m.K) == (25088, 3072))
    out = {}
    peak = json.load(open(PEAKS_FILE)).get("bf16_tflops") if os.path.exists(PEAKS_FILE) else None
    kinds = {}
    for M in (128, 512):
        kinds[M] = q4.prefill_kernel(W.K, M)
        X = torch.randn((M, W.K), device=dev).to(torch.bfloat16)
        Y = torch.empty((M, W.N), device=dev)
        ws = q4.Workspace(int(q4.lib.q4_prefill_workspace_bytes(W.K, M)), dev)
        side = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(side):
            q4.gemm_prefill(W, X, Y, ws, stream=side)
            side.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for _ in range(5):
                    q4.gemm_prefill(W, X, Y, ws, stream=side)
        for _ in range(3):
            g.replay()
        n = max(10, args.steps // 100)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / (n * 5)
        tf = 2 * M * W.N * W.K / (us * 1e-6) / 1e12
        out[f"m{M}"] = {"us_per_call": round(us, 2), "TFLOP/s": round(tf, 1),
                        "frac_of_bf16_peak": round(tf / peak, 4) if peak else None}
    names = {"tcgen05": "q4_tc_prep_kernel + q4_prefill_tc_kernel (tcgen05.mma 128x128x16 bf16, TMEM "
                        "accumulators, TMA activations; fused 25088x3072)",
             "mma.sync": "q4_xprep_kernel + q4_prefill_kernel (mma.sync m16n8k16 bf16, fused 25088x3072)"}
    out["kernel"] = "; ".join(sorted({f"M={m}: {names[k]}" for m, k in kinds.items()}))
    out["bound"] = "tensor"
    out["peak_source"] = "measured bf16 burst (MEASURED_PEAKS.json bf16_tflops)"
    return out


def attention_bench(q4, torch, dev, args):
    """Flash-decoding attention (q4_flash_decode): 24 query heads sharing 6 KV heads, head_dim 128.
    The page's case -- batch 1 over a 2,000-position cache -- as one call per layer for 36 layers
    (36 distinct caches, 221 MB, so nothing stays in L2) in one CUDA graph; and a long cache,
    batch 8 over 8,192 positions (2 layers, 403 MB).  Microseconds per call and GB/s of
    algorithmic bytes (keys, values, queries, outputs)."""
    Hq, Hkv, D = 24, 6, 128
    peak, src = measured_peak_gbs()
    out = {"heads": f"{Hq} query / {Hkv} KV heads, head_dim {D}", "chunk_capacity_per_kv_head": int(q4.lib.q4_flash_decode_chunks(Hkv, 0)),
           "chunks_in_use": "at most ceil(max_len / 32) per KV head (63 for the page's 2,000 positions)"}
    for name, B, L, layers, C in (("page_b1_2000", 1, 2000, 36, 0), ("page_b1_2000_16chunks", 1, 2000, 36, 16),
                                  ("long_b8_8192", 8, 8192, 2, 0)):
        g = torch.Generator(device=dev).manual_seed(args.seed)
        Qs = [torch.randn((B, Hq, D), device=dev, generator=g).to(torch.bfloat16) for _ in range(layers)]
        Ks = [torch.randn((B, Hkv, L, D), device=dev, generator=g).to(torch.bfloat16) for _ in range(layers)]
        Vs = [torch.randn((B, Hkv, L, D), device=dev, generator=g).to(torch.bfloat16) for _ in range(layers)]
        lens = torch.full((B,), L, dtype=torch.int32, device=dev)
        O = torch.empty((B, Hq, D), device=dev)
        ws = q4.flash_decode_workspace(B, Hq, Hkv, D, C, dev)
        reps = max(1, 36 // layers)
        side = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(side):
            for i in range(layers):
                q4.flash_decode(Qs[i], Ks[i], Vs[i], lens, O, n_chunks=C, workspace=ws, stream=side)
            side.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                for _ in range(reps):
                    for i in range(layers):
                        q4.flash_decode(Qs[i], Ks[i], Vs[i], lens, O, n_chunks=C, workspace=ws, stream=side)
        for _ in range(max(3, args.warmup)):
            graph.replay()
        n = max(10, args.steps // 100)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / (n * reps * layers)
        nbytes = 2 * B * Hkv * L * D * 2 + B * Hq * D * (2 + 4)
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"us_per_call": round(us, 2), "GB/s": round(gbs, 1), "frac_of_hbm_peak": round(gbs / peak, 4),
                     "algorithmic_bytes": nbytes}
        del Qs, Ks, Vs, graph
    out["kernel"] = "q4_flash_split_kernel<128, 3> + q4_flash_combine_kernel<128> (per call)"
    out["bound"] = "hbm"
    out["peak_source"] = src
    return out


def end_to_end(q4, torch, g, xs, dev, steps, barrier):
    """Per step through the public API: the step's activations host->device (one pinned buffer laid
    out like the graph's activation buffer), graph replay, the step's result (the head's argmax
    token per batch row) device->host, and a wait for it."""
    flat = np.concatenate([np.ascontiguousarray(x).reshape(-1) for x in xs]).view(np.int16)
    hx = torch.from_numpy(flat).view(torch.bfloat16).pin_memory()
    hidx = torch.empty(g.idx.shape, dtype=g.idx.dtype).pin_memory()
    bi = hx.numel() * hx.element_size()
    bo = hidx.numel() * hidx.element_size()
    for _ in range(3):
        g.run_host(hx, None, hidx)
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        g.run_host(hx, None, hidx)
    dt = (time.perf_counter() - t0) / steps
    value = step_bytes(g.B) / dt / 1e9
    return {"value": round(value, 1), "unit": "GB/s", "ms_per_step": round(dt * 1e3, 4),
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}


def run_profile_case(args) -> int:
    """A small case for ncu: `layers` decode layers + the head with seeded random codes in the tiled
    layout, activations prepared once, then five step_stream launches and one argmax (no timing)."""
    import torch
    import int4_weight_only_q4_gb300 as q4
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed)
    B = args.profile_batch
    shapes = [sh for sh in step_shapes()[:3 * args.profile_step]] + [step_shapes()[-1]]
    mats = []
    for N, K in shapes:
        codes = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev, generator=gen)
        sc = (torch.rand((N, K // 128), device=dev, generator=gen) * 0.01 + 1e-3).half()
        mn = (torch.rand((N, K // 128), device=dev, generator=gen) * -0.05).half()
        W = q4.QuantizedMatrix(codes, sc, mn, N, K).build_tiled()
        W.codes = W.scales = W.mins = None
        mats.append(W)
    X = [torch.randn((B, K), device=dev, generator=gen).to(torch.bfloat16) for _, K in shapes]
    Y = [torch.empty((B, N), device=dev) for N, _ in shapes]
    ws = q4.Workspace(q4.step_workspace_bytes([K for _, K in shapes], B))
    q4.step_prepare(mats, X, ws)
    for _ in range(5):
        q4.step_stream(mats, Y, B, ws)
    q4.argmax(Y[-1])
    torch.cuda.synchronize()
    q4.device_status()
    print(json.dumps({"profile_case": f"{args.profile_step} layers + head", "B": B, "matrices": len(shapes),
                      "algorithmic_bytes_per_stream_launch": sum(algo_bytes(N, K, B) for N, K in shapes)}))
    return 0


def run_profile_small(args) -> int:
    """Small cases for ncu: `--profile-head8` one int8-head call (65,536 x 3072, seeded random codes on
    the device, B = --profile-batch, logits + argmax) after two warm-up calls; `--profile-sampler`
    one top-k (k = 50) Gumbel-max sampling call over 65,536 logits after two warm-up calls;
    `--profile-attn` three flash-decoding calls, batch --profile-batch over an 8,192-position cache;
    `--profile-prefill M` three prefill GEMM calls of M tokens on a 25,088 x 3072 matrix with seeded
    random codes (the fused projection's shape)."""
    import torch
    import int4_weight_only_q4_gb300 as q4
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed)
    B = args.profile_batch
    N, K, _ = synthetic.SHAPES["head"]
    if args.profile_head8:
        H = q4.Int8Head.from_device(torch.randint(-127, 128, (N, K), dtype=torch.int8, device=dev, generator=gen),
                                    (torch.rand((N,), device=dev, generator=gen) * 1e-3 + 1e-4).half())
        X = torch.randn((B, K), device=dev, generator=gen).to(torch.bfloat16)
        for _ in range(3):
            Y, idx = H(X)
    elif args.profile_prefill:
        Np, Kp, _ = synthetic.SHAPES["fused"]
        W = q4.QuantizedMatrix(torch.randint(0, 256, (Np, Kp // 2), dtype=torch.uint8, device=dev, generator=gen),
                               (torch.rand((Np, Kp // 128), device=dev, generator=gen) * 0.01 + 1e-3).half(),
                               (torch.rand((Np, Kp // 128), device=dev, generator=gen) * -0.05).half(), Np, Kp)
        W.build_tiled()
        X = torch.randn((args.profile_prefill, Kp), device=dev, generator=gen).to(torch.bfloat16)
        for _ in range(3):
            Y = q4.gemm_prefill(W, X)
        idx = [float(Y.abs().mean()), q4.prefill_kernel(Kp, args.profile_prefill)]
    elif args.profile_sampler:
        Y = torch.randn((B, N), device=dev, generator=gen) * 3
        noise = torch.zeros((B, 50), device=dev)
        for _ in range(3):
            idx = q4.sample_topk(Y, 50, 1.0, noise)
    else:  # attention: batch --profile-batch over an 8,192-position cache (24 / 6 heads, head_dim 128)
        L = 8192
        Q = torch.randn((B, 24, 128), device=dev, generator=gen).to(torch.bfloat16)
        Kc = torch.randn((B, 6, L, 128), device=dev, generator=gen).to(torch.bfloat16)
        Vc = torch.randn((B, 6, L, 128), device=dev, generator=gen).to(torch.bfloat16)
        lens = torch.full((B,), L, dtype=torch.int32, device=dev)
        for _ in range(3):
            O = q4.flash_decode(Q, Kc, Vc, lens)
        idx = [float(O.abs().mean())]
    torch.cuda.synchronize()
    q4.device_status()
    case = ("int8 head" if args.profile_head8 else "sampler" if args.profile_sampler
            else "prefill" if args.profile_prefill else "attention")
    print(json.dumps({"profile_case": case, "B": B, "idx": idx if isinstance(idx, list) else idx.cpu().tolist()}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-step", type=int, default=0,
                    help="run only a small profiling case of this many layers + the head, then exit")
    ap.add_argument("--profile-batch", type=int, default=1)
    ap.add_argument("--profile-head8", action="store_true", help="run only a small int8-head case for ncu")
    ap.add_argument("--profile-sampler", action="store_true", help="run only a small sampler case for ncu")
    ap.add_argument("--profile-attn", action="store_true", help="run only a flash-decoding attention case for ncu")
    ap.add_argument("--profile-prefill", type=int, default=0, help="run only a prefill GEMM case of this many tokens")
    args = ap.parse_args()
    if args.profile_step > 0:
        return run_profile_case(args)
    if args.profile_head8 or args.profile_sampler or args.profile_attn or args.profile_prefill:
        return run_profile_small(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
