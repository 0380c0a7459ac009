"""Benchmark of the multi-LoRA delta step (one JSON line on stdout, rank 0).

A step is one pass of the whole hot path over one batch: the scheduler step that
groups the batch by adapter, then the delta kernel over every (layer, projection)
of the model, in one C-ABI call.  Default workload: Llama-7B-shaped decode BGMV,
h=4096, 32 layers x q/k/v/o, 64 one-token requests, 2,000 resident adapters with
ranks in {8,16,32,64}, adapter ids Zipf(1.0).  Synthetic, seeded inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config C]

--impl reference times the fp64 CPU oracle (the reference arm of this project) on
the host cores, on a bounded sample of the same workload.  Under torchrun (N > 1)
every rank runs an independent replica (tokens shard with no collective on the
data path); rank 0 prints the whole-job aggregate.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LoRA-delta tokens/s (BGMV decode, SGMV prefill); % of HBM roofline"
UNIT = "tokens/s"


# ----------------------------------------------------------------------------- helpers

def workload_for(name: str):
    """A named workload of the workload module, or a small variant of one for profiler
    captures: "decode-small" (4 layers, 300 adapters, ~2.4 GB pool), "decode-l12" (12 layers,
    100 adapters, ~2.4 GB: enough projections per launch for a sweep), "stress-distinct-small"
    and "stress-zipf-small" (the unified-pool stress shape at 8 layers, 500 adapters, a 2^18-page
    pool of one-layer slices), "prefill-small" (2
    layers x 2 projections, ~2 GB on the device), "mixed-small" (1 layer x 2 projections),
    "llama3-decode-small" and "llama3-prefill-small" (1 layer)."""
    from workloads import spec
    if name == "decode-small":
        return spec.decode_workload("llama7b-decode-bgmv-h4096-t64-a300-l4", 1001, 4096, 4, 4,
                                    300, [8, 16, 32, 64], 64, 1.0)
    if name == "decode-l12":
        return spec.decode_workload("llama7b-decode-bgmv-h4096-t64-a100-l12", 1001, 4096, 12, 4,
                                    100, [8, 16, 32, 64], 64, 1.0)
    if name in ("stress-distinct-small", "stress-zipf-small"):
        v = name.split("-")[1]
        return spec.decode_workload(f"unified-pool-stress-{v}-h4096-t256-a500-l8", 1004 if v == "distinct" else 1014,
                                    4096, 8, 4, 500, [8, 16, 32, 64], 256, 1.2 if v == "zipf" else None,
                                    num_pages=1 << 18, distinct=(v == "distinct"), layer_slices=True)
    if name == "prefill-small":
        return spec.prefill_workload("llama7b-prefill-sgmv-h4096-s32-a1000-l2p2", 1002, 4096, 2, 2,
                                     1000, [8, 16, 32, 64], 32, 64, 1024, 1.0)
    if name == "mixed-small":
        return spec.mixed_workload("13b-mixed-h5120-p8-d192-a2000-l1p2", 1003, 5120, 1, 2, 2000,
                                   [8, 16, 32, 64, 128], 8, 128, 2048, 192, 20, 0.8,
                                   pool_pages=1 << 18)
    if name == "llama3-decode-small":
        return spec.llama3_8b_decode(layers=1)
    if name == "llama3-prefill-small":
        return spec.llama3_8b_prefill(layers=1)
    if name not in spec.WORKLOADS:
        raise SystemExit(f"unknown workload {name!r}; choose from {sorted(spec.WORKLOADS)} or a "
                         "-small variant")
    return spec.WORKLOADS[name]()


def cpu_model() -> str:
    """The host CPU's model name as lscpu reports it (architecture if unavailable)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip() + f" ({platform.machine()})"
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


KERNEL_SOURCES = {   # the kernel's code and the launch file that picks its instantiation
    "bgmv_ring_kernel": ["bgmv_ring.cuh", "common.cuh", "ptx.cuh", "launch_ring.cu"],
    "sgmv_mma_kernel": ["sgmv_mma.cuh", "common.cuh", "ptx.cuh", "launch_tile.cu"],
    "delta_fused_kernel": ["fused.cuh", "bgmv_ring.cuh", "sgmv_mma.cuh", "common.cuh", "ptx.cuh", "launch_tile.cu"],
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the code of the source files a kernel is built from, comments and
    whitespace removed (traffic figures taken on other code are not reused)."""
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        src = open(os.path.join(ROOT, "heterogeneous_adapters_gb300", "csrc", f)).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str, units_per_launch: float):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, scaled to this
    launch by units processed; None when absent or taken on other kernel sources."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    src = kernel_source_hash(kernel)
    for line in open(p):
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if f.get("kernel") == kernel and f.get("workload") == workload and f.get("src") == src:
            return float(f["dram_bytes"]) / float(f["units"]) * units_per_launch
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out = ""

    def summary(self) -> dict:
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for line in (self.out or "").strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 6:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus: int):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("LORA_BENCH_BACKEND", "nccl")
        dist.init_process_group(backend)
    return rank, world, local


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (the job ends when its slowest rank ends)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_step: float, steps: int, world: int, elapsed_local: float):
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    elapsed = max_over_ranks(elapsed_local, world)
    return units_per_step * steps * world / elapsed, elapsed


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- oracle arm

class OracleRunner:
    """The fp64 CPU oracle, as it stands, on the workload's first `n_prep` projections
    (inputs regenerated on the host once; only the oracle calls are timed)."""

    def __init__(self, wl, n_prep: int):
        from workloads import valuegen as vg
        from workloads.materialize import host_inputs
        self.wl = wl
        self.probs = wl.problems[:max(1, min(n_prep, len(wl.problems)))]
        self.hi = host_inputs(wl, problems=self.probs)
        self.y0 = {k: vg.bf16_bits_to_f64(v) for k, v in self.hi.y0.items()}
        self.ids = wl.batch.token_adapter()
        self.next = 0
        self.threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))

    def run(self, n: int) -> float:
        """Seconds spent by the oracle on n projections (cycling through the prepared ones)."""
        import oracle
        pool = self.wl.pool
        t0 = time.perf_counter()
        for _ in range(n):
            l, p = self.probs[self.next % len(self.probs)]
            self.next += 1
            oracle.lora_delta(self.hi.pool, self.hi.pt, pool.pt_off, pool.ranks, pool.scales,
                              pool.num_layers, pool.num_proj, l, p, self.hi.x[(l, p)],
                              self.y0[(l, p)], self.ids, proj_dims=pool.proj_dims)
        return time.perf_counter() - t0

    def rate(self, seconds: float, n_problems: int) -> float:
        """tokens/s of the whole step, extrapolated from n_problems projections."""
        adapted = int((self.ids >= 0).sum())
        return adapted / (seconds / n_problems * len(self.wl.problems))

    def single_thread_sample(self, budget_s: float):
        """timed_sample with the oracle's OpenMP team cut to one thread (restored after);
        None where the OpenMP runtime cannot be reached."""
        import ctypes
        try:
            gomp = ctypes.CDLL("libgomp.so.1")
        except OSError:
            return None
        before = gomp.omp_get_max_threads()
        gomp.omp_set_num_threads(1)
        try:
            return self.timed_sample(budget_s)
        finally:
            gomp.omp_set_num_threads(before)

    def timed_sample(self, budget_s: float):
        """Time as many projections as fit in about budget_s seconds of wall time (more
        than one step's worth when a step is quicker than that, up to 64 steps)."""
        one = self.run(1)
        n = max(1, min(64 * len(self.wl.problems), int(budget_s / max(one, 1e-6))))
        dt = self.run(n)
        return self.rate(dt, n), dt, n


def selected_workload(args):
    """The workload of --config, with q, k and v reading one x per layer under --shared-x."""
    import dataclasses
    wl = workload_for(args.config)
    if args.shared_x:
        wl = dataclasses.replace(wl, shared_x=True, name=wl.name + "-shared-x")
    return wl


def tuning_args(args) -> dict:
    """--tuning k=v,k=v: lora_pool_set_tuning fields (kernel choice and stage shapes)."""
    out = {}
    for kv in filter(None, (args.tuning or "").split(",")):
        k, v = kv.split("=")
        out[k.strip()] = float(v) if k.strip() == "fused_ring_speed" else int(v)
    return out


def apply_tuning(pool, args):
    t = tuning_args(args)
    if t:
        pool.set_tuning(**t)


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    wl = selected_workload(args)
    runner = OracleRunner(wl, args.ref_problems)
    one = runner.run(1)
    for _ in range(args.warmup):
        runner.run(1)
    per_step_budget = args.ref_budget_s / max(1, args.steps + args.warmup)
    n = max(1, min(len(wl.problems), int(per_step_budget / max(one, 1e-6))))
    t0 = time.perf_counter()
    secs = [runner.run(n) for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    value = runner.rate(statistics.mean(secs), n)
    sample = (f"{n} of {len(wl.problems)} projections of one step per timed step (all "
              f"{wl.batch.num_tokens} tokens), extrapolated linearly to the full step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.mean(secs) / n * len(wl.problems),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(wl, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": runner.threads,
                             "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

def graph_timing(capture_fn, tokens_step: int, dev, replays: int) -> dict:
    """Capture capture_fn(stream handle) once in a CUDA graph, replay it 10 times untimed,
    then `replays` times, each between two events; median and p10 / p90 in ms."""
    import torch
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=cap):
        capture_fn(cap.cuda_stream)
    for _ in range(10):
        g.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(replays)]
    for e0, e1 in ev:
        e0.record(cur)
        g.replay()
        e1.record(cur)
    torch.cuda.synchronize()
    ms = np.array([e0.elapsed_time(e1) for e0, e1 in ev])
    med = float(np.median(ms))
    return {"ms_median": med, "ms_p10": float(np.percentile(ms, 10)),
            "ms_p90": float(np.percentile(ms, 90)), "replays": replays,
            "tokens_per_s": tokens_step / (med / 1e3)}


def step_model(wl, ids=None, problems=None) -> dict:
    """Algorithmic bytes and flops of one launch over the given problems (all of the
    workload's by default): each projection at its own widths, each distinct x buffer
    read once, each distinct physical page once (pools whose layers share a slice of
    pages read those pages once per launch from DRAM)."""
    from heterogeneous_adapters_gb300 import costmodel
    p = wl.pool
    problems = wl.problems if problems is None else problems
    ids = wl.batch.token_adapter() if ids is None else ids
    dims = [p.dims(pj) for (_, pj) in problems]
    x_widths = [p.dims(pj)[0] for (_, pj) in {wl.x_source(l, pj) for (l, pj) in problems}]
    U, pre, _, _ = p.layout_units()
    blocks = [(l * U + pre[pj],) + p.dims(pj) for (l, pj) in problems]
    phys, _ = costmodel.physical_page_bytes(p.pt, p.pt_off, p.ranks, ids, p.h, blocks)
    return costmodel.decode_step_bytes(p.ranks, ids, p.h, len(problems), dims=dims,
                                       x_widths=x_widths, page_bytes_physical=phys)


def config_dict(wl, args) -> dict:
    p = wl.pool
    m = step_model(wl)
    return {"workload": wl.name, "h": p.h, "layers": p.num_layers, "projections": p.num_proj,
            "tokens": wl.batch.num_tokens, "adapted_tokens": m["adapted_tokens"],
            "adapters": p.num_adapters, "distinct_adapters": m["distinct_adapters"],
            "ranks": sorted(set(int(r) for r in np.unique(p.ranks))), "batch": wl.batch.kind,
            "seed": wl.seed, "shared_x": wl.shared_x, "bytes_per_step": m["bytes"],
            "page_bytes_per_step": m["page_bytes"],
            "page_bytes_logical_per_step": m["page_bytes_logical"],
            "l2": "inputs larger than L2: every step streams %.2f GB" % (m["bytes"] / 1e9),
            "parallelism": "replicas (weak scaling, no collective)"}


def run_ours(args, rank: int, world: int, local: int):
    import torch

    import heterogeneous_adapters_gb300 as lora
    from workloads.materialize import device_inputs

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    wl = selected_workload(args)
    d = device_inputs(wl, device=dev, nan_dummies=False)
    p = wl.pool
    pool = lora.Pool(d.pool, p.num_pages, p.h, d.pt, p.pt.size, d.pt_off, d.ranks, d.scales,
                     p.num_adapters, p.num_layers, p.num_proj, p.r_max, p.proj_dims)
    apply_tuning(pool, args)
    b = wl.batch
    T, S, Td = b.num_tokens, b.num_segments, b.num_decode
    nbytes = lora.workspace_size(pool, T, S + Td)
    x_idx = sorted(set(d.x_src))   # the distinct x buffers (fewer when inputs are shared)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream_obj = torch.cuda.current_stream(dev)
    stream = stream_obj.cuda_stream
    lora.workspace_init(ws, nbytes, stream)
    probs = [(d.x[d.x_src[i]], d.y[i], d.x.shape[2], d.y.shape[2], l, pj)
             for i, (l, pj) in enumerate(d.problems)]
    seg_start = d.seg_start if S else None
    seg_adapter = d.seg_adapter if S else None
    dec = d.dec_adapter if Td else None

    def segment():
        lora.segment(pool, seg_start, seg_adapter, S, dec, Td, T, ws, nbytes, stream)

    def delta():
        lora.delta_grouped(pool, probs, T, S, ws, nbytes, stream)

    m = step_model(wl)
    # the delta launches of the step: the CUDA-core kernel alone for decode batches (up to
    # 256 projections a launch); for batches with prefill segments the fused two-class
    # kernel where h allows it (h a multiple of 128, h <= 5120; up to 64 projections a
    # launch), else the CUDA-core kernel followed by the tensor-core one (64 a launch)
    ceil = lambda a, c: -(-a // c)  # noqa: E731
    nprob = len(probs)
    if b.kind == "decode":
        kname, delta_launches = "bgmv_ring_kernel", ceil(nprob, lora.LORA_MAX_PROBLEMS_PER_LAUNCH)
    elif p.h % 128 == 0 and p.h // 8 <= 640:
        kname, delta_launches = "delta_fused_kernel", ceil(nprob, 64)
    else:
        kname = "bgmv_ring_kernel+sgmv_mma_kernel"
        delta_launches = ceil(nprob, lora.LORA_MAX_PROBLEMS_PER_LAUNCH) + ceil(nprob, 64)
    launches_per_step = 1 + delta_launches   # the grouping kernel and the delta launches

    for _ in range(max(3, args.warmup)):
        segment()
        delta()
    torch.cuda.synchronize()
    assert lora.get_device_error(ws, stream) == 0

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream_obj)
        for k in range(args.steps):
            e0, e1, e2 = ev[k]
            e0.record(stream_obj)
            segment()
            e1.record(stream_obj)
            delta()
            e2.record(stream_obj)
        end.record(stream_obj)
        torch.cuda.synchronize()
    barrier(world)
    elapsed = start.elapsed_time(end) / 1e3
    kern = [ev[k][1].elapsed_time(ev[k][2]) / 1e3 for k in range(args.steps)]
    err = lora.get_device_error(ws, stream)
    assert err == 0, f"device error bits {err:#x}"
    tokens_step = m["adapted_tokens"]
    value, elapsed_max = aggregate_throughput(tokens_step, args.steps, world, elapsed)

    # roofline of the dominant kernel (the delta kernel): per launch, the step's delta
    # launches being of equal size (problems are split into balanced batches)
    peaks = measured_peaks()
    kern_avg = statistics.mean(kern) / delta_launches
    bytes_launch = m["bytes"] / delta_launches
    achieved = bytes_launch / kern_avg / 1e9
    traffic = ncu_traffic(kname, wl.name, bytes_launch) if kname in KERNEL_SOURCES else None
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "kernel": kname, "kernel_ms": kern_avg * 1e3, "launches_per_step": delta_launches,
                "peak_source": peaks["source"] + " (hbm_gbs, copy kernel)",
                "bytes_per_launch": bytes_launch}

    # one step (grouping + delta launches) captured in a CUDA graph and replayed: median and
    # p10 / p90 of the replays; for decode also with one delta launch per projection (the
    # shape of a serving loop that applies each projection's delta next to its base GEMM)
    graph = {"step": graph_timing(lambda st: (lora.segment(pool, seg_start, seg_adapter, S, dec, Td, T, ws,
                                                           nbytes, st),
                                              lora.delta_grouped(pool, probs, T, S, ws, nbytes, st)),
                                  tokens_step, dev, args.graph_replays)}
    if b.kind == "decode":
        graph["per_projection"] = graph_timing(
            lambda st: (lora.segment(pool, seg_start, seg_adapter, S, dec, Td, T, ws, nbytes, st),
                        [lora.delta_grouped(pool, [pr], T, S, ws, nbytes, st) for pr in probs]),
            tokens_step, dev, args.graph_replays)
    assert lora.get_device_error(ws, stream) == 0

    # end to end through the C ABI with host buffers: every step copies its inputs (x, y and
    # the batch's adapter ids) in from pinned host memory and reads its result y back, inside
    # the timed region.  Steps run as a serving loop runs them, over three device slots: the
    # inputs of step k+1 and the result of step k-1 move on their own streams while step k
    # computes; a slot is refilled only once its previous result has been read back (with two
    # slots that wait would chain copy-in, call and copy-out of alternate steps).
    xh = torch.empty_like(d.x, device="cpu").pin_memory()
    yh = torch.empty_like(d.y, device="cpu").pin_memory()
    xh.copy_(d.x)
    yh.copy_(d.y)
    yo = torch.empty_like(yh).pin_memory()
    if b.kind == "decode":
        meta_src = [d.token_adapter]
    elif b.kind == "prefill":
        meta_src = [d.seg_start, d.seg_adapter]
    else:
        meta_src = [d.seg_start, d.seg_adapter, d.dec_adapter]
    meta_h = [m.cpu().pin_memory() for m in meta_src]
    n_slots = args.e2e_slots
    slots = []
    for k in range(n_slots):
        xs = d.x if k == 0 else torch.empty_like(d.x)
        ys = d.y if k == 0 else torch.empty_like(d.y)
        metas = [torch.empty_like(m) for m in meta_src]
        probs_k = [(xs[d.x_src[i]], ys[i], xs.shape[2], ys.shape[2], l, pj)
                   for i, (l, pj) in enumerate(d.problems)]
        slots.append((xs, ys, metas, probs_k))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    e2e_steps = max(3, min(args.steps, 50))

    def api_call(slot):
        _, _, metas, probs_k = slot
        if b.kind == "decode":
            lora.bgmv(pool, probs_k, metas[0], T, ws, nbytes, stream)
        elif b.kind == "prefill":
            lora.sgmv(pool, probs_k, metas[0], metas[1], S, T, ws, nbytes, stream)
        else:
            lora.apply_mixed(pool, probs_k, metas[0], metas[1], S, metas[2], Td, T, ws, nbytes,
                             stream)

    def e2e_run(nsteps, first_event=None):
        ev_out = [None] * n_slots
        last = None
        for k in range(nsteps):
            slot = slots[k % n_slots]
            xs, ys, metas, _ = slot
            with torch.cuda.stream(s_in):
                if k == 0 and first_event is not None:
                    first_event.record(s_in)
                if ev_out[k % n_slots] is not None:
                    s_in.wait_event(ev_out[k % n_slots])
                if len(x_idx) == len(d.problems):
                    xs.copy_(xh, non_blocking=True)
                else:   # only the x buffers that are read
                    for i in x_idx:
                        xs[i].copy_(xh[i], non_blocking=True)
                ys.copy_(yh, non_blocking=True)
                for m_d, m_h in zip(metas, meta_h):
                    m_d.copy_(m_h, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            stream_obj.wait_event(ev_in)
            api_call(slot)
            ev_c = torch.cuda.Event()
            ev_c.record(stream_obj)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c)
                yo.copy_(ys, non_blocking=True)
                last = torch.cuda.Event(enable_timing=True)
                last.record(s_out)
                ev_out[k % n_slots] = last
        return last

    e2e_run(n_slots)
    torch.cuda.synchronize()
    barrier(world)
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = e2e_run(e2e_steps, first_event=s0)
    torch.cuda.synchronize()
    assert lora.get_device_error(ws, stream) == 0
    e2e_elapsed = max_over_ranks(s0.elapsed_time(s1) / 1e3, world)
    api_name = {"decode": "lora_bgmv", "prefill": "lora_sgmv"}.get(b.kind, "lora_apply_mixed")
    e2e = {"value": tokens_step * e2e_steps * world / e2e_elapsed, "unit": UNIT,
           "h2d_bytes_per_step": d.x[0].numel() * 2 * len(x_idx) + d.y.numel() * 2 +
                                 sum(m.numel() * 4 for m in meta_h),
           "d2h_bytes_per_step": d.y.numel() * 2, "steps": e2e_steps,
           "api": f"{api_name} (C ABI); pinned host x, y and adapter ids in, y out, every step; "
                  f"three device slots, copies of neighbouring steps overlapping the call"}

    staging = None
    if args.config in ("stress-distinct", "stress-zipf") and args.stage_steps > 0:
        variant = args.config.split("-")[1]
        wl_steps = step_batches(wl, args.stage_steps, variant)
        staging = run_staging(args, wl_steps, pool, d, ws, nbytes, stream_obj, dev)

    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            runner = OracleRunner(wl, args.ref_problems)
            rate, dt, done = runner.timed_sample(args.ref_seconds)
            cpu = {"value": rate, "unit": UNIT, "cores": runner.threads, "kind": "oracle",
                   "sample": f"{done} projection deltas ({done / len(wl.problems):.2f} steps of "
                             f"{len(wl.problems)}, cycling over the first {len(runner.probs)}), "
                             f"all {wl.batch.num_tokens} tokens each, {dt:.1f} s wall on "
                             f"{runner.threads} threads, rate scaled to whole steps",
                   "cpu_model": cpu_model()}
            one = runner.single_thread_sample(args.ref_seconds / 3)
            if one is not None:
                rate1, dt1, done1 = one
                cpu["single_thread"] = {"value": rate1, "unit": UNIT,
                                        "sample": f"{done1} projection deltas, {dt1:.1f} s wall on 1 thread"}
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": max(3, args.warmup),
                "ms_per_step": 1e3 * elapsed_max / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": config_dict(wl, args), "roofline": roofline, "cpu_baseline": cpu,
                "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
                "graph": graph, "clocks": clk.summary(), "impl": "ours",
                "tuning": pool.get_tuning()}
        if staging is not None:
            line["staging"] = staging
        print(json.dumps(line), flush=True)
    pool.close()


# ----------------------------------------------------------------------------- distinct-adapter sweep

def run_sweep_distinct(args, local: int):
    """The decode workload's pool and projections (--config; the Llama-7B decode workload by
    default); its decode tokens spread round-robin over D adapters drawn without replacement
    from its adapters (seed 7000 + D), D = 1, 2, 4, ..., 64
    (--sweep-counts).
    One JSON line per D: step time of the delta launch (CUDA events, K steps after W warm-up),
    adapted tokens/s and the fraction of the measured HBM peak."""
    import torch

    import heterogeneous_adapters_gb300 as lora
    from workloads.materialize import device_inputs

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    wl = workload_for(args.config)
    d = device_inputs(wl, device=dev, nan_dummies=False)
    p = wl.pool
    pool = lora.Pool(d.pool, p.num_pages, p.h, d.pt, p.pt.size, d.pt_off, d.ranks, d.scales,
                     p.num_adapters, p.num_layers, p.num_proj, p.r_max, p.proj_dims)
    apply_tuning(pool, args)
    T = wl.batch.num_tokens
    nbytes = lora.workspace_size(pool, T, T)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream_obj = torch.cuda.current_stream(dev)
    stream = stream_obj.cuda_stream
    lora.workspace_init(ws, nbytes, stream)
    probs = [(d.x[i], d.y[i], d.x.shape[2], d.y.shape[2], l, pj) for i, (l, pj) in enumerate(d.problems)]
    peaks = measured_peaks()
    for D in (int(v) for v in args.sweep_counts.split(",")):
        rng = np.random.default_rng(7000 + D)
        chosen = rng.choice(p.num_adapters, size=D, replace=False)
        ids = chosen[np.arange(T) % D].astype(np.int32)
        d.token_adapter.copy_(torch.from_numpy(ids))
        lora.segment(pool, None, None, 0, d.token_adapter, T, T, ws, nbytes, stream)
        for _ in range(max(3, args.warmup)):
            lora.delta_grouped(pool, probs, T, 0, ws, nbytes, stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream_obj)
        for _ in range(args.steps):
            lora.delta_grouped(pool, probs, T, 0, ws, nbytes, stream)
        e1.record(stream_obj)
        torch.cuda.synchronize()
        assert lora.get_device_error(ws, stream) == 0
        ms = e0.elapsed_time(e1) / args.steps
        m = step_model(wl, ids=ids)
        gbs = m["bytes"] / (ms / 1e3) / 1e9
        print(json.dumps({"sweep": "distinct_adapters", "workload": wl.name, "distinct": D,
                          "ranks_mean": float(p.ranks[chosen].mean()), "delta_ms": ms,
                          "tokens_per_s": T / (ms / 1e3), "bytes_per_step": m["bytes"],
                          "achieved_gbs": gbs, "frac_of_peak": gbs / peaks["hbm_gbs"],
                          "steps": args.steps}), flush=True)
    pool.close()


# ----------------------------------------------------------------------------- few-projection launches

def run_sweep_few(args, local: int):
    """Launches of 1 .. 8 projections of the Llama-7B decode batch (the shape of a serving
    loop that applies each projection's delta next to its base GEMM): per launch time of the
    cluster kernel and the ring kernel, each launch on the next
    projections of the step (no launch re-reads the previous one's x, y or pages from L2).
    One JSON line per (projections, kernel)."""
    import torch

    import heterogeneous_adapters_gb300 as lora
    from workloads.materialize import device_inputs

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    wl = workload_for(args.config)   # the Llama-7B decode batch unless --config names another
    d = device_inputs(wl, device=dev, nan_dummies=False)
    p = wl.pool
    pool = lora.Pool(d.pool, p.num_pages, p.h, d.pt, p.pt.size, d.pt_off, d.ranks, d.scales,
                     p.num_adapters, p.num_layers, p.num_proj, p.r_max, p.proj_dims)
    T = wl.batch.num_tokens
    nbytes = lora.workspace_size(pool, T, T)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream_obj = torch.cuda.current_stream(dev)
    stream = stream_obj.cuda_stream
    lora.workspace_init(ws, nbytes, stream)
    probs = [(d.x[i], d.y[i], d.x.shape[2], d.y.shape[2], l, pj) for i, (l, pj) in enumerate(d.problems)]
    peaks = measured_peaks()
    lora.segment(pool, None, None, 0, d.token_adapter, T, T, ws, nbytes, stream)
    kernels = {"cluster": dict(split_max_problems=8), "ring": dict(split_max_problems=0)}
    for n in (1, 2, 3, 4, 6, 8):
        groups = [probs[i:i + n] for i in range(0, len(probs) - n + 1, n)]
        if not groups:
            continue
        m = step_model(wl, problems=wl.problems[:n])
        for name, tun in kernels.items():
            pool.set_tuning(**tun)
            for g in groups[:4]:
                lora.delta_grouped(pool, g, T, 0, ws, nbytes, stream)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            launches = max(len(groups), args.steps)
            e0.record(stream_obj)
            for k in range(launches):
                lora.delta_grouped(pool, groups[k % len(groups)], T, 0, ws, nbytes, stream)
            e1.record(stream_obj)
            torch.cuda.synchronize()
            assert lora.get_device_error(ws, stream) == 0
            ms = e0.elapsed_time(e1) / launches
            gbs = m["bytes"] / (ms / 1e3) / 1e9
            print(json.dumps({"sweep": "few_projections", "projections": n, "kernel": name,
                              "launch_ms": ms, "bytes_per_launch": m["bytes"], "achieved_gbs": gbs,
                              "frac_of_peak": gbs / peaks["hbm_gbs"], "launches": launches}), flush=True)
    pool.set_tuning()
    pool.close()


# ----------------------------------------------------------------------------- FMA / MMA threshold sweep

def run_sweep_threshold(args, local: int):
    """Where the tensor cores start to pay: prefill batches of T = 2,048 rows cut into
    segments of n rows (n = 1, 2, 4 ... 128), every segment with its own adapter (so every
    segment reads its pages once), all adapters of one rank r (8, 16, 64, 128), h = 4096,
    2 layers x 4 projections per launch.  Each point runs once with every segment on the
    CUDA-core kernels (tuning mma_min_rows = 0) and once with every segment of n >= 2 rows on
    the tensor-core tiles (mma_min_rows = n).  One JSON line per (r, n, path)."""
    import torch

    import heterogeneous_adapters_gb300 as lora
    from workloads import spec
    from workloads.materialize import device_inputs

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    peaks = measured_peaks()
    h, L, P, T = 4096, 2, 4, 2048
    ranks_swept = [int(r) for r in args.sweep_ranks.split(",")]
    lengths = [int(n) for n in args.sweep_lengths.split(",")]
    for r in ranks_swept:
        rng = np.random.default_rng(8000 + r)
        N = T
        pool_d = spec.make_pool_all_resident(rng, h, L, P, np.full(N, r, np.int32))
        order = rng.permutation(N).astype(np.int32)
        batch = spec.Batch(np.asarray([0, T], np.int32), order[:1].copy(), np.zeros(0, np.int32))
        wl = spec.Workload(f"threshold-h{h}-r{r}", 8000 + r, pool_d, batch, spec.all_problems(L, P))
        d = device_inputs(wl, device=dev, nan_dummies=False)
        pool = lora.Pool(d.pool, pool_d.num_pages, h, d.pt, pool_d.pt.size, d.pt_off, d.ranks,
                         d.scales, N, L, P, pool_d.r_max)
        probs = [(d.x[i], d.y[i], d.x.shape[2], d.y.shape[2], l, pj)
                 for i, (l, pj) in enumerate(d.problems)]
        stream_obj = torch.cuda.current_stream(dev)
        stream = stream_obj.cuda_stream
        for n in lengths:
            S = T // n
            seg_start = torch.arange(0, S * n + 1, n, dtype=torch.int32, device=dev)
            seg_adapter = torch.from_numpy(order[:S].copy()).to(dev)
            ids = np.repeat(order[:S], n)
            nbytes = lora.workspace_size(pool, T, S)
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            lora.workspace_init(ws, nbytes, stream)
            m = step_model(dataclasses_replace_batch(wl, spec.Batch(seg_start.cpu().numpy(), order[:S].copy(),
                                                                    np.zeros(0, np.int32))), ids=ids)
            for path, mma_min in (("cuda-core", 0), ("tensor-core", max(2, n))):
                if path == "tensor-core" and n < 2:
                    continue
                pool.set_tuning(**dict(tuning_args(args), mma_min_rows=mma_min))
                for _ in range(max(3, args.warmup)):
                    lora.sgmv(pool, probs, seg_start, seg_adapter, S, T, ws, nbytes, stream)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream_obj)
                for _ in range(args.steps):
                    lora.sgmv(pool, probs, seg_start, seg_adapter, S, T, ws, nbytes, stream)
                e1.record(stream_obj)
                torch.cuda.synchronize()
                assert lora.get_device_error(ws, stream) == 0
                ms = e0.elapsed_time(e1) / args.steps
                gbs = m["bytes"] / (ms / 1e3) / 1e9
                print(json.dumps({"sweep": "fma_mma_threshold", "rank": r, "segment_rows": n,
                                  "segments": S, "path": path, "step_ms": ms,
                                  "bytes_per_step": m["bytes"], "achieved_gbs": gbs,
                                  "frac_of_peak": gbs / peaks["hbm_gbs"],
                                  "tflops": m["flops"] / (ms / 1e3) / 1e12, "steps": args.steps}),
                      flush=True)
            del ws
        pool.close()
        del d
        torch.cuda.empty_cache()


def dataclasses_replace_batch(wl, batch):
    import dataclasses
    return dataclasses.replace(wl, batch=batch)


# ----------------------------------------------------------------------------- staging scenario

class SliceUnits:
    """The unified-pool stress workload's slices as units of the library's adapter cache
    (lora_cache_*): unit s is slice s (one layer's pages of one adapter, P * 2 * r_s pages,
    listed in the pool description slice by slice), read by every page-table entry that
    points into it.  Holds the fixed maps page-table entry -> (slice, position in the
    slice), the slices a batch reads, and the pinned host copy of every slice (the host
    tier the misses are staged from)."""

    def __init__(self, wl, pool_t):
        p = wl.pool
        self.wl = wl
        n = p.num_adapters
        self.spp = (p.num_proj * 2 * p.ranks.astype(np.int64)).astype(np.int32)   # pages per slice
        self.slice_off = np.concatenate([[0], np.cumsum(self.spp)[:-1]])
        owner = np.repeat(np.arange(n), self.spp)
        page_slice = np.full(p.num_pages, -1, np.int64)
        page_slice[p.page_ids] = owner
        page_pos = np.full(p.num_pages, -1, np.int64)
        page_pos[p.page_ids] = np.arange(p.page_ids.size) - self.slice_off[owner]
        self.ent_slice = page_slice[p.pt]
        self.ent_pos = page_pos[p.pt]
        order = np.argsort(self.ent_slice, kind="stable")
        counts = np.bincount(self.ent_slice, minlength=n)
        self.ent_off = np.concatenate([[0], np.cumsum(counts)])
        self.ent_sorted = order.astype(np.int64)
        self.host = None
        if pool_t is not None:
            import torch
            allp = torch.from_numpy(p.page_ids.astype(np.int64)).to(pool_t.device)
            self.host = pool_t[allp].cpu().pin_memory()

    def needed(self, token_adapter) -> np.ndarray:
        """Slices read by a batch: every slice its adapters' page-table blocks point into."""
        p = self.wl.pool
        ids = np.unique(token_adapter[token_adapter >= 0])
        ent = np.concatenate([np.arange(p.pt_off[a], p.pt_off[a] + p.num_layers * p.num_proj * 2 *
                                        int(p.ranks[a])) for a in ids])
        return np.unique(self.ent_slice[ent])

    def rewrite(self, s: int, pages: np.ndarray):
        """Page-table entries of slice s and the pages they take once s sits in `pages`."""
        ent = self.ent_sorted[self.ent_off[s]:self.ent_off[s + 1]]
        return ent, pages[self.ent_pos[ent]]

    def plan(self, cache, need):
        """Acquire every slice of `need` in the adapter cache (one more user each): the
        misses' host rows, destination pages and page-table rewrites, and the slices that
        became LOADING (None when every slice was resident)."""
        rows, dst, ui, up, loading = [], [], [], [], []
        for s in need:
            got = cache.try_acquire(int(s))
            if got is None:
                raise SystemExit("adapter cache full: every resident slice is in use (raise --stage-headroom)")
            loaded, pages, _ = got
            if loaded:
                rows.append(np.arange(self.slice_off[s], self.slice_off[s] + self.spp[s]))
                dst.append(pages)
                ent, new = self.rewrite(int(s), pages.astype(np.int64))
                ui.append(ent)
                up.append(new)
                loading.append(int(s))
        if not loading:
            return None
        return np.concatenate(rows), np.concatenate(dst), np.concatenate(ui), np.concatenate(up), loading


def step_batches(wl, n: int, variant: str):
    """n batches over the same pool: 256 distinct adapters, or Zipf(1.2) ids, per step."""
    import dataclasses

    from workloads import spec
    out = []
    N = wl.pool.num_adapters
    T = wl.batch.num_tokens
    for k in range(n):
        rng = np.random.default_rng(wl.seed * 1000 + k)
        if variant == "distinct":
            ids = rng.choice(N, size=T, replace=False)
        else:
            ids = rng.choice(N, size=T, p=spec.zipf_probs(N, 1.2))
        b = spec.Batch(np.zeros(1, np.int32), np.zeros(0, np.int32), ids.astype(np.int32))
        out.append(dataclasses.replace(wl, batch=b))
    return out


def run_staging(args, wl_steps, pool, d, ws, nbytes, stream_obj, dev):
    """Unified-pool stress with staging, driven by the library's host runtime: each step's
    requests go through the batch scheduler (lora_sched_*), the adapter cache (lora_cache_*)
    keeps the slices resident in a fixed share of the pool's pages (least recently used
    slices no running request reads are evicted), and the misses of step k+1 are staged
    during step k on a side stream through the copy engines (lora_stage_pages_ce: one host
    to device copy per run of consecutive destination pages straight into the pool -- the
    cache hands a slice's pages out of its free list in a run -- then one small kernel
    rewriting the page table).  Reported: the decode kernel's time per step with staging
    running beside it and, for the same steps' batches, without; the staged bytes over the
    copies' duration."""
    import torch

    import heterogeneous_adapters_gb300 as lora
    wl0 = wl_steps[0]
    p = wl0.pool
    units = SliceUnits(wl0, d.pool)
    # The cache's pages: the pages the slices occupy now plus stage_headroom of them taken
    # from the pool's other pages (the rest stands for KV-cache blocks).  Under this
    # workload's reading a step reads nearly every slice (each of its adapters reads a
    # different slice in each of the 32 layers), so the cache must hold about all of them;
    # the headroom is what lets the slices a step newly needs come in while the ones it
    # no longer reads leave.
    n_slice_pages = p.page_ids.size
    extra = int(n_slice_pages * args.stage_headroom)
    spare = np.setdiff1d(np.arange(p.num_pages), p.page_ids)[:extra]
    managed = np.concatenate([p.page_ids, spare]).astype(np.int32)
    cache = lora.AdapterCache(managed, units.spp)
    sched = lora.Scheduler(None)
    side = torch.cuda.Stream(device=dev)
    probs = [(d.x[i], d.y[i], d.x.shape[2], d.y.shape[2], l, pj) for i, (l, pj) in enumerate(d.problems)]
    # room for every slice: the first step stages everything it reads
    staging = torch.empty(int(units.spp.sum()) * p.h * 2, dtype=torch.uint8, device=dev)
    T = wl0.batch.num_tokens
    keep = []   # host buffers of staging calls in flight

    def batch_of(k):
        """Step k's requests through the scheduler: one decode token per request."""
        ids = wl_steps[k].batch.token_adapter()
        for i, a in enumerate(ids):
            sched.enqueue(k * T + i, int(a), 1)
        _, ads, _ = sched.pick(T, T)
        return ads.astype(np.int32)

    def plan(need):
        return units.plan(cache, need)

    def launch_stage(plan_, stream):
        rows, dst, ui, up, loading = plan_
        src = units.host[torch.from_numpy(rows)].pin_memory()
        dst_t = torch.from_numpy(dst.astype(np.int32)).pin_memory()
        ui_t = torch.from_numpy(ui.astype(np.int64)).pin_memory()
        up_t = torch.from_numpy(up.astype(np.int32)).pin_memory()
        assert dst.size * p.h * 2 <= staging.numel(), "staging buffer too small for one step's misses"
        e0, e_copy, e1 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e_copy.record(stream)   # creates the event; the library records it again after the copy
        e0.record(stream)
        lora.stage_pages_ce(pool, src, staging, staging.numel(), dst_t, dst.size, d.pt, ui_t, up_t, ui.size,
                            stream.cuda_stream, copied_event=e_copy)
        e1.record(stream)
        keep.append((src, dst_t, ui_t, up_t))
        return e0, e_copy, e1, dst.size * p.h * 2, loading

    # step 0's slices, staged before the loop
    ads0 = batch_of(0)
    need = units.needed(ads0)
    pl = plan(need)
    if pl is not None:
        _, _, _, _, loading = launch_stage(pl, stream_obj)
        torch.cuda.synchronize()
        for s in loading:
            cache.loaded(s)
    kern_ms, copy_ms, stage_ms, stage_bytes, misses, step_ads = [], [], [], [], [], []
    staged = None
    ads = ads0
    for k in range(len(wl_steps)):
        if staged is not None:   # step k's misses, staged during step k-1
            stream_obj.wait_event(staged[2])
            staged[2].synchronize()
            copy_ms.append(staged[0].elapsed_time(staged[1]))
            stage_ms.append(staged[0].elapsed_time(staged[2]))
            stage_bytes.append(staged[3])
            misses.append(len(staged[4]))
            for s in staged[4]:
                cache.loaded(s)
            staged = None
        tok = torch.from_numpy(ads).to(dev)
        step_ads.append(ads)
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record(stream_obj)
        lora.bgmv(pool, probs, tok, T, ws, nbytes, stream_obj.cuda_stream)
        k1.record(stream_obj)
        nxt_ads, nxt_need = None, None
        if k + 1 < len(wl_steps):
            nxt_ads = batch_of(k + 1)
            nxt_need = units.needed(nxt_ads)
            pl = plan(nxt_need)   # step k's slices have users: they are never evicted
            if pl is not None:
                with torch.cuda.stream(side):
                    staged = launch_stage(pl, side)
        k1.synchronize()
        kern_ms.append(k0.elapsed_time(k1))
        for s in need:   # step k is done with its slices
            cache.release(int(s))
        keep[:] = keep[-2:]
        ads, need = nxt_ads, nxt_need
    torch.cuda.synchronize()
    err = lora.get_device_error(ws, stream_obj.cuda_stream)
    # the same decode steps (each step's batch, every slice resident) with nothing staged beside them
    alone = []
    for ads_k in step_ads:
        tok = torch.from_numpy(ads_k).to(dev)
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record(stream_obj)
        lora.bgmv(pool, probs, tok, T, ws, nbytes, stream_obj.cuda_stream)
        k1.record(stream_obj)
        k1.synchronize()
        alone.append(k0.elapsed_time(k1))
    # the copy alone: the median step's bytes (and 4x as many) with nothing else running
    alone_copy = {}
    for mult in (1, 4):
        nbytes_c = int(min(staging.numel(), (statistics.median(stage_bytes) if stage_bytes else 0) * mult))
        if nbytes_c <= 0:
            break
        src = torch.empty(nbytes_c, dtype=torch.uint8).pin_memory()
        ms = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(side)
            with torch.cuda.stream(side):
                staging[:nbytes_c].copy_(src, non_blocking=True)
            e1.record(side)
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
        alone_copy[f"{nbytes_c}"] = {"ms": statistics.median(ms), "gbs": nbytes_c / (statistics.median(ms) * 1e6)}
    st = cache.stats()
    cache.close()
    sched.close()
    med = statistics.median
    return {"steps": len(wl_steps), "runtime": "lora_cache_* (slices as units), lora_sched_*, lora_stage_pages_ce",
            "kernel_ms_median": med(kern_ms), "kernel_ms_alone_median": med(alone),
            "kernel_slowdown": med(kern_ms) / med(alone) - 1.0,
            "kernel_slowdown_per_step_median": med([a / b - 1.0 for a, b in zip(kern_ms, alone)]),
            "copy_ms_median": med(copy_ms) if copy_ms else 0.0,
            "stage_ms_median": med(stage_ms) if stage_ms else 0.0,
            "stage_bytes_median": med(stage_bytes) if stage_bytes else 0,
            "copy_gbs_median": (med([b / (t * 1e6) for b, t in zip(stage_bytes, copy_ms)]) if copy_ms else None),
            "copy_alone": alone_copy,
            "slices_staged_median": med(misses) if misses else 0, "cache_pages": int(managed.size),
            "cache": st, "device_error": err}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="decode",
                    help="workload: tiny, decode, prefill, mixed, stress-distinct, stress-zipf, "
                         "llama3-decode, llama3-prefill, llama3-mixed, or a -small variant")
    ap.add_argument("--graph-replays", type=int, default=50,
                    help="timed replays of the CUDA graph of one step")
    ap.add_argument("--e2e-slots", type=int, default=3, choices=[1, 2, 3, 4],
                    help="device slots of the end-to-end leg's copy/compute pipeline")
    ap.add_argument("--ref-seconds", type=float, default=15.0,
                    help="CPU seconds of the oracle sample beside our arm")
    ap.add_argument("--ref-budget-s", type=float, default=120.0,
                    help="total oracle seconds of the reference arm's timed steps")
    ap.add_argument("--ref-problems", type=int, default=16,
                    help="projections whose host inputs the oracle prepares")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stage-headroom", type=float, default=0.05,
                    help="unified-pool stress: pages the adapter cache holds beyond the slices' own, "
                         "as a fraction of them")
    ap.add_argument("--stage-steps", type=int, default=20,
                    help="steps of the staging scenario (stress-distinct / stress-zipf)")
    ap.add_argument("--shared-x", action="store_true",
                    help="q, k and v of a layer read one x (as in a transformer), not one each")
    ap.add_argument("--sweep-distinct", action="store_true",
                    help="instead of the bench line: decode tokens/s against the number of "
                         "distinct adapters in the batch (1..64) at the Llama-7B decode shape")
    ap.add_argument("--sweep-threshold", action="store_true",
                    help="instead of the bench line: CUDA-core against tensor-core step time "
                         "over segment length x rank (the FMA / MMA crossover)")
    ap.add_argument("--tuning", default="",
                    help="launch tuning of the pool, k=v,...: ring_rows_per_stage, "
                         "split_max_problems, mma_min_rows, mma_y_stages, fused_ring_speed "
                         "(the defaults otherwise)")
    ap.add_argument("--sweep-few", action="store_true",
                    help="instead of the bench line: launches of 1 .. 8 projections of the decode "
                         "batch through the cluster and ring kernels")
    ap.add_argument("--sweep-ranks", default="8,16,64,128")
    ap.add_argument("--sweep-lengths", default="1,2,4,8,16,32,64,128")
    ap.add_argument("--sweep-counts", default="1,2,4,8,16,32,64",
                    help="distinct-adapter counts of --sweep-distinct")
    args = ap.parse_args()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.sweep_distinct:
        run_sweep_distinct(args, local)
    elif args.sweep_threshold:
        run_sweep_threshold(args, local)
    elif args.sweep_few:
        run_sweep_few(args, local)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
