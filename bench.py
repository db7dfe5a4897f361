"""Benchmark of the ZeRO-3 sharded layer step on one GB300 (or N replicas).

One step = one pass of the whole hot path over one layer: forward
all-gather, backward all-gather, fused reduce-scatter + Adam (three kernel
launches, one C-ABI call ``z3_step_layer``).  Default workload: one d=1024
transformer layer (Wqkv, Wo, W_up, W_down, two norm gains; Psi = 12,584,960)
over N_d = 8 logical ranks, bf16 params/grads, fp32 master/m/v.

Metric: algorithmic HBM bytes of the step ((2 N_d + 34) bytes per unpadded
element) per second, plus params/s and the fraction of the 8 TB/s HBM
figure.  Every step works on one of several rotating replicas of the layer
state whose total is far above the 129 MB L2, so each step starts cold.

Timed region: the clock sampler starts before the warm-up; the K timed steps
are captured once (through z3_step_layer) as one CUDA graph and replayed
(--eager: stream launches); a 512 MiB buffer write queued just before the
start event leaves L2 cold and keeps the GPU busy while the host enqueues
the region, so the region opens on queued work.

The line also carries: the roofline of the fused kernel (timed per launch in
a second event-bracketed pass; DRAM traffic per launch and per whole step
from the committed ncu summaries while the kernel source is unchanged), the
e2e rate through the C ABI from pinned host memory (z3_host_step_run,
uploads and read-backs inside the timed region), sampled SM clocks, the
launch count, and the CPU oracle on the full layer, every kernel on all host
cores (one contiguous piece of the layer per thread) and on one.

Arms:
  default            the CUDA library (inputs resident in HBM)
  --impl reference   the plain CPU oracle on all host cores, on a bounded
                     sample of the same workload (rank 0 only)
Other workloads (--workload): the 7B-style and prime-length layers, every
device call alone (kernels_<layer>), the 24-layer model step with buckets,
prefetch and resident units, the stage-1/2 and plain-DP variants, and the
prime-length sweep; --graph replays their timed steps as one CUDA graph.
Under torchrun (N > 1) every rank runs an independent replica (weak
scaling); the timed region is bracketed by a barrier and the max over ranks
is taken.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sharded ZeRO-3 layer step GB/s and params/s, % of GB300 8 TB/s HBM roofline"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time (the timed region ends when every rank ends)."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(world: int, step_bytes: int, steps: int, ms_max: float) -> float:
    """Whole-job GB/s: every rank ran `steps` steps of `step_bytes` each."""
    return world * step_bytes * steps / (ms_max * 1e-3) / 1e9


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest() -> str:
    """Digest of what decides the code a kernel launch runs: the kernels and
    their launchers, their argument blocks, the layout code that builds the
    launch tables (not the C-ABI validation layer), and the compiler flags
    the kernels are built with."""
    import hashlib
    from optimizer_state_gb300 import build as libbuild
    h = hashlib.sha256()
    for name in ("z3_kernels.cu", "z3_launch.h", "z3_internal.h", "z3_layout.cpp"):
        with open(os.path.join(ROOT, "optimizer_state_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    # include paths name where the repository sits, not what is compiled
    flags = [f for f in libbuild.NVCC_FLAGS if not f.startswith("-I")]
    h.update(repr((flags, libbuild.ARCH)).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(kernel, {}).get(workload)
    if not ent or ent.get("source_digest") != kernel_source_digest():
        return None
    return ent.get("dram_bytes_per_launch")


def profiled_step_traffic(workload: str):
    """DRAM bytes of one whole layer step (forward gather, backward gather,
    fused update) from the committed ncu capture taken with caches left
    alone, so that each kernel carries the write-backs its predecessor left
    in L2; None unless that capture was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get("_per_step", {}).get(workload)
    if not ent or ent.get("source_digest") != kernel_source_digest():
        return None
    return {"dram_bytes": ent["dram_bytes_per_step"],
            "algorithmic_bytes": ent["algorithmic_bytes_per_step"],
            "ratio": round(ent["dram_bytes_per_step"] / ent["algorithmic_bytes_per_step"], 4),
            "capture": ent.get("capture")}


class ClockSampler:
    """nvidia-smi samples taken while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            rows.append((t, parts))
        inside = [r for t, r in rows if self.t0 is not None and self.t0 - 0.06 <= t <= self.t1 + 0.06]
        use = inside if inside else rows
        sm = sorted(float(r[1]) for r in use if r[1].replace(".", "").isdigit())
        mx = [float(r[2]) for r in use if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons,
                "samples": len(use),
                "samples_inside_timed_region": len(inside)}


class LeadIn:
    """Device work enqueued just before a timed region's start event: it
    writes a 512 MiB buffer (four times the 129 MB L2, so the region starts
    with a cold cache) and keeps the GPU busy, about 80 us, while the host
    enqueues the start event and the first launches.  Without it the region
    would open on an idle GPU and count the host's first launch latency."""

    NBYTES = 512 << 20

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(self.NBYTES, dtype=torch.uint8, device=dev)

    def enqueue(self, stream):
        import torch
        with torch.cuda.stream(stream):
            self.buf.zero_()


# --------------------------------------------------------------------------
# the CUDA arm
# --------------------------------------------------------------------------

class Replica:
    """One copy of the layer state: shards, master, m, v, gradients, and the
    transient gathered buffer."""

    def __init__(self, z3, L, w, seed, dev):
        import torch
        from optimizer_state_gb300 import inputs as I
        T = L.psi_padded
        gen = I.make_generator(seed, dev)
        full = I.draw_master(w, gen, dev)
        self.shards = torch.empty(T, dtype=torch.bfloat16, device=dev)
        self.master = torch.empty(T, dtype=torch.float32, device=dev)
        self.m = torch.empty(T, dtype=torch.float32, device=dev)
        self.v = torch.empty(T, dtype=torch.float32, device=dev)
        self.full = torch.empty(L.psi, dtype=torch.bfloat16, device=dev)
        self.grads = I.draw_grads(w, gen, dev)
        z3.z3_partition(L, full, self.shards, self.master, self.m, self.v)
        del full
        self.step = 0


def run_cuda(args, world, rank, local):
    import torch
    import torch.distributed as dist
    from optimizer_state_gb300 import build as libbuild
    from optimizer_state_gb300 import inputs as I
    from optimizer_state_gb300 import z3

    libbuild.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    w = layer_workload(args.workload)
    L = z3.Layout(w.numel, w.n_ranks)
    stats = L.stats()
    step_bytes = stats["hbm_step_layer"]
    scale = 1.0 / w.n_ranks
    state_bytes = (2 + 4 * 3) * L.psi_padded + 2 * L.psi + 2 * w.n_ranks * w.grad_stride
    n_rep = max(2, -(-args.cold_bytes // state_bytes))
    reps = [Replica(z3, L, w, seed=1000 * rank + i, dev=dev) for i in range(n_rep)]
    stream = torch.cuda.current_stream()
    sid = stream.cuda_stream
    launches_per_step = 2 * len_tabs(L, "gather") + len_tabs(L, "reduce")

    def step(rep):
        rep.step += 1
        z3.z3_step_layer(L, rep.shards, rep.full, rep.grads, w.grad_stride, scale, rep.master,
                         rep.m, rep.v, HP, rep.step, stream=sid)

    # the clock sampler starts before the warm-up, so that no idle gap
    # precedes the timed region
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for i in range(args.warmup):
        step(reps[i % n_rep])
    torch.cuda.synchronize()

    # The K timed steps (each with its own step counter) are captured once,
    # through the same C-ABI calls, as one CUDA graph and replayed inside the
    # timed region, unless --eager asks for stream launches (or the graph
    # would hold more than 50,000 launches).
    use_graph = not args.eager and launches_per_step * args.steps <= 50000
    graph = None
    if use_graph:
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap), torch.cuda.graph(graph, stream=cap):
            for i in range(args.steps):
                rep = reps[i % n_rep]
                rep.step += 1
                z3.z3_step_layer(L, rep.shards, rep.full, rep.grads, w.grad_stride, scale,
                                 rep.master, rep.m, rep.v, HP, rep.step, stream=cap.cuda_stream)
        stream.wait_stream(cap)
        torch.cuda.synchronize()
    lead = LeadIn(dev)

    # ---- timed region: K layer steps
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    lead.enqueue(stream)
    clocks.mark(True)
    e0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step(reps[i % n_rep])
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark(False)
    if world > 1:
        dist.barrier()
    ms_total = e0.elapsed_time(e1)
    clock_info = clocks.stop()

    # ---- per-kernel timing pass (same launches, events between kernels):
    # one untimed iteration, then kernel_steps iterations behind a lead-in
    kernel_steps = max(1, args.kernel_steps)

    def kernel_iteration(rep):
        rep.step += 1
        z3.z3_allgather(L, rep.shards, rep.full, stream=sid)
        z3.z3_allgather(L, rep.shards, rep.full, stream=sid)
        z3.z3_reduce_scatter_adam(L, rep.grads, w.grad_stride, scale, None, rep.master, rep.m,
                                  rep.v, rep.shards, HP, rep.step, stream=sid)
    kernel_iteration(reps[0])
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(kernel_steps)]
    torch.cuda.synchronize()
    lead.enqueue(stream)
    for i in range(kernel_steps):
        rep = reps[i % n_rep]
        rep.step += 1
        ev[i][0].record(stream)
        z3.z3_allgather(L, rep.shards, rep.full, stream=sid)
        ev[i][1].record(stream)
        z3.z3_allgather(L, rep.shards, rep.full, stream=sid)
        ev[i][2].record(stream)
        z3.z3_reduce_scatter_adam(L, rep.grads, w.grad_stride, scale, None, rep.master, rep.m,
                                  rep.v, rep.shards, HP, rep.step, stream=sid)
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    t_ag = sum(e[0].elapsed_time(e[1]) + e[1].elapsed_time(e[2]) for e in ev) / (2 * kernel_steps)
    t_rs = sum(e[2].elapsed_time(e[3]) for e in ev) / kernel_steps
    # the gather back to back (kernel_steps calls between two events, rotating
    # replicas): its launch latency overlaps the previous call's drain, as
    # when a caller issues several gathers in a row
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    lead.enqueue(stream)
    b0.record(stream)
    for i in range(kernel_steps):
        rep = reps[i % n_rep]
        z3.z3_allgather(L, rep.shards, rep.full, stream=sid)
    b1.record(stream)
    torch.cuda.synchronize()
    t_ag_b2b = b0.elapsed_time(b1) / kernel_steps

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(args, z3, L, w, reps[0], stream, sid, step_bytes, world)

    ms_max = max_over_ranks(ms_total, world, dev)
    ms_step = ms_max / args.steps
    value = aggregate_gbs(world, step_bytes, args.steps, ms_max)

    if rank == 0:
        peak, peak_kind = measured_hbm_peak()
        rs_bytes = stats["hbm_reduce_scatter_adam"]
        achieved = rs_bytes / (t_rs * 1e-3) / 1e9
        traffic = profiled_traffic("k_reduce_rs_adam", args.workload)
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_step, 6),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": {
                **layer_config(args.workload, w, L.psi, L.S),
                "l2": f"{n_rep} rotating replicas of the layer state "
                      f"({n_rep * state_bytes / 1e9:.2f} GB > 129 MB L2), every step cold",
                "parallelism": f"{world} independent replica(s), one per GPU",
                "launch": (f"one CUDA graph of the {args.steps} timed steps (captured through "
                           f"z3_step_layer)" if use_graph else "stream launches"),
            },
            "params_per_s": round(world * L.psi * args.steps / (ms_max * 1e-3), 1),
            "pct_of_8tbs": round(100.0 * value / (NOMINAL_HBM_GBS * world), 2),
            "kernels_ms": {"allgather": round(t_ag, 6), "reduce_scatter_adam": round(t_rs, 6),
                           "allgather_back_to_back": round(t_ag_b2b, 6)},
            "kernels_ms_how": "allgather and reduce_scatter_adam: each launch alone between two "
                              "events (the roofline pass); allgather_back_to_back: consecutive "
                              "calls between two events",
            "roofline": {
                "kernel": f"{reduce_kernel_name(L)}<RSAdam> (fused reduce-scatter + Adam)",
                "bound": "hbm",
                "achieved": round(achieved, 2),
                "peak": peak,
                "peak_kind": peak_kind,
                "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": traffic,
                "traffic_scope": "one launch captured alone with caches flushed: a lower bound "
                                 "(the write-backs a kernel leaves in L2 land in the next one)",
                "algorithmic_bytes_per_launch": rs_bytes,
                "traffic_per_step": profiled_step_traffic(args.workload),
            },
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clock_info,
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


LAYER_WORKLOADS = ("layer_d1024_nd8", "layer_7b_nd8", "layer_7b_nd64", "layer_primes_nd8",
                   "layer_primes_small_nd8")


def layer_workload(name: str):
    from optimizer_state_gb300 import inputs as I
    if name == "layer_d1024_nd8":
        return I.LAYER_D1024
    if name.startswith("layer_7b_nd"):
        return I.layer_7b(int(name[len("layer_7b_nd"):]))
    if name.startswith("layer_primes_nd"):
        return I.layer_primes(int(name[len("layer_primes_nd"):]))
    if name.startswith("layer_primes_small_nd"):
        return I.layer_primes(int(name[len("layer_primes_small_nd"):]), small=True)
    raise SystemExit(f"unknown layer workload {name}")


def reduce_kernel_name(L) -> str:
    """The reduce kernel a layer's launches run.  The library launches once
    per table of up to 40 non-empty parameters; a table runs the aligned
    kernel when every (parameter, rank) chunk in it has equal full-space and
    shard-space indices modulo the 8-element vector, else the
    window-shifting one.  Tables that disagree give "mixed"."""
    names = set()
    params = [(s, o, F) for n, s, o, F in zip(L.numel, L.shard_numel, L.shard_off, L.full_off)
              if n]
    for t0 in range(0, len(params), 40):
        aligned = all((F + r * s - (r * L.S + o)) % 8 == 0 for s, o, F in params[t0:t0 + 40]
                      for r in range(L.n_ranks))
        names.add("k_reduce_aligned" if aligned else "k_reduce_shifted")
    if len(names) == 1:
        return names.pop()
    return "mixed: k_reduce_aligned and k_reduce_shifted"


def len_tabs(L, kind):
    """Launches per call: one per launch table (a table holds <= 40 params)."""
    n = sum(1 for x in L.numel if x > 0)
    return -(-n // 40)


def parse_full_step(name: str):
    """full_step_nd16[_prefetch[<D>]][_bucket<k>][_persist<T>] -> (prefetch
    depth D (1 when the digits are omitted, 0 without _prefetch), layers per
    bucket k (1), persistence threshold T (0))."""
    m = re.fullmatch(r"full_step_nd16(_prefetch(\d*))?(_bucket(\d+))?(_persist(\d+))?", name)
    if m is None:
        raise SystemExit(f"unknown workload {name}")
    depth = (int(m.group(2)) if m.group(2) else 1) if m.group(1) else 0
    bucket = int(m.group(4)) if m.group(3) else 1
    persist = int(m.group(6)) if m.group(5) else 0
    if bucket < 1 or depth > 7:
        raise SystemExit(f"{name}: buckets of >= 1 layer, prefetch depth <= 7")
    return depth, bucket, persist


def run_multi(args, world, rank, local):
    """Full step (24 layers + embedding, N_d = 16) or one sweep point
    (AG, AG, 4 micro-batches reduced and accumulated, Adam fused with the
    last): the step is timed as a whole with CUDA events."""
    import torch
    from optimizer_state_gb300 import build as libbuild
    from optimizer_state_gb300 import inputs as I
    from optimizer_state_gb300 import schedule, z3
    libbuild.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream()
    sid = stream.cuda_stream
    if args.workload.startswith("full_step_nd16"):
        depth, bucket, persist = parse_full_step(args.workload)
        model = schedule.full_step_model(dev, seed=rank, prefetch=depth, bucket_layers=bucket,
                                         persistence_threshold=persist)
        step_bytes, psi, launches = model.step_bytes, model.psi, model.launches_per_step()

        def step(i):
            model.step(HP, stream=sid)
        extra = {"units": len(model.units), "n_ranks": 16, "bucket_layers": bucket,
                 "prefetch_depth": depth, "persistence_threshold": persist,
                 "resident_params": sum(len(u.L.numel) for u in model.units
                                        if u.resident is not None),
                 "bytes_per_param": round(step_bytes / psi, 4),
                 "transient_buffer_elems": model.full.numel()}
    elif args.workload.startswith("sweep_n"):
        n_s, nd_s = args.workload[len("sweep_n"):].split("_nd")
        w = I.sweep(int(n_s), int(nd_s))
        u = schedule.Unit(w, dev, I.make_generator(rank, dev))
        full = torch.empty(u.L.psi, dtype=torch.bfloat16, device=dev)
        acc = torch.empty(u.L.psi_padded, dtype=torch.float32, device=dev)
        st = u.L.stats()
        step_bytes = 2 * st["hbm_allgather"] + st["hbm_reduce_scatter"] + \
            (w.micro_batches - 2) * st["hbm_reduce_scatter_accumulate"] + \
            st["hbm_reduce_scatter_adam"] + 4 * u.L.psi
        psi, launches = u.L.psi, 2 + w.micro_batches
        scale = 1.0 / w.n_ranks

        def step(i):
            z3.z3_allgather(u.L, u.shards, full, stream=sid)
            z3.z3_allgather(u.L, u.shards, full, stream=sid)
            z3.z3_reduce_scatter(u.L, u.grads, w.grad_stride, acc, scale, stream=sid)
            for _ in range(w.micro_batches - 2):
                z3.z3_reduce_scatter(u.L, u.grads, w.grad_stride, acc, scale, accumulate=True,
                                     stream=sid)
            z3.z3_reduce_scatter_adam(u.L, u.grads, w.grad_stride, scale, acc, u.master, u.m,
                                      u.v, u.shards, HP, i + 1, stream=sid)
        extra = {"n": w.numel[0], "n_ranks": w.n_ranks, "micro_batches": w.micro_batches,
                 "note": "one gradient buffer re-read by every micro-batch"}
    elif args.workload in ("dp_d1024_nd8", "stage1_d1024_nd8", "stage2_d1024_nd8"):
        w = I.LAYER_D1024
        kind = args.workload.split("_")[0]
        n_rep = 4                                   # rotating replicas: every step cold
        if kind == "dp":
            reps = [schedule.DPReplica(w, dev, I.make_generator(100 * rank + i, dev))
                    for i in range(n_rep)]
            bpp = (2 * w.n_ranks + 4) + 30

            def step(i):
                reps[i % n_rep].step(HP, i + 1, stream=sid)
        else:
            reps = [schedule.Unit(w, dev, I.make_generator(100 * rank + i, dev))
                    for i in range(n_rep)]
            L0 = reps[0].L
            full = torch.empty(L0.psi, dtype=torch.bfloat16, device=dev)
            gfull = torch.empty(L0.psi, dtype=torch.float32, device=dev)
            gsh = torch.empty(L0.psi_padded, dtype=torch.float32, device=dev)
            if kind == "stage1":
                bpp = (2 * w.n_ranks + 4) + 8 + 30 + 4

                def step(i):
                    schedule.stage1_step(reps[i % n_rep], gfull, gsh, full, HP, i + 1, stream=sid)
            else:
                bpp = (2 * w.n_ranks + 26) + 4

                def step(i):
                    schedule.stage2_step(reps[i % n_rep], full, HP, i + 1, stream=sid)
        psi = w.psi
        step_bytes = bpp * psi
        launches = {"dp": 2, "stage1": 4, "stage2": 2}[kind]
        extra = {"n_ranks": w.n_ranks, "bytes_per_param": bpp, "variant": kind,
                 "l2": f"{n_rep} rotating replicas"}
    else:
        raise SystemExit(f"unknown workload {args.workload}")
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    graph = None
    if args.graph and launches * args.steps > 50000:
        raise SystemExit(f"--graph: {launches * args.steps} launches in one graph; use fewer --steps")
    if args.graph:
        # the K timed steps (step counter advancing) captured as one CUDA
        # graph, replayed once inside the timed region: no host launch cost
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap), torch.cuda.graph(graph, stream=cap):
            sid_saved = sid
            sid = cap.cuda_stream
            for i in range(args.steps):
                step(args.warmup + i)
            sid = sid_saved
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        extra["launch"] = f"one CUDA graph of the {args.steps} timed steps"
    lead = LeadIn(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    lead.enqueue(stream)
    clocks.mark(True)
    e0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step(args.warmup + i)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark(False)
    if world > 1:
        dist.barrier()
    clock_info = clocks.stop()
    ms_max = max_over_ranks(e0.elapsed_time(e1), world, dev)
    value = aggregate_gbs(world, step_bytes, args.steps, ms_max)
    if rank == 0:
        peak, kind = measured_hbm_peak()
        print(json.dumps({
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_max / args.steps, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(workload=args.workload, psi=psi, step_bytes=step_bytes, **extra),
            "params_per_s": round(world * psi * args.steps / (ms_max * 1e-3), 1),
            "pct_of_8tbs": round(100.0 * value / (NOMINAL_HBM_GBS * world), 2),
            "frac_of_measured_peak": round(value / world / peak, 4), "peak_kind": kind,
            "clocks": clock_info, "gpu_launches": launches * args.steps}), flush=True)


def run_kernels(args, local):
    """Every device entry point alone on one layer (kernels_<layer workload>):
    mean CUDA-event time per call over rotating replicas, algorithmic GB/s
    and the fraction of the measured copy peak."""
    import torch
    from optimizer_state_gb300 import build as libbuild
    from optimizer_state_gb300 import inputs as I
    from optimizer_state_gb300 import schedule, z3
    libbuild.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    w = layer_workload(args.workload[len("kernels_"):])
    N = w.n_ranks
    reps = [schedule.Unit(w, dev, I.make_generator(i, dev)) for i in range(3)]
    L = reps[0].L
    L2 = z3.Layout(w.numel, 2 * N)
    bufs = [dict(full=torch.empty(L.psi, dtype=torch.bfloat16, device=dev),
                 gs=torch.zeros(L.psi_padded, dtype=torch.float32, device=dev),
                 gf=torch.empty(L.psi, dtype=torch.float32, device=dev),
                 rs=torch.empty(L2.psi_padded, dtype=torch.float32, device=dev),
                 p32=I.draw_master(w, I.make_generator(50 + i, dev), dev))
            for i in range(len(reps))]
    st = L.stats()
    psi = L.psi
    sc = 1.0 / N
    calls = {
        # the initial partition (once per run): reads 4 B of fp32, writes the
        # bf16 shard and fp32 master, m, v (14 B) per element
        "partition": (18 * psi, lambda u, b, t: z3.z3_partition(u.L, b["p32"], u.shards, u.master,
                                                               u.m, u.v)),
        "allgather": (st["hbm_allgather"], lambda u, b, t: z3.z3_allgather(u.L, u.shards, b["full"])),
        "reduce_scatter": (st["hbm_reduce_scatter"], lambda u, b, t: z3.z3_reduce_scatter(
            u.L, u.grads, w.grad_stride, b["gs"], sc)),
        "reduce_scatter_accumulate": (st["hbm_reduce_scatter_accumulate"],
                                      lambda u, b, t: z3.z3_reduce_scatter(
                                          u.L, u.grads, w.grad_stride, b["gs"], sc, accumulate=True)),
        "adam_shard_step": (st["hbm_adam"], lambda u, b, t: z3.z3_adam_shard_step(
            u.L, u.master, u.m, u.v, b["gs"], u.shards, HP, t)),
        "reduce_scatter_adam": (st["hbm_reduce_scatter_adam"], lambda u, b, t: z3.z3_reduce_scatter_adam(
            u.L, u.grads, w.grad_stride, sc, None, u.master, u.m, u.v, u.shards, HP, t)),
        "allreduce": ((2 * N + 4) * psi, lambda u, b, t: z3.z3_allreduce(
            u.L, u.grads, w.grad_stride, b["gf"], sc)),
        "scatter": (8 * psi, lambda u, b, t: z3.z3_scatter(u.L, b["gf"], b["gs"])),
        "reshard_fp32_to_2N": (8 * psi, lambda u, b, t: z3.z3_reshard(u.L, L2, u.master, b["rs"])),
    }
    peak, kind = measured_hbm_peak()
    out = {}
    for name, (nbytes, fn) in calls.items():
        for i in range(args.warmup):
            fn(reps[i % 3], bufs[i % 3], i + 1)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(args.steps):
            fn(reps[i % 3], bufs[i % 3], i + 1)
        e1.record()
        torch.cuda.synchronize()
        us = 1e3 * e0.elapsed_time(e1) / args.steps
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"us": round(us, 3), "gbs": round(gbs, 1),
                     "bytes_per_param": round(nbytes / psi, 3), "frac": round(gbs / peak, 4)}
    print(json.dumps({"workload": args.workload, "psi": psi, "n_ranks": N, "peak": peak,
                      "peak_kind": kind, "steps": args.steps,
                      "l2": "3 rotating replicas", "kernels": out}), flush=True)


def run_e2e(args, z3, L, w, rep, stream, sid, step_bytes, world):
    """The same step through the C ABI with host buffers (z3_host_step_run):
    every step uploads its gradients from page-locked host memory into one of
    two device staging buffers and reads the updated bf16 shards back into
    host memory, inside the timed region.  The library overlaps the upload
    of step i+1 with the compute and read-back of step i, ordering every
    buffer reuse with CUDA events."""
    import torch
    k = max(3, min(args.steps, args.e2e_steps))
    host_grads = torch.empty(rep.grads.shape, dtype=rep.grads.dtype, pin_memory=True)
    host_grads.copy_(rep.grads)
    host_out = torch.empty(rep.shards.shape, dtype=rep.shards.dtype, pin_memory=True)
    h2d = host_grads.numel() * host_grads.element_size()
    d2h = host_out.numel() * host_out.element_size()
    staging = [rep.grads, torch.empty_like(rep.grads)]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    pipe = z3.HostStep(L, staging[0], staging[1], w.grad_stride, up, down)

    def run(n):
        for _ in range(n):
            rep.step += 1
            pipe.run(host_grads, rep.shards, rep.full, 1.0 / w.n_ranks, rep.master, rep.m,
                     rep.v, HP, rep.step, shards_host=host_out, stream=sid)
        stream.wait_stream(down)                 # the last read-back is part of the step
        stream.wait_stream(up)
    run(2)
    torch.cuda.synchronize()
    link = host_link_h2d_gbs(host_grads, staging[1], up)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_event(e0)
    down.wait_event(e0)
    run(k)
    e1.record(stream)
    torch.cuda.synchronize()
    pipe.close()
    # the slowest rank's time: every rank runs this leg (world > 1 under torchrun)
    ms = max_over_ranks(e0.elapsed_time(e1), world, stream.device)
    value = aggregate_gbs(world, step_bytes, k, ms)
    # no step can finish faster than its upload: step bytes / (upload bytes / link rate)
    bound = world * step_bytes / (h2d / (link * 1e9)) / 1e9
    return {"value": round(value, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k,
            "ms_per_step": round(ms / k, 6),
            "api": "z3_host_step_run (C ABI, pinned host buffers)",
            "pipeline": "upload of step i+1 overlaps compute and read-back of step i",
            "host_link_h2d_gbs": round(link, 1), "upload_bound": round(bound, 2),
            "frac_of_upload_bound": round(value / bound, 4)}


def host_link_h2d_gbs(host, dev_buf, stream, reps: int = 5) -> float:
    """Pinned host -> device copy rate of one upload-sized buffer, timed
    with CUDA events on the copy stream (best of `reps`)."""
    import torch
    best = 0.0
    nbytes = host.numel() * host.element_size()
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        with torch.cuda.stream(stream):
            dev_buf.copy_(host, non_blocking=True)
        b.record(stream)
        b.synchronize()
        best = max(best, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    return best


# --------------------------------------------------------------------------
# the oracle on the host cores
# --------------------------------------------------------------------------

# Oracle calls timed per kernel, with their algorithmic bytes per unpadded
# element (the GPU kernels' accounting).
CPU_KERNELS = ("allgather", "reduce_scatter", "reduce_scatter_accumulate", "adam", "step_layer")


def cpu_bytes_per_elem(kernel: str, n_ranks: int) -> int:
    return {"allgather": 4, "reduce_scatter": 2 * n_ranks + 4,
            "reduce_scatter_accumulate": 2 * n_ranks + 8, "adam": 30,
            "step_layer": 2 * n_ranks + 34}[kernel]


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(w, n_elems: int, seed: int):
    """A bounded sample of the workload for the CPU oracle: the first
    n_elems elements of the layer's parameter list as one layer (same N_d,
    same value distributions)."""
    import numpy as np
    import torch
    from optimizer_state_gb300 import inputs as I
    numel, left = [], n_elems
    for n in w.numel:
        take = min(n, left)
        if take > 0:
            numel.append(take)
        left -= take
    sw = I.Workload(w.name + "_sample", tuple((n,) for n in numel), w.n_ranks, w.param_std,
                    w.grad_std)
    gen = I.make_generator(seed, "cpu")
    full = I.draw_master(sw, gen, "cpu").numpy()
    grads = I.draw_grads(sw, gen, "cpu").view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return sw, full, grads


class OraclePiece:
    """One thread's share of an oracle run over a sample: the contiguous
    range [a, b) of the sample's unpadded elements, as a one-parameter layer
    over the same N_d with its own state and gradient buffers.  The oracle's
    arithmetic is elementwise (plus the rank fold of each element), so a
    piece's elements end up with exactly the values they get when the
    oracle runs on the whole sample; only where they are stored differs."""

    def __init__(self, orc, sw, full, grads, a: int, b: int):
        import numpy as np
        from optimizer_state_gb300 import inputs as I
        n = b - a
        self.a, self.b, self.n = a, b, n
        self.O = orc.layout([n], sw.n_ranks)
        self.stride = I.grad_stride(n)
        self.grads = np.zeros(sw.n_ranks * self.stride, np.uint16)
        for k in range(sw.n_ranks):
            self.grads[k * self.stride:k * self.stride + n] = \
                grads[k * sw.grad_stride + a:k * sw.grad_stride + b]
        self.shards, self.master, self.m, self.v = orc.partition(
            self.O, np.ascontiguousarray(full[a:b]))
        self.gs = np.zeros(self.O.psi_padded, np.float32)
        self.scale = 1.0 / sw.n_ranks

    def run(self, orc, kernel: str, t: int):
        """One call of `kernel` on this piece (t: the Adam step number)."""
        if kernel == "allgather":
            orc.allgather(self.O, self.shards)
        elif kernel == "reduce_scatter":
            orc.reduce_scatter(self.O, self.grads, self.stride, self.scale, out=self.gs)
        elif kernel == "reduce_scatter_accumulate":
            orc.reduce_scatter(self.O, self.grads, self.stride, self.scale, out=self.gs,
                               accumulate=True)
        elif kernel == "adam":
            orc.adam(self.master, self.m, self.v, self.gs, self.shards, HP["lr"], HP["beta1"],
                     HP["beta2"], HP["eps"], HP["weight_decay"], t)
        elif kernel == "step_layer":
            orc.step_layer(self.O, self.shards, self.grads, self.stride, self.scale, self.master,
                           self.m, self.v, HP, t)
        else:
            raise ValueError(kernel)


def split_sample(orc, sample, cores: int) -> list:
    """The sample cut into min(cores, elements) near-equal contiguous pieces."""
    sw, full, grads = sample
    n = sw.psi
    c = max(1, min(cores, n))
    bounds = [n * i // c for i in range(c + 1)]
    return [OraclePiece(orc, sw, full, grads, bounds[i], bounds[i + 1]) for i in range(c)]


def run_pieces(orc, pieces, kernel: str, iters: int, t0: int) -> float:
    """Every piece runs `iters` calls of `kernel` (Adam steps t0, t0+1, ...)
    in its own thread; the oracle's C calls release the GIL.  Returns the
    wall time from the common start to the last thread's end."""
    if len(pieces) == 1:
        start = time.perf_counter()
        for i in range(iters):
            pieces[0].run(orc, kernel, t0 + i)
        return time.perf_counter() - start
    barrier = threading.Barrier(len(pieces) + 1)
    errors = []

    def work(p):
        barrier.wait()
        try:
            for i in range(iters):
                p.run(orc, kernel, t0 + i)
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)
    threads = [threading.Thread(target=work, args=(p,)) for p in pieces]
    for th in threads:
        th.start()
    barrier.wait()
    start = time.perf_counter()
    for th in threads:
        th.join()
    dt = time.perf_counter() - start
    if errors:
        raise errors[0]
    return dt


def time_kernel(orc, pieces, kernel: str, n_ranks: int, seconds: float, t0: int) -> dict:
    """One untimed call, then as many calls as fill about `seconds`."""
    t1 = run_pieces(orc, pieces, kernel, 1, t0)
    iters = max(1, min(10 ** 6, int(round(seconds / max(t1, 1e-6)))))
    dt = run_pieces(orc, pieces, kernel, iters, t0 + 1)
    n = sum(p.n for p in pieces)
    return dict(gbs=cpu_bytes_per_elem(kernel, n_ranks) * n * iters / dt / 1e9,
                params_per_s=n * iters / dt, iters=iters, seconds=dt, t_next=t0 + 1 + iters)


def cpu_baseline(seconds: float) -> dict:
    """The oracle, as it stands, on the full d=1024 layer: every kernel
    single-threaded and split over all host cores (one contiguous piece of
    the layer per thread), about seconds/10 each and seconds/4 for the layer
    step.  `value` is the layer step on all cores; `cores` the threads it
    used."""
    import oracle
    from optimizer_state_gb300 import inputs as I
    oracle.build()
    w = I.LAYER_D1024
    sample = oracle_sample(w, w.psi, seed=0)
    cores = host_cores()
    per_kernel = {}
    modes = (("single", 1), ("all_cores", cores))
    res = {}
    threads = {}
    for mode, c in modes:
        pieces = split_sample(oracle, sample, c)
        threads[mode] = len(pieces)
        t = 1
        for k in CPU_KERNELS:
            share = 0.25 if k == "step_layer" else 0.1
            r = time_kernel(oracle, pieces, k, w.n_ranks, seconds * share, t)
            t = r["t_next"]
            per_kernel.setdefault(k, {})[mode] = round(r["gbs"], 4)
            res[(mode, k)] = r
    step_all, step_one = res[("all_cores", "step_layer")], res[("single", "step_layer")]
    return {"value": round(step_all["gbs"], 4), "unit": "GB/s", "cores": threads["all_cores"],
            "kind": "oracle",
            "params_per_s": round(step_all["params_per_s"], 1),
            "single": {"value": round(step_one["gbs"], 4), "cores": 1,
                       "params_per_s": round(step_one["params_per_s"], 1)},
            "per_kernel_gbs": per_kernel,
            "sample": f"the full layer_d1024_nd8 layer (Psi={w.psi}); all_cores: "
                      f"{threads['all_cores']} threads, "
                      f"each running the unchanged oracle on one contiguous piece of the layer "
                      f"as its own one-parameter layer over N_d={w.n_ranks}; single: one thread; "
                      f"about {seconds * 0.1:.1f} s per kernel and mode, "
                      f"{seconds * 0.25:.1f} s for the layer step "
                      f"({step_all['iters']} all-core and {step_one['iters']} single layer steps)"}


def layer_config(name: str, w, L_psi: int, S: int) -> dict:
    """The config keys that name a layer workload; both arms report them."""
    return {"workload": name,
            "layer": " ".join("x".join(map(str, sh)) for sh in w.shapes),
            "psi": L_psi, "n_ranks": w.n_ranks, "S": S,
            "storage": "bf16 params/grads, fp32 master/m/v",
            "bytes_per_param": 2 * w.n_ranks + 34,
            "step_bytes": (2 * w.n_ranks + 34) * L_psi}


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm: each step is the layer step on a
    bounded sample of the d=1024 layer (the whole layer when the budget
    allows), split over all host cores as in cpu_baseline."""
    if rank != 0:
        return
    import oracle
    from optimizer_state_gb300 import inputs as I
    oracle.build()
    w = I.LAYER_D1024
    cores = host_cores()
    # size the per-step sample so that warmup + steps fit the time budget
    probe_n = 1 << 20
    probe = split_sample(oracle, oracle_sample(w, probe_n, seed=1), cores)
    per_elem_s = run_pieces(oracle, probe, "step_layer", 1, 1) / probe_n
    budget = args.reference_seconds / max(1, args.steps + args.warmup)
    n = int(min(w.psi, max(w.n_ranks * 8 * cores, budget / per_elem_s)))
    pieces = split_sample(oracle, oracle_sample(w, n, seed=0), cores)
    run_pieces(oracle, pieces, "step_layer", args.warmup, 1)
    dt = run_pieces(oracle, pieces, "step_layer", args.steps, 1 + args.warmup)
    gbs = (2 * w.n_ranks + 34) * n * args.steps / dt / 1e9
    O = oracle.layout(w.numel, w.n_ranks)
    config = layer_config("layer_d1024_nd8", w, O.psi, O.S)
    config["sample_psi"] = n
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(gbs, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * dt / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": config,
        "params_per_s": round(n * args.steps / dt, 1),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": len(pieces),
                         "kind": "oracle",
                         "sample": f"each step: the first {n} elements of the layer, cut into "
                                   f"{len(pieces)} contiguous pieces, each a one-parameter layer "
                                   f"over N_d={w.n_ranks} run by the unchanged oracle in its own "
                                   f"thread"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="layer_d1024_nd8",
                    help="layer_d1024_nd8 (default), layer_7b_nd8, layer_7b_nd64, "
                         "full_step_nd16[_prefetch[<D>]][_bucket<k>][_persist<T>], {dp,stage1,stage2}_d1024_nd8, "
                         "or sweep_n<N>_nd<R>")
    ap.add_argument("--kernel-steps", type=int, default=200,
                    help="iterations of the per-kernel event pass (layer workloads)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cold-bytes", type=int, default=1536 << 20,
                    help="total bytes of rotating state replicas")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="full-step, sweep and stage workloads: replay the timed steps as one "
                         "CUDA graph (layer workloads always do, unless --eager)")
    ap.add_argument("--eager", action="store_true",
                    help="layer workloads: time stream launches instead of one CUDA graph")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if world != args.gpus:
        if world == 1 and args.gpus > 1:
            sys.exit("--gpus N > 1 must be launched with torchrun (one process per GPU)")
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.workload in LAYER_WORKLOADS:
        run_cuda(args, world, rank, local)
    elif args.workload.startswith("kernels_"):
        run_kernels(args, local)
    else:
        run_multi(args, world, rank, local)


if __name__ == "__main__":
    main()
