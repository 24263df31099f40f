#!/usr/bin/env python3
"""Benchmark of the MoE routing + FP8 hot path on one GB300 (or N, as replicas).

One step is one pass of the whole path over the large-prefill workload
(T=65536 tokens, E=256 experts, top-8, hidden 7168):
    topk_gate -> route_map -> expand_cast_fp8 -> swiglu_cast_fp8 -> combine
The SwiGLU input is [T*k, 2*2048] bf16 (the SwiGLU workload's row shape, one
row per routed copy) and the combine input y is [T*k, 7168] bf16; both stand
in for the expert GEMM outputs, which this path does not compute.

`value` is the headline metric: routed tokens (T*k) per second through
route + expand + cast (topk_gate + route_map + expand_cast_fp8), timed with
CUDA events inside each step; `ms_per_step` is the whole step.  Inputs are
resident in HBM before timing; every input tensor but the 67 MB score matrix
is larger than L2, and the step moves ~19 GB, so nothing is L2-resident when a
step starts.

The printed JSON line is kept short: besides the contract's keys it carries
`configs`, one compact entry per benchmarked workload (the tiny and decode
batches, the skewed routing, the SwiGLU rows, the large prefill) with its time
and fraction of the measured HBM peak, and the rooflines of the step's and of
the headline's dominant kernels.  Everything else (per-op bytes, two-stream
and variant rows, decode tables, the copy kernel) goes to the JSON file that
`detail` names.

--impl reference times the CPU oracle (test infrastructure) on the same
metric and the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "routed tokens/s and achieved HBM GB/s (% of GB300 peak) for route+expand+cast"
UNIT = "routed tokens/s"
WORKLOAD = "prefill_64k"
SWIGLU_N = 2048
FALLBACK_HBM_GBS = 6800.0
DETAIL_DEFAULT = os.path.join("bench_out", "bench_detail.json")


# ---------------------------------------------------------------- helpers

def algorithmic_bytes(T, E, k, H, N=SWIGLU_N, M=None):
    """Bytes each op must move (reads + writes), per launch."""
    R = T * k
    G = H // 128
    M = R if M is None else M
    b = {
        "topk_gate": T * E * 4 + R * 8,
        "route_map": R * 4 + R * 8 + (2 * E + 1) * 4,
        "expand_cast_fp8": T * H * 2 + R * 4 + R * H + R * G * 4,
        "swiglu_cast_fp8": M * 2 * N * 2 + M * N + M * (N // 128) * 4,
        "combine": R * H * 2 + R * 4 + R * 4 + T * H * 2,
    }
    b["route_expand_cast"] = b["topk_gate"] + b["route_map"] + b["expand_cast_fp8"]
    return b


def config_dict(world: int, name: str = WORKLOAD) -> dict:
    """The benchmarked workload, named the same way by both arms."""
    from moe_routing_precision_gb300 import workloads
    w = workloads.WORKLOADS[name]
    return {"workload": f"{name}: T={w.T} E={w.E} k={w.k} H={w.H}, route+expand+cast",
            "T": w.T, "E": w.E, "k": w.k, "H": w.H, "seed": "rank",
            "parallelism": f"replicas x{world}, no collective",
            "l2": f"inputs > L2 (x {w.T * w.H * 2 / 1e9:.2f} GB)" if w.T * w.H * 2 > 129e6
                  else "x evicted from L2 by the rest of the step"}


# GB300's nominal HBM3e bandwidth per GPU as NVIDIA states it (context for the
# measured copy peak, which is what the fractions are taken against)
NOMINAL_HBM_GBS = 7900.0

KERNEL_OF_OP = {  # op -> (kernel name in ncu, source file), for E <= 256 and H <= 16384
    "topk_gate": ("topk_gate_sorted_kernel", "topk_gate.cu"),
    "expand_cast_fp8": ("expand_cast_bulk_kernel", "expand_cast.cu"),
    "swiglu_cast_fp8": ("swiglu_cast_kernel", "swiglu_cast.cu"),
    "combine": ("combine_kernel", "combine.cu"),
}


def source_sha(fname):
    """Hash of a kernel's source file and every header of the kernel tree
    (a change to any of them invalidates the recorded traffic)."""
    d = os.path.join(ROOT, "moe_routing_precision_gb300", "csrc")
    h = hashlib.sha256()
    for q in [fname] + sorted(f for f in os.listdir(d) if f.endswith(".cuh")):
        with open(os.path.join(d, q), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(op, units):
    """DRAM bytes per launch of `op`'s kernel for `units` units of work (tokens
    or rows), from the committed ncu summary, if it was taken on the current
    kernel source: the captured bytes per unit times `units`; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if op not in KERNEL_OF_OP or not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(KERNEL_OF_OP[op][0])
    if not rec or rec.get("source_sha") != source_sha(KERNEL_OF_OP[op][1]):
        return None
    return round(rec["dram_bytes_per_launch"] / rec["units"] * units)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        if p.get("hbm_gbs"):
            return float(p["hbm_gbs"]), "of measured"
    return FALLBACK_HBM_GBS, "of fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_seed(rank: int) -> int:
    """Weak scaling: every rank routes its own batch of the same shape, drawn
    from its own seed; the path needs no exchange between ranks."""
    return int(rank)


def max_over_ranks(v: float, world: int, device=None) -> float:
    """The slowest rank's time (the job's time); a control-plane collective
    only, outside every timed region."""
    if world == 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, seconds: float) -> float:
    """Units all ranks processed / the job's time."""
    return units_per_rank * world / seconds


# ---------------------------------------------------------------- GPU arm


# ---------------------------------------------------------------- GPU arm

def gpu_arm(args):
    import torch
    import torch.distributed as dist

    from moe_routing_precision_gb300 import ops, workloads
    from moe_routing_precision_gb300._build import build

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build()
    L = ops.lib()

    w = workloads.WORKLOADS[args.workload]
    T, E, k, H, R, G = w.T, w.E, w.k, w.H, w.R, w.G
    N = SWIGLU_N
    # weak scaling: every rank routes its own batch (seed = rank), no collective
    full = args.ops == "all"
    inp = workloads.make_inputs(w, seed=shard_seed(rank), device=dev, with_y=full, with_swiglu=full,
                                swiglu_rows=R, swiglu_n=N)
    ran = {"topk_gate", "route_map", "expand_cast_fp8"} | \
        ({"swiglu_cast_fp8", "combine"} if full else set())
    scores, x = inp["scores"], inp["x"]
    y, hx = inp.get("y"), inp.get("swiglu_x")
    i32 = dict(dtype=torch.int32, device=dev)
    idx = torch.empty(T, k, **i32)
    wt = torch.empty(T, k, dtype=torch.float32, device=dev)
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    pos, src = torch.empty(T, k, **i32), torch.empty(R, **i32)
    ws = torch.empty(max(1, ops.route_map_workspace_bytes(T, E, k)), dtype=torch.uint8, device=dev)
    ws1 = ops.route_expand_cast_workspace(T, E, k, x)   # the one-call path's (zeroed once)
    q = torch.empty(R, H, dtype=torch.uint8, device=dev)
    sf = torch.empty(R, G, dtype=torch.float32, device=dev)
    if full:
        q2 = torch.empty(R, N, dtype=torch.uint8, device=dev)
        sf2 = torch.empty(R, N // 128, dtype=torch.float32, device=dev)
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream or None

    def chk(rc, what):
        if rc != 0:
            raise ops.MoeError(rc, what)

    def route_expand_cast(p=sp):
        """topk_gate + route_map + expand_cast_fp8 as a caller runs them: the
        one-call entry point (AUTO: the separate launches at this size), or
        with --headline-path calls the three individual calls."""
        if args.headline_path == "calls":
            chk(L.moe_topk_gate(scores.data_ptr(), T, E, k, idx.data_ptr(), wt.data_ptr(), 1, p),
                "topk")
            chk(L.moe_route_map(idx.data_ptr(), T, E, k, counts.data_ptr(), offsets.data_ptr(),
                                pos.data_ptr(), src.data_ptr(), ws.data_ptr(), ws.numel(), p),
                "route")
            chk(L.moe_expand_cast_fp8(x.data_ptr(), T, H, k, pos.data_ptr(), R, q.data_ptr(),
                                      sf.data_ptr(), 128, p), "expand")
        else:
            chk(L.moe_route_expand_cast_fp8(scores.data_ptr(), T, E, k, x.data_ptr(), H,
                                            idx.data_ptr(), wt.data_ptr(), counts.data_ptr(),
                                            offsets.data_ptr(), pos.data_ptr(), src.data_ptr(),
                                            q.data_ptr(), sf.data_ptr(), ws1.data_ptr(),
                                            ws1.numel(), ops.PATH_AUTO, 128, p), "route_expand_cast")

    def step(ev=None, split=True):
        """One step.  ev: 2 events around route + expand + cast (the timed
        steps), or, split, 6 events around each op with the route + expand +
        cast run as the three individual calls (the per-op breakdown, in
        separate steps: an event between two kernels ends their
        programmatic-dependent-launch overlap)."""
        def rec(i):
            if ev and (split or i in (0, 3)):
                ev[i if split else (0 if i == 0 else 1)].record(stream)
        rec(0)
        if split:
            chk(L.moe_topk_gate(scores.data_ptr(), T, E, k, idx.data_ptr(), wt.data_ptr(), 1, sp),
                "topk")
            rec(1)
            chk(L.moe_route_map(idx.data_ptr(), T, E, k, counts.data_ptr(), offsets.data_ptr(),
                                pos.data_ptr(), src.data_ptr(), ws.data_ptr(), ws.numel(), sp),
                "route")
            rec(2)
            chk(L.moe_expand_cast_fp8(x.data_ptr(), T, H, k, pos.data_ptr(), R, q.data_ptr(),
                                      sf.data_ptr(), 128, sp), "expand")
        else:
            route_expand_cast()
        rec(3)
        if full:
            chk(L.swiglu_cast_fp8(hx.data_ptr(), R, N, q2.data_ptr(), sf2.data_ptr(), 128, sp),
                "swiglu")
        rec(4)
        if full:
            chk(L.moe_combine(y.data_ptr(), wt.data_ptr(), pos.data_ptr(), T, H, k, R,
                              out.data_ptr(), 0, sp), "combine")
        rec(5)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    if L.moe_get_device_status(sp, None) != 0:
        raise RuntimeError("device error flagged during warm-up")

    # ---- timed region: exactly K steps
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    launches0 = L.moe_kernel_launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(K):
        step(evs[i], split=False)
    t_end.record(stream)
    barrier()
    launches = L.moe_kernel_launch_count() - launches0
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    rec_ms = [e[0].elapsed_time(e[1]) for e in evs]
    # per-op breakdown: separate instrumented steps after the timed region
    ops_names = ["topk_gate", "route_map", "expand_cast_fp8", "swiglu_cast_fp8", "combine"]
    per_op = {n: [] for n in ops_names}
    kb = min(K, 20)
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(kb)]
    for i in range(kb):
        step(evb[i], split=True)
    torch.cuda.synchronize(dev)
    for e in evb:
        for j, n in enumerate(ops_names):
            per_op[n].append(e[j].elapsed_time(e[j + 1]))
    if L.moe_get_device_status(sp, None) != 0:
        raise RuntimeError("device error flagged during the timed region")

    def maxr(v):
        return max_over_ranks(v, world, dev)

    step_ms = maxr(total_ms / K)
    rec_ms_mean = maxr(sum(rec_ms) / K)
    op_ms = {n: maxr(sum(v) / kb) for n, v in per_op.items()}

    # ---- e2e: the same metric through the C ABI from pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = e2e_leg(args, L, dev, stream, sp, scores, x, idx, wt, counts, offsets, pos, src,
                      ws1, q, sf, T, E, k, H, R, chk, barrier, maxr)

    peak, peak_src = load_peaks()
    # ---- the other workloads: compact per-config entries + detail (rank 0)
    summaries, detail = {}, {}
    if rank == 0 and not args.no_extra:
        summaries, detail = other_configs(L, dev, stream, sp, chk, args, peak)
        detail["peak_copy_GB_s"] = measure_peak_copy(L, dev, stream, sp)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_leg(scores, x, k, E, total=T)

    if world > 1:
        dist.barrier()
    if rank != 0:
        dist.destroy_process_group()
        return None

    B = algorithmic_bytes(T, E, k, H, N, R)
    breakdown = {}
    for n in ops_names:
        if n not in ran:
            continue
        ms = op_ms[n]
        gbs = B[n] / (ms * 1e-3) / 1e9
        breakdown[n] = {"ms": round(ms, 4), "algorithmic_bytes": B[n], "GB_s": round(gbs, 1),
                        "frac_of_peak": round(gbs / peak, 4)}
    rec_gbs = B["route_expand_cast"] / (rec_ms_mean * 1e-3) / 1e9
    units = {"topk_gate": T, "expand_cast_fp8": T, "swiglu_cast_fp8": R, "combine": T}

    def roofline(op):
        gbs = B[op] / (op_ms[op] * 1e-3) / 1e9
        return {"bound": "hbm", "kernel": KERNEL_OF_OP[op][0], "achieved": round(gbs, 1),
                "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4), "peak_source": peak_src,
                "traffic": ncu_traffic(op, units[op]), "ms": round(op_ms[op], 4)}

    dom = max((n for n in ops_names if n in KERNEL_OF_OP and n in ran), key=lambda n: op_ms[n])
    head_dom = max(("topk_gate", "expand_cast_fp8"), key=lambda n: op_ms[n])
    value = job_throughput(R, world, rec_ms_mean * 1e-3)
    head_key = "c4_prefill_64k" if w.name == WORKLOAD else f"timed_{w.name}"
    summaries[head_key] = {"ms": round(rec_ms_mean, 4), "frac": round(rec_gbs / peak, 4)}
    if full:
        summaries[head_key]["combine_frac"] = breakdown["combine"]["frac_of_peak"]
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e4m3",
        "data": "synthetic (seeded, no dataset)",
        "config": config_dict(world, w.name),
        "roofline": roofline(dom),
        "roofline_headline": roofline(head_dom),
        "configs": summaries,
        "configs_note": "c0-c3 ms/us: one batch after a 512 MB L2 flush, median; sus: back to "
                        "back, inputs not in L2, mean; c4: the timed steps; frac of measured peak",
        "cpu_baseline": None if cpu is None else {
            "value": cpu["value"], "unit": UNIT, "cores": cpu["cores"], "kind": "oracle",
            "sample": cpu["sample_short"]},
        "e2e": None if e2e is None else {
            "value": e2e["value"], "unit": UNIT, "ms_per_step": e2e["ms_per_step"],
            "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
            "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
            "link_bound_ms": e2e["link"]["copy_bound_ms_per_step"],
            "link_both_ms": e2e["link"]["both_directions_ms_per_step"]},
        "gpu_launches": int(launches),
        "clocks": clk,
        "detail": None,
    }
    detail.update({
        "line": {k2: v for k2, v in line.items() if k2 != "detail"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "breakdown": breakdown,
        "breakdown_timing": "per-op CUDA events in separate steps after the timed region (an "
                            "event between two kernels ends their launch overlap, so the "
                            "timed steps bracket only topk+route+expand and the whole step)",
        "route_expand_cast": {"ms": round(rec_ms_mean, 4), "GB_s": round(rec_gbs, 1),
                              "frac_of_peak": round(rec_gbs / peak, 4),
                              "frac_of_nominal": round(rec_gbs / NOMINAL_HBM_GBS, 4),
                              "algorithmic_bytes": B["route_expand_cast"],
                              "tokens_per_s": round(T * world / (rec_ms_mean * 1e-3), 1),
                              "routed_rows_per_s": round(R * world / (rec_ms_mean * 1e-3), 1)},
        "step_routed_tokens_per_s": round(R * world / (step_ms * 1e-3), 1),
    })
    if args.detail_out:
        try:
            os.makedirs(os.path.dirname(os.path.abspath(args.detail_out)), exist_ok=True)
            with open(args.detail_out, "w") as f:
                json.dump(detail, f, indent=1)
            line["detail"] = args.detail_out
        except OSError:
            line["detail"] = None
    return line


def gpu_numa_cpus(dev):
    """(NUMA node, its CPU ids) of the host memory attached to `dev`, from
    sysfs; (None, None) where the system does not say."""
    import torch
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id.lower()
        dom, rest = bus.split(":", 1)
        path = f"/sys/bus/pci/devices/{int(dom, 16):04x}:{rest}/numa_node"
        node = int(open(path).read().strip())
        if node < 0:
            return None, None
        cpus = []
        for part in open(f"/sys/devices/system/node/node{node}/cpulist").read().strip().split(","):
            a, _, b = part.partition("-")
            cpus.extend(range(int(a), int(b or a) + 1))
        return node, cpus
    except (OSError, ValueError, AttributeError, RuntimeError):
        return None, None


def e2e_leg(args, L, dev, stream, sp, scores, x, idx, wt, counts, offsets, pos, src, ws, q, sf,
            T, E, k, H, R, chk, barrier, maxr):
    """route+expand+cast with the inputs copied from pinned host memory and
    every output copied back to pinned host memory, all inside the timing.
    Consecutive steps alternate between two streams, each with its own device
    and host buffers, so one step's device-to-host copy overlaps the next
    step's host-to-device copy and kernels (as a caller streaming batches
    would run it); every step still makes all of its own copies."""
    import torch
    # pinned host buffers on the NUMA node the GPU is attached to: the thread
    # runs there while it allocates and touches them (first touch places the
    # pages); a buffer on the other socket crosses the socket link
    node, cpus = gpu_numa_cpus(dev)
    old_aff = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
    if cpus and old_aff is not None:
        try:
            os.sched_setaffinity(0, cpus)
        except OSError:
            node = None
    h_scores = torch.empty_like(scores, device="cpu").pin_memory()
    h_x = torch.empty_like(x, device="cpu").pin_memory()
    h_scores.copy_(scores)
    h_x.copy_(x)
    names = ["scores", "x", "idx", "wt", "counts", "offsets", "pos", "src", "ws", "q", "sf"]
    slot0 = dict(zip(names, [scores, x, idx, wt, counts, offsets, pos, src, ws, q, sf]))
    # ws: the one-call path's workspace, whose control words start at zero
    slots = [slot0, {n: (torch.zeros_like if n == "ws" else torch.empty_like)(t)
                     for n, t in slot0.items()}]
    out_names = ["idx", "wt", "counts", "offsets", "pos", "src", "q", "sf"]
    h_outs = [[torch.empty_like(sl[n], device="cpu").pin_memory() for n in out_names]
              for sl in slots]
    for hs in h_outs:
        for h in hs:
            h.zero_()  # touch every page now, on this node
    streams = [torch.cuda.Stream(device=dev) for _ in slots]
    h2d = h_scores.numel() * 4 + h_x.numel() * 2
    d2h = sum(slot0[n].numel() * slot0[n].element_size() for n in out_names)
    # the first step's H2D and kernels (about 5.5 ms at prefill size) precede
    # any D2H inside the timed region; over N steps that adds 5.5/N ms a step
    steps = max(4, args.e2e_steps)

    def one(i):
        sl, st = slots[i % 2], streams[i % 2]
        p = st.cuda_stream
        with torch.cuda.stream(st):
            sl["scores"].copy_(h_scores, non_blocking=True)
            sl["x"].copy_(h_x, non_blocking=True)
            chk(L.moe_route_expand_cast_fp8(
                sl["scores"].data_ptr(), T, E, k, sl["x"].data_ptr(), H, sl["idx"].data_ptr(),
                sl["wt"].data_ptr(), sl["counts"].data_ptr(), sl["offsets"].data_ptr(),
                sl["pos"].data_ptr(), sl["src"].data_ptr(), sl["q"].data_ptr(), sl["sf"].data_ptr(),
                sl["ws"].data_ptr(), sl["ws"].numel(), 0, 128, p), "route_expand_cast")
            for h, n in zip(h_outs[i % 2], out_names):
                h.copy_(sl[n], non_blocking=True)

    one(0)
    one(1)
    barrier()
    clk = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clk.start()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for st in streams:
        st.wait_event(a)
    step_ends = []
    for i in range(steps):
        one(i)
        ev = torch.cuda.Event(enable_timing=True)
        ev.record(streams[i % 2])
        step_ends.append(ev)
    for st in streams:
        ev = torch.cuda.Event()
        ev.record(st)
        stream.wait_event(ev)
    b.record(stream)
    barrier()
    e2e_clocks = clk.stop()
    ends = [a.elapsed_time(ev) for ev in step_ends]
    ms = maxr(a.elapsed_time(b) / steps)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    # the host link on its own, for context: the largest output alone back to
    # pinned host memory, and x alone to the device (best of 3 each)
    qd, qh = slots[0]["q"], h_outs[0][out_names.index("q")]

    def copy_ms(dst, src):
        best = float("inf")
        for _ in range(3):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            with torch.cuda.stream(stream):
                dst.copy_(src, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        return best

    d2h_gbs = qd.numel() / (copy_ms(qh, qd) * 1e-3) / 1e9
    h2d_gbs = h_x.numel() * 2 / (copy_ms(slots[0]["x"], h_x) * 1e-3) / 1e9
    bound_ms = max(d2h / (d2h_gbs * 1e9), h2d / (h2d_gbs * 1e9)) * 1e3

    # one step's copies alone, both directions at once as the two-stream
    # steps run them (every output of slot 0 back, the inputs of slot 1 in):
    # the link's own time for a step, with the two directions sharing it
    def both_ms():
        best = float("inf")
        for _ in range(3):
            e0 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for st in streams:
                st.wait_event(e0)
            with torch.cuda.stream(streams[0]):
                for h, n in zip(h_outs[0], out_names):
                    h.copy_(slots[0][n], non_blocking=True)
            with torch.cuda.stream(streams[1]):
                slots[1]["scores"].copy_(h_scores, non_blocking=True)
                slots[1]["x"].copy_(h_x, non_blocking=True)
            for st in streams:
                ev = torch.cuda.Event()
                ev.record(st)
                stream.wait_event(ev)
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record(stream)
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        return best

    both = both_ms()
    del slots, h_outs
    if cpus and old_aff is not None:
        os.sched_setaffinity(0, old_aff)
    return {"value": round(R * world / (ms * 1e-3), 1), "unit": UNIT, "ms_per_step": round(ms, 3),
            "steps": steps, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "host_numa_node": node, "clocks": e2e_clocks,
            "step_end_ms": [round(v, 2) for v in ends],
            "step_ms_median": round(statistics.median(
                [ends[0]] + [ends[i] - ends[i - 1] for i in range(1, len(ends))]), 3),
            "link": {"d2h_GB_s": round(d2h_gbs, 1), "h2d_GB_s": round(h2d_gbs, 1),
                     "copy_bound_ms_per_step": round(bound_ms, 3),
                     "both_directions_ms_per_step": round(both, 3),
                     "note": "d2h/h2d: one direction at a time, best of 3; copy_bound: the "
                             "slower direction's time for a step's bytes; both_directions: a "
                             "step's outputs back while the next step's inputs go in, copies "
                             "only, best of 3 (the link is shared by the two directions)"},
            "path": "pinned host -> device, C ABI moe_route_expand_cast_fp8 (AUTO), "
                    "all outputs -> pinned host; steps alternate between two streams"}


def measure_peak_copy(L, dev, stream, sp):
    import torch
    n = 1 << 30  # 1 GiB each way
    a = torch.empty(n, dtype=torch.uint8, device=dev)
    b = torch.empty(n, dtype=torch.uint8, device=dev)
    a.fill_(1)
    best = 0.0
    for _ in range(3):
        L.moe_peak_copy(a.data_ptr(), b.data_ptr(), n, sp)
    for _ in range(10):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        L.moe_peak_copy(a.data_ptr(), b.data_ptr(), n, sp)
        e1.record(stream)
        e1.synchronize()
        best = max(best, 2 * n / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del a, b
    return round(best, 1)


def other_configs(L, dev, stream, sp, chk, args, peak):
    """The other benchmarked workloads, on rank 0: the tiny and decode
    batches, the skewed routing and the SwiGLU rows, each with a compact
    summary for the printed line; and the variant rows (two streams, the
    padded layout, the scale options, FP4, more decode sizes) for the detail
    file.  Each single-batch time is taken after an L2 flush (a 512 MB
    device write outside the timed events), median of the iterations."""
    import torch

    from moe_routing_precision_gb300 import ops, workloads
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    iters = args.extra_iters
    summ, det = {}, {}

    def timed(fn, n=iters):
        ts = []
        for i in range(n + 3):
            flush.fill_(i & 0xFF)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    def back_to_back(fn, reps):
        """Mean time per call of `reps` calls back to back (one before, untimed)."""
        fn(0)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(reps):
            fn(i)
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps

    def frac(b, ms):
        return round(b / (ms * 1e-3) / 1e9 / peak, 4)

    def route_bufs(T, E, k, H):
        R, G = T * k, H // 128
        i32 = dict(dtype=torch.int32, device=dev)
        return dict(idx=torch.empty(T, k, **i32), wt=torch.empty(T, k, device=dev),
                    counts=torch.empty(E, **i32), offsets=torch.empty(E + 1, **i32),
                    pos=torch.empty(T, k, **i32), src=torch.empty(R, **i32),
                    ws=torch.empty(max(1, ops.route_map_workspace_bytes(T, E, k)),
                                   dtype=torch.uint8, device=dev),
                    ws1=torch.zeros(L.moe_route_expand_cast_fp8_workspace_bytes(T, E, k),
                                    dtype=torch.uint8, device=dev),
                    q=torch.empty(R, H, dtype=torch.uint8, device=dev),
                    sf=torch.empty(R, G, device=dev))

    def rec_call(b, s, x, T, E, k, H, p=sp, calls=False, mode=None):
        """topk_gate + route_map + expand_cast_fp8: the one-call entry point
        (AUTO, or `mode`), or with calls=True the three individual C-ABI calls."""
        if not calls:
            chk(L.moe_route_expand_cast_fp8(s.data_ptr(), T, E, k, x.data_ptr(), H,
                                            b["idx"].data_ptr(), b["wt"].data_ptr(),
                                            b["counts"].data_ptr(), b["offsets"].data_ptr(),
                                            b["pos"].data_ptr(), b["src"].data_ptr(),
                                            b["q"].data_ptr(), b["sf"].data_ptr(),
                                            b["ws1"].data_ptr(), b["ws1"].numel(),
                                            ops.PATH_AUTO if mode is None else mode, 128, p),
                "route_expand_cast")
            return
        chk(L.moe_topk_gate(s.data_ptr(), T, E, k, b["idx"].data_ptr(), b["wt"].data_ptr(), 1, p),
            "topk")
        chk(L.moe_route_map(b["idx"].data_ptr(), T, E, k, b["counts"].data_ptr(),
                            b["offsets"].data_ptr(), b["pos"].data_ptr(), b["src"].data_ptr(),
                            b["ws"].data_ptr(), b["ws"].numel(), p), "route")
        chk(L.moe_expand_cast_fp8(x.data_ptr(), T, H, k, b["pos"].data_ptr(), T * k,
                                  b["q"].data_ptr(), b["sf"].data_ptr(), 128, p), "expand")

    def two_stream_batches(T, E, k, H, sets, reps):
        """Device time per batch of topk + route_map + expand_cast_fp8 with
        consecutive batches on two streams, each stream with its own routing
        and output buffers: every batch does all of its own work, and one
        batch's latency-bound routing overlaps the other's expand."""
        bufs = [route_bufs(T, E, k, H) for _ in range(2)]
        streams = [torch.cuda.Stream(device=dev) for _ in range(2)]

        def one(i):
            si, xi = sets[i % len(sets)]
            rec_call(bufs[i % 2], si, xi, T, E, k, H, streams[i % 2].cuda_stream)

        for i in range(4):
            one(i)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for st in streams:
            st.wait_event(e0)
        for i in range(reps):
            one(i)
        for st in streams:
            ev = torch.cuda.Event()
            ev.record(st)
            stream.wait_event(ev)
        e1.record(stream)
        e1.synchronize()
        if L.moe_get_device_status(sp, None) != 0:
            raise RuntimeError("device error in the two-stream batches")
        del bufs
        return e0.elapsed_time(e1) / reps

    # ---- configs[0], configs[1]: the tiny and decode batches through the
    # one-call entry point (AUTO: the path measured fastest for the shape)
    for key, name in (("c0_tiny", "tiny"), ("c1_decode_1k", "decode_1k")):
        w = workloads.WORKLOADS[name]
        d = decode_workload(L, dev, stream, sp, chk, flush, iters, peak, w=w)
        det[name] = d
        auto = d["auto"]
        summ[key] = {"us": auto["us"], "frac": auto["frac_of_peak"]}

    # ---- configs[2]: skewed routing (and its mild-skew variant, detail only)
    def skewed(name):
        w = workloads.WORKLOADS[name]
        inp = workloads.make_inputs(w, seed=0, device=dev, with_y=(name == "skewed_8k"))
        s, x = inp["scores"], inp["x"]
        T, E, k, H, R = w.T, w.E, w.k, w.H, w.R
        b = route_bufs(T, E, k, H)
        B = algorithmic_bytes(T, E, k, H)
        ms = timed(lambda: rec_call(b, s, x, T, E, k, H))
        ms_c = timed(lambda: rec_call(b, s, x, T, E, k, H, calls=True))
        ms_ch = timed(lambda: rec_call(b, s, x, T, E, k, H, mode=ops.PATH_CHAINED))
        ms_e = timed(lambda: chk(L.moe_expand_cast_fp8(x.data_ptr(), T, H, k, b["pos"].data_ptr(),
                                                       R, b["q"].data_ptr(), b["sf"].data_ptr(),
                                                       128, sp), "expand"))
        # sustained: back-to-back batches over NSETS independent input sets
        # (seeds 0..NSETS-1), so each batch's inputs were last touched NSETS-1
        # batches (~1.8 GB of traffic) ago and are no longer in L2
        nsets = 4
        sets = [(s, x)] + [(d["scores"], d["x"]) for d in
                           (workloads.make_inputs(w, seed=i, device=dev) for i in range(1, nsets))]
        reps = max(8, 2 * iters)
        ms_s = back_to_back(lambda i: rec_call(b, sets[i % nsets][0], sets[i % nsets][1], T, E, k, H),
                            reps)
        ms_2 = two_stream_batches(T, E, k, H, sets, reps)
        r = {"single_ms": round(ms, 4), "single_frac": frac(B["route_expand_cast"], ms),
             "single_calls_ms": round(ms_c, 4),
             "single_calls_frac": frac(B["route_expand_cast"], ms_c),
             "single_chained_ms": round(ms_ch, 4),
             "single_chained_frac": frac(B["route_expand_cast"], ms_ch),
             "sustained_ms": round(ms_s, 4), "sustained_frac": frac(B["route_expand_cast"], ms_s),
             "two_streams_ms": round(ms_2, 4),
             "two_streams_frac": frac(B["route_expand_cast"], ms_2),
             "expand_only_ms": round(ms_e, 4), "expand_only_frac": frac(B["expand_cast_fp8"], ms_e),
             "skew": workloads.skew_stats(b["counts"].cpu()),
             "timing": "single: one batch after a 512 MB L2 flush, median (the one-call entry "
                       "point, AUTO; single_calls: the three individual calls); sustained: batches "
                       f"back to back over {nsets} input sets (inputs not in L2), mean; two "
                       "streams: consecutive batches on two streams with their own buffers, mean"}
        if "y" in inp:
            out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
            ms_cb = timed(lambda: chk(L.moe_combine(inp["y"].data_ptr(), b["wt"].data_ptr(),
                                                   b["pos"].data_ptr(), T, H, k, R, out.data_ptr(),
                                                   0, sp), "combine"))
            r["combine_ms"] = round(ms_cb, 4)
            r["combine_frac"] = frac(B["combine"], ms_cb)
        del inp, sets, b
        torch.cuda.empty_cache()
        return r

    det["skewed_8k"] = sk = skewed("skewed_8k")
    summ["c2_skewed_8k"] = {
        "ms": sk["single_ms"], "frac": sk["single_frac"], "sus_ms": sk["sustained_ms"],
        "sus_frac": sk["sustained_frac"], "combine_frac": sk.get("combine_frac"),
        "experts_half": sk["skew"]["experts_taking_half"], "empty": sk["skew"]["empty_experts"]}
    det["skewed_8k_mild"] = skewed("skewed_8k_mild")

    # ---- configs[3]: SwiGLU rows
    w = workloads.WORKLOADS["swiglu_64k"]
    hx = workloads.make_inputs(w, seed=0, device=dev)["swiglu_x"]
    M, N = w.M, w.N
    q2 = torch.empty(M, N, dtype=torch.uint8, device=dev)
    sf2 = torch.empty(M, N // 128, dtype=torch.float32, device=dev)

    def sw(i=0):
        chk(L.swiglu_cast_fp8(hx.data_ptr(), M, N, q2.data_ptr(), sf2.data_ptr(), 128, sp), "swiglu")

    ms = timed(sw)
    bsw = M * 2 * N * 2 + M * N + M * (N // 128) * 4
    # sustained: back to back; the 537 MB input exceeds L2, so each pass
    # starts on lines the previous pass evicted
    ms_s = back_to_back(sw, max(8, 2 * iters))
    det["swiglu_64k"] = {"single_ms": round(ms, 4), "single_frac": frac(bsw, ms),
                         "sustained_ms": round(ms_s, 4), "sustained_frac": frac(bsw, ms_s),
                         "rows_per_s": round(M / (ms * 1e-3), 1), "algorithmic_bytes": bsw}
    summ["c3_swiglu_64k"] = {"ms": round(ms, 4), "frac": frac(bsw, ms), "sus_ms": round(ms_s, 4),
                             "sus_frac": frac(bsw, ms_s)}
    del hx, q2, sf2
    torch.cuda.empty_cache()

    # ---- detail only: the large prefill on two streams, the padded layout,
    # the scale options and FP4, more decode sizes
    wp = workloads.WORKLOADS[WORKLOAD]
    pin = workloads.make_inputs(wp, seed=0, device=dev)
    reps_p = max(8, iters)
    ms_p = two_stream_batches(wp.T, wp.E, wp.k, wp.H, [(pin["scores"], pin["x"])], reps_p)
    Bp = algorithmic_bytes(wp.T, wp.E, wp.k, wp.H)["route_expand_cast"]
    det[f"{WORKLOAD}_two_streams"] = {"ms": round(ms_p, 4), "frac": frac(Bp, ms_p),
                                      "timing": f"{reps_p} steps on two streams, mean per step"}
    del pin
    torch.cuda.empty_cache()
    det["prefill_64k_padded"] = padded_workload(L, dev, stream, sp, chk, flush, iters, peak)
    torch.cuda.empty_cache()
    det.update(cast_options_workloads(L, dev, stream, sp, chk, flush, iters, peak))
    torch.cuda.empty_cache()
    base = workloads.WORKLOADS["decode_1k"]
    for t in (64, 256):
        det[f"decode_{t}"] = decode_workload(
            L, dev, stream, sp, chk, flush, iters, peak,
            w=workloads.Workload(f"decode_{t}", T=t, E=base.E, k=base.k, H=base.H))
    del flush
    torch.cuda.empty_cache()
    return summ, det


def padded_workload(L, dev, stream, sp, chk, flush, iters, peak, align=128):
    """route + expand + cast into the padded layout (each expert's segment
    rounded up to `align` rows, the rest zero-filled in the expand's launch),
    on the large-prefill inputs, with the buffers sized for the worst case
    (T*k + E*(align-1) rows), as a caller without a host sync must."""
    import torch

    from moe_routing_precision_gb300 import ops, workloads
    w = workloads.WORKLOADS[WORKLOAD]
    inp = workloads.make_inputs(w, seed=0, device=dev)
    s, x = inp["scores"], inp["x"]
    T, E, k, H, R, G = w.T, w.E, w.k, w.H, w.R, w.G
    NR = R + E * (align - 1)
    i32 = dict(dtype=torch.int32, device=dev)
    idx, wt = torch.empty(T, k, **i32), torch.empty(T, k, dtype=torch.float32, device=dev)
    counts, offsets, pos, src = (torch.empty(E, **i32), torch.empty(E + 1, **i32),
                                 torch.empty(T, k, **i32), torch.empty(NR, **i32))
    ws = torch.empty(max(1, ops.route_map_workspace_bytes(T, E, k)), dtype=torch.uint8, device=dev)
    q = torch.empty(NR, H, dtype=torch.uint8, device=dev)
    sf = torch.empty(NR, G, dtype=torch.float32, device=dev)

    def rec():
        chk(L.moe_topk_gate(s.data_ptr(), T, E, k, idx.data_ptr(), wt.data_ptr(), 1, sp), "topk")
        chk(L.moe_route_map_aligned(idx.data_ptr(), T, E, k, align, NR, counts.data_ptr(),
                                    offsets.data_ptr(), pos.data_ptr(), src.data_ptr(),
                                    ws.data_ptr(), ws.numel(), sp), "route")
        chk(L.moe_expand_cast_fp8_padded(x.data_ptr(), T, H, k, pos.data_ptr(), src.data_ptr(),
                                         NR, q.data_ptr(), sf.data_ptr(), 128, sp), "expand")

    ts = []
    for i in range(max(3, iters // 2) + 2):
        flush.fill_(i & 0xFF)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        rec()
        e1.record(stream)
        e1.synchronize()
        if i >= 2:
            ts.append(e0.elapsed_time(e1))
    ms = statistics.median(ts)
    if L.moe_get_device_status(sp, None) != 0:
        raise RuntimeError("device error in the padded workload")
    padded_total = int(offsets[E].item())
    zero_rows = NR - R
    B = algorithmic_bytes(T, E, k, H)
    # plus: sorted_src -1 entries, the expand's scan of sorted_src, zeroed rows
    b = B["route_expand_cast"] + zero_rows * 4 + NR * 4 + zero_rows * (H + 4 * G)
    gbs = b / (ms * 1e-3) / 1e9
    del inp, s, x, q, sf
    return {"op": "topk + route_map_aligned + expand_cast_fp8_padded", "align": align,
            "rows": NR, "padded_total": padded_total, "zero_filled_rows": zero_rows,
            "ms": round(ms, 4), "routed_tokens_per_s": round(R / (ms * 1e-3), 1),
            "algorithmic_bytes": b, "GB_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
            "timing": "one batch after a 512 MB L2 flush, median"}


def cast_options_workloads(L, dev, stream, sp, chk, flush, iters, peak):
    """The cast variants on the large-prefill and SwiGLU workloads: scales as
    packed UE8M0 exponents in the TMA-aligned column-major layout (flags
    COLMAJOR | POW2 | UE8M0); the SwiGLU with clamp 7.0, per-row weights and
    the clamp counter as well.  One batch after an L2 flush, median."""
    import torch

    from moe_routing_precision_gb300 import ops, workloads
    flags = ops.SF_COLMAJOR | ops.SF_POW2 | ops.SF_UE8M0

    def timed(fn, n):
        ts = []
        for i in range(n + 2):
            flush.fill_(i & 0xFF)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if i >= 2:
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    res = {}
    w = workloads.WORKLOADS[WORKLOAD]
    inp = workloads.make_inputs(w, seed=0, device=dev)
    s, x = inp["scores"], inp["x"]
    T, E, k, H, R, G = w.T, w.E, w.k, w.H, w.R, w.G
    ld = (R + 3) // 4 * 4
    i32 = dict(dtype=torch.int32, device=dev)
    idx, wt = torch.empty(T, k, **i32), torch.empty(T, k, dtype=torch.float32, device=dev)
    counts, offsets, pos, src = (torch.empty(E, **i32), torch.empty(E + 1, **i32),
                                 torch.empty(T, k, **i32), torch.empty(R, **i32))
    ws = torch.empty(max(1, ops.route_map_workspace_bytes(T, E, k)), dtype=torch.uint8, device=dev)
    q = torch.empty(R, H, dtype=torch.uint8, device=dev)
    sfb = torch.empty((G + 3) // 4, ld, 4, dtype=torch.uint8, device=dev)
    ws2 = torch.empty(ops.expand_cast_fp8_ex_workspace_bytes(T, H, flags), dtype=torch.uint8,
                      device=dev)

    def rec():
        chk(L.moe_topk_gate(s.data_ptr(), T, E, k, idx.data_ptr(), wt.data_ptr(), 1, sp), "topk")
        chk(L.moe_route_map(idx.data_ptr(), T, E, k, counts.data_ptr(), offsets.data_ptr(),
                            pos.data_ptr(), src.data_ptr(), ws.data_ptr(), ws.numel(), sp), "route")
        chk(L.moe_expand_cast_fp8_ex(x.data_ptr(), T, H, k, pos.data_ptr(), src.data_ptr(), R,
                                     q.data_ptr(), sfb.data_ptr(), flags, ld, ws2.data_ptr(),
                                     ws2.numel(), 128, sp), "expand_ex")

    ms = timed(rec, max(3, iters // 2))
    B = algorithmic_bytes(T, E, k, H)
    b = B["route_expand_cast"] - R * G * 4 + R * G      # one scale byte per group
    gbs = b / (ms * 1e-3) / 1e9
    # FP4 E2M1, 32-channel groups, f32 scales (same routing, same inputs)
    q4 = torch.empty(R, H // 2, dtype=torch.uint8, device=dev)
    sf4 = torch.empty(R, H // 32, dtype=torch.float32, device=dev)

    def rec4():
        chk(L.moe_topk_gate(s.data_ptr(), T, E, k, idx.data_ptr(), wt.data_ptr(), 1, sp), "topk")
        chk(L.moe_route_map(idx.data_ptr(), T, E, k, counts.data_ptr(), offsets.data_ptr(),
                            pos.data_ptr(), src.data_ptr(), ws.data_ptr(), ws.numel(), sp), "route")
        chk(L.moe_expand_cast_fp4(x.data_ptr(), T, H, k, pos.data_ptr(), None, R, q4.data_ptr(),
                                  sf4.data_ptr(), 0, 0, None, 0, 32, sp), "expand_fp4")

    ms4 = timed(rec4, max(3, iters // 2))
    b4 = B["topk_gate"] + B["route_map"] + T * H * 2 + R * 4 + R * (H // 2) + R * (H // 32) * 4
    gbs4 = b4 / (ms4 * 1e-3) / 1e9
    res["prefill_64k_fp4_group32"] = {
        "op": "topk + route_map + expand_cast_fp4 (E2M1, 32-channel groups, f32 scales)",
        "ms": round(ms4, 4), "routed_tokens_per_s": round(R / (ms4 * 1e-3), 1),
        "algorithmic_bytes": b4, "GB_s": round(gbs4, 1), "frac_of_peak": round(gbs4 / peak, 4),
        "timing": "one batch after a 512 MB L2 flush, median"}
    # the same with packed UE8M0 scales, row-major (the MX FP4 layout: one
    # power-of-two exponent byte per 32 channels)
    sf4b = torch.empty(R, H // 32, dtype=torch.uint8, device=dev)

    def rec4b():
        chk(L.moe_topk_gate(s.data_ptr(), T, E, k, idx.data_ptr(), wt.data_ptr(), 1, sp), "topk")
        chk(L.moe_route_map(idx.data_ptr(), T, E, k, counts.data_ptr(), offsets.data_ptr(),
                            pos.data_ptr(), src.data_ptr(), ws.data_ptr(), ws.numel(), sp), "route")
        chk(L.moe_expand_cast_fp4(x.data_ptr(), T, H, k, pos.data_ptr(), None, R, q4.data_ptr(),
                                  sf4b.data_ptr(), 6, 0, None, 0, 32, sp), "expand_fp4_ue8m0")

    ms4b = timed(rec4b, max(3, iters // 2))
    b4b = b4 - R * (H // 32) * 4 + R * (H // 32)
    gbs4b = b4b / (ms4b * 1e-3) / 1e9
    res["prefill_64k_fp4_group32_ue8m0"] = {
        "op": "topk + route_map + expand_cast_fp4 (E2M1, 32-channel groups, packed UE8M0 "
              "row-major scales)",
        "ms": round(ms4b, 4), "routed_tokens_per_s": round(R / (ms4b * 1e-3), 1),
        "algorithmic_bytes": b4b, "GB_s": round(gbs4b, 1), "frac_of_peak": round(gbs4b / peak, 4),
        "timing": "one batch after a 512 MB L2 flush, median"}
    del q4, sf4, sf4b
    res["prefill_64k_ue8m0_colmajor"] = {
        "op": "topk + route_map + expand_cast_fp8_ex (packed UE8M0, column-major)",
        "ms": round(ms, 4), "routed_tokens_per_s": round(R / (ms * 1e-3), 1),
        "algorithmic_bytes": b, "GB_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
        "timing": "one batch after a 512 MB L2 flush, median"}
    del inp, s, x, q, sfb
    torch.cuda.empty_cache()

    w = workloads.WORKLOADS["swiglu_64k"]
    hx = workloads.make_inputs(w, seed=0, device=dev)["swiglu_x"]
    M, N = w.M, w.N
    G2, ld2 = N // 128, (M + 3) // 4 * 4
    q2 = torch.empty(M, N, dtype=torch.uint8, device=dev)
    sf2 = torch.empty((G2 + 3) // 4, ld2, 4, dtype=torch.uint8, device=dev)
    wr = torch.rand(M, generator=torch.Generator(device=dev).manual_seed(1), device=dev)
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)

    def sw():
        chk(L.swiglu_cast_fp8_ex(hx.data_ptr(), M, N, q2.data_ptr(), sf2.data_ptr(), flags, ld2,
                                 1, 7.0, wr.data_ptr(), cnt.data_ptr(), 128, sp), "swiglu_ex")

    ms = timed(sw, iters)
    b = M * 2 * N * 2 + M * 4 + M * N + M * G2
    gbs = b / (ms * 1e-3) / 1e9
    res["swiglu_64k_clamp_weight_ue8m0"] = {
        "op": "swiglu_cast_fp8_ex (clamp 7, per-row weight, clamp count, packed UE8M0 col-major)",
        "ms": round(ms, 4), "rows_per_s": round(M / (ms * 1e-3), 1), "algorithmic_bytes": b,
        "GB_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
        "clamped_inputs_per_pass": int(cnt.item()) // (iters + 2),
        "timing": "after a 512 MB L2 flush, median"}
    q5 = torch.empty(M, N // 2, dtype=torch.uint8, device=dev)
    sf5 = torch.empty(M, N // 32, dtype=torch.float32, device=dev)

    def sw4():
        chk(L.swiglu_cast_fp4(hx.data_ptr(), M, N, q5.data_ptr(), sf5.data_ptr(), 0, 0, 0, 0.0,
                              None, None, 32, sp), "swiglu_fp4")

    ms = timed(sw4, iters)
    b = M * 2 * N * 2 + M * (N // 2) + M * (N // 32) * 4
    gbs = b / (ms * 1e-3) / 1e9
    res["swiglu_64k_fp4_group32"] = {
        "op": "swiglu_cast_fp4 (E2M1, 32-channel groups, f32 scales)",
        "ms": round(ms, 4), "rows_per_s": round(M / (ms * 1e-3), 1), "algorithmic_bytes": b,
        "GB_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
        "timing": "after a 512 MB L2 flush, median"}
    if L.moe_get_device_status(sp, None) != 0:
        raise RuntimeError("device error in the cast-option workloads")
    return res


def decode_workload(L, dev, stream, sp, chk, flush, iters, peak, w):
    """route + expand + cast of a small batch `w` through the one-call entry
    point moe_route_expand_cast_fp8: AUTO (what a caller gets), the separate
    launches (chained by programmatic dependent launch), the same captured in
    a CUDA graph, the fused single cooperative launch and the
    replicated-routing path, where the shape allows each.  Each timed after a
    512 MB L2 flush that also keeps the GPU busy while the host enqueues
    (device time only)."""
    import torch

    from moe_routing_precision_gb300 import ops, workloads
    inp = workloads.make_inputs(w, seed=0, device=dev)
    s, x = inp["scores"], inp["x"]
    T, E, k, H, R, G = w.T, w.E, w.k, w.H, w.R, w.G
    i32 = dict(dtype=torch.int32, device=dev)
    idx, wt = torch.empty(T, k, **i32), torch.empty(T, k, dtype=torch.float32, device=dev)
    counts, offsets, pos, src = (torch.empty(E, **i32), torch.empty(E + 1, **i32),
                                 torch.empty(T, k, **i32), torch.empty(R, **i32))
    q = torch.empty(R, H, dtype=torch.uint8, device=dev)
    sf = torch.empty(R, G, dtype=torch.float32, device=dev)
    ws = ops.route_expand_cast_workspace(T, E, k, x)

    def raw(mode, st=sp):
        return L.moe_route_expand_cast_fp8(s.data_ptr(), T, E, k, x.data_ptr(), H, idx.data_ptr(),
                                           wt.data_ptr(), counts.data_ptr(), offsets.data_ptr(),
                                           pos.data_ptr(), src.data_ptr(), q.data_ptr(),
                                           sf.data_ptr(), ws.data_ptr(), ws.numel(), mode, 128, st)

    def call(mode, st=sp):
        chk(raw(mode, st), "route_expand_cast")

    def timed(fn):
        ts = []
        for i in range(iters + 3):
            flush.fill_(i & 0xFF)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    res = {"op": f"topk + route_map + expand_cast_fp8 (T={T}, E={E}, k={k}, H={H})"}
    B = algorithmic_bytes(T, E, k, H)["route_expand_cast"]
    times = {"auto": timed(lambda: call(ops.PATH_AUTO)),
             "separate_launches": timed(lambda: call(ops.PATH_SEPARATE))}
    for name, mode in (("fused_single_launch", ops.PATH_FUSED),
                       ("replicated_routing", ops.PATH_REPLICATED),
                       ("chained", ops.PATH_CHAINED)):
        rc = raw(mode)
        if rc == ops.MOE_ERR_UNSUPPORTED:
            continue
        chk(rc, name)
        times[name] = timed(lambda m=mode: call(m))
    call(ops.PATH_SEPARATE)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(device=dev)
    with torch.cuda.graph(g, stream=cs):
        call(ops.PATH_SEPARATE, cs.cuda_stream)
    times["separate_in_cuda_graph"] = timed(lambda: g.replay())
    if L.moe_get_device_status(sp, None) != 0:
        raise RuntimeError("device error in the decode workload")
    for name, us in times.items():
        gbs = B / (us * 1e-6) / 1e9
        res[name] = {"us": round(us, 2), "routed_tokens_per_s": round(R / (us * 1e-6), 1),
                     "GB_s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4)}
    res["algorithmic_bytes"] = B
    res["timing"] = "one call after a 512 MB L2 flush, median; device time"
    del g
    return res


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleChain:
    """topk_gate + route_map + expand_cast_fp8 of the oracle as it stands.
    With threads > 1 the per-token steps (top-k, expand + cast) run on token
    shards in a thread pool (each shard is one C call, which releases the
    GIL) and the route map runs once over all tokens, as it must."""

    def __init__(self, scores, x_bits, k, E, threads=1):
        import numpy as np
        self.s, self.x, self.k, self.E = scores, x_bits, k, E
        self.threads = max(1, int(threads))
        T = scores.shape[0]
        self.shards = [sl for sl in np.array_split(np.arange(T), self.threads) if sl.size]
        self.pool = None
        if self.threads > 1:
            from concurrent.futures import ThreadPoolExecutor
            self.pool = ThreadPoolExecutor(self.threads)

    def run(self) -> float:
        """One pass; returns its wall time in seconds."""
        import numpy as np

        import oracle
        s, xb, k, E = self.s, self.x, self.k, self.E
        sl = [(int(a[0]), int(a[-1]) + 1) for a in self.shards]
        each = map if self.pool is None else self.pool.map
        t0 = time.perf_counter()
        idx = np.concatenate(list(each(lambda r: oracle.topk_gate(s[r[0]:r[1]], k)[0], sl)))
        _, _, pos, _ = oracle.route_map(idx, E)
        T, H = xb.shape
        q = np.zeros((T * k, H), dtype=np.uint8)
        sf = np.zeros((T * k, H // 128), dtype=np.float32)
        list(each(lambda r: oracle.expand_cast_fp8_into(xb[r[0]:r[1]], pos[r[0]:r[1]], q, sf), sl))
        return time.perf_counter() - t0

    def close(self):
        if self.pool is not None:
            self.pool.shutdown()


def cpu_baseline_leg(scores, x, k, E, total=65536, single_tokens=16384):
    """The oracle as it stands on the host cores: every token of the
    benchmarked workload over all host threads (token shards), and a
    single-threaded pass over its first `single_tokens` tokens."""
    import oracle
    s = scores.cpu().numpy()
    xb = oracle.bf16_bits(x.cpu())
    n = host_threads()
    chain = OracleChain(s, xb, k, E, threads=n)
    dt = min(chain.run() for _ in range(2))
    chain.close()
    ts = min(single_tokens, s.shape[0])
    one = OracleChain(s[:ts], xb[:ts], k, E, threads=1)
    dt1 = one.run()
    T = s.shape[0]
    return {"value": round(T * k / dt, 1), "unit": UNIT, "cores": n, "kind": "oracle",
            "cpu": cpu_model(), "host_cores": os.cpu_count(),
            "sample": f"all {T} of {total} tokens of the benchmarked workload (topk_gate + "
                      f"route_map + expand_cast_fp8), {n} threads over token shards (route map "
                      f"serial), best of 2 passes, {dt:.2f} s",
            "sample_short": f"all {T} tokens, {n} threads, best of 2 passes ({dt:.2f} s)",
            "single_thread": {"value": round(ts * k / dt1, 1), "unit": UNIT, "cores": 1,
                              "sample": f"first {ts} tokens, one thread, {dt1:.1f} s"}}


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, or the Arm
    implementer/part codes), else the platform string."""
    import platform
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        info = []
    for key in ("model name", "Model name"):
        for line in info:
            if line.startswith(key):
                return line.split(":", 1)[1].strip()
    parts = {}
    for line in info:
        for key in ("CPU implementer", "CPU part"):
            if line.startswith(key):
                parts[key] = line.split(":", 1)[1].strip()
    if parts:
        return f"{platform.machine()} implementer {parts.get('CPU implementer')} part {parts.get('CPU part')}"
    return platform.processor() or platform.machine()


# ---------------------------------------------------------------- reference arm


# ---------------------------------------------------------------- reference arm

def reference_arm(args):
    """The oracle timed on the host cores (all host threads, token shards),
    same metric and workload: every step is one pass over all tokens of the
    large-prefill batch (rank 0's: seed 0), drawn on the host."""
    import oracle
    from moe_routing_precision_gb300 import workloads
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    oracle.build()
    w = workloads.WORKLOADS[WORKLOAD]
    tokens = w.T if args.ref_tokens <= 0 else min(w.T, args.ref_tokens)
    sub = w if tokens == w.T else workloads.Workload(w.name, T=tokens, E=w.E, k=w.k, H=w.H,
                                                     bias=w.bias, x_std=w.x_std)
    inp = workloads.make_inputs(sub, seed=shard_seed(rank), device="cpu")
    s = inp["scores"].numpy()
    xb = oracle.bf16_bits(inp["x"])
    del inp

    n = host_threads()
    chain = OracleChain(s, xb, w.k, w.E, threads=n)
    for _ in range(args.warmup):
        chain.run()
    dt = sum(chain.run() for _ in range(args.steps)) / args.steps
    chain.close()
    value = tokens * w.k / dt
    sample = (f"all {tokens} tokens per step" if tokens == w.T else
              f"{tokens} of {w.T} tokens per step") + \
        f" (topk_gate + route_map + expand_cast_fp8), the C oracle on {n} threads over token " \
        "shards (route map serial)"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 (CPU oracle)", "data": "synthetic",
        "config": config_dict(world),
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": n, "kind": "oracle",
                         "cpu": cpu_model(), "host_cores": os.cpu_count(), "sample": sample},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=int(os.environ.get("MOE_BENCH_ITERS", "300")),
                    help="timed steps (default: $MOE_BENCH_ITERS, else 300)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--e2e-steps", type=int, default=30,
                    help="steps of the end-to-end leg (its own count, not --steps)")
    ap.add_argument("--extra-iters", type=int, default=30)
    ap.add_argument("--ref-tokens", type=int, default=0,
                    help="reference arm: tokens per step (0: the whole workload)")
    ap.add_argument("--workload", choices=["prefill_64k", "skewed_8k", "decode_1k", "tiny"],
                    default=WORKLOAD)
    ap.add_argument("--ops", choices=["all", "route_expand_cast"], default="all",
                    help="all: the whole step (route+expand+cast, SwiGLU, combine); "
                         "route_expand_cast: the headline ops only")
    ap.add_argument("--headline-path", choices=["one_call", "calls"], default="one_call",
                    help="route+expand+cast as the one-call entry point (AUTO) or as the three "
                         "individual calls")
    ap.add_argument("--detail-out", default=DETAIL_DEFAULT,
                    help="where the long-form results go ('' to skip)")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    line = reference_arm(args) if args.impl == "reference" else gpu_arm(args)
    if line is not None:
        print(json.dumps(line, separators=(",", ":")), flush=True)


if __name__ == "__main__":
    main()
