"""Benchmark of the CSR sparse-adapter hot path on GB300.

One step = one pass of the whole path over one workload:
  sort_rows (row_idx) -> plan_build (row bins + dense panels, shared by both products)
  -> spmm (C = A X) -> sddmm (structure-aware backend, grad = dY^T X sampled on the mask)
  -> csr_add (W + A)
(operators the workload does not define are left out). metric: GFLOP/s counting
2 * nnz * N for SpMM and 2 * nnz * kd for SDDMM; every operator's time is in the step.

By default every configuration is measured in one run (tiny 256^2, the RoSA adapter, the
LLaMA MLP weight, the Zipf matrix, the pixelfly butterfly layer, plus the narrow-N SpMM
workload) and the headline fields (value, ms_per_step, roofline, cpu_baseline, e2e) are the
butterfly layer's, the largest configuration; `per_config` holds each workload's record.
Each step is one CUDA-graph replay of the library calls in which spmm, sddmm and csr_add
(independent once row_idx and the plan exist) run on three streams (csr_add beside the plan,
sddmm beside spmm); a second loop replays one graph per operator in order to give the
per-operator times. L2 is flushed (a 256 MB
write) before every timed step, outside the step's events.

--impl reference times the fp64 CPU oracle on the host cores on the headline workload, with
the same metric, unit and config (a deliberately slow baseline, not a target).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
METRIC = "SpMM+SDDMM GFLOP/s (2*nnz*N + 2*nnz*kd per step; step = sort_rows+plan+spmm+sddmm+csr_add)"
DESCRIPTION = {
    "tiny": "tiny_256x256_fp32_5pct_uniform_N64",
    "rosa": "rosa_adapter_4096x4096_fp16_1pct_clustered_2048tok",
    "llama_mlp": "llama_mlp_11008x4096_bf16_0.5pct_uniform_4096tok",
    "zipf": "zipf_131072x131072_fp32_band8192_N128",
    "butterfly": "pixelfly_butterfly_8192x2048_bf16_64x64blocks_8192tok",
    "spmv": "narrow_spmm_8192x8192_fp16_90pct_sparse_N8",
}
for _n, _s in wl.SPECS.items():
    if _n.startswith("fly_"):
        DESCRIPTION[_n] = f"pixelfly_mlp_layer_{_s.m}x{_s.n}_bf16_block{dict(_s.mask_kw)['block']}_{_s.N}tok"
HEADLINE = "butterfly"            # the largest configuration carries the headline fields
EXTRA_WORKLOADS = ["spmv"]       # measured after the five configurations (narrow-N SpMM)
SINGLE_THREAD_BASELINE = ("tiny", "rosa", "llama_mlp")  # oracle also timed on one core


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def index_dtype(w):
    return torch.int16 if max(w.m, w.n) <= 32768 else torch.int32


def max_over_ranks(value: float, device=None) -> float:
    """The largest value over all ranks of the default process group (the job's time is
    the slowest rank's). Returns value unchanged without a process group."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ work accounting


def accounting(w):
    """Algorithmic flops and compulsory HBM bytes of each operator on workload w."""
    ro = w.row_offsets.numpy()
    col = w.col_idx.numpy()
    m, n, nnz = w.m, w.n, w.nnz
    b = w.values.element_size()
    ib = 2 if max(m, n) <= 32768 else 4
    lens = np.diff(ro)
    active_rows = int((lens > 0).sum())
    active_cols = int(np.unique(col).size)
    csr_bytes = nnz * (b + ib) + 4 * (m + 1) + ib * m
    acc = {"sort_rows": {"flops": 0, "bytes": 4 * (m + 1) + ib * m},
           "plan": {"flops": 0, "bytes": 4 * (m + 1) + ib * m + nnz * ib}}
    if w.B is not None:
        N = w.B.shape[1]
        acc["spmm"] = {"flops": 2 * nnz * N, "bytes": csr_bytes + active_cols * N * b + m * N * b}
    if w.A is not None:
        kd = w.A.shape[1]
        acc["sddmm"] = {"flops": 2 * nnz * kd,
                        "bytes": csr_bytes - nnz * b + active_rows * kd * b + active_cols * kd * b + nnz * b}
    if w.W is not None:
        acc["csr_add"] = {"flops": nnz, "bytes": csr_bytes - ib * m + 2 * m * n * b}
    return acc


def step_flops(acc):
    return acc.get("spmm", {}).get("flops", 0) + acc.get("sddmm", {}).get("flops", 0)


# ------------------------------------------------------------------ clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_dir: str | None = None):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.log_dir = log_dir or tempfile.gettempdir()

    def start(self):
        try:
            os.makedirs(self.log_dir, exist_ok=True)
            self.path = os.path.join(self.log_dir, f"clocks_rank{self.gpu}.csv")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                             "reasons": parts[4:9]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        seen = set()
        for r in rows:
            for nm, v in zip(names[1:], r["reasons"][1:]):
                if v.lower() in ("active", "1", "yes"):
                    seen.add(nm)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(seen), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ------------------------------------------------------------------ profile summary (traffic)


def kernel_source_hash(paths):
    """sha256[:16] over the listed source files ('+'-separated), in order."""
    h = hashlib.sha256()
    for p in paths.split("+"):
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(op: str, workload: str):
    """DRAM bytes per call of the op (its kernels summed) on this workload from the committed
    ncu summary, if the kernel sources still match the hash recorded with the counters:
    {"bytes": read + write, "read": ..., "write": ...} (read / write None in rows that give
    only the sum), or None."""
    p = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(p):
        return None
    pat = re.compile(r"\|\s*" + re.escape(workload) + r"\s*\|\s*" + re.escape(op) +
                     r"\s*\|\s*([\w./+]+)\s*\|\s*([0-9a-f]+)\s*\|\s*([0-9]+)\s*\|"
                     r"(?:\s*([0-9]+)\s*\|\s*([0-9]+)\s*\|)?(?:\s*([0-9]+)\s*\|)?")
    for line in open(p):
        mt = pat.match(line)
        if mt:
            src, h = mt.group(1), mt.group(2)
            if mt.group(4) is not None:  # | read | write | sum | (L2 write |)
                rd, wr, total = int(mt.group(3)), int(mt.group(4)), int(mt.group(5))
            else:
                rd, wr, total = None, None, int(mt.group(3))
            l2w = int(mt.group(6)) if mt.group(6) is not None else None
            try:
                if kernel_source_hash(src) != h:
                    return None
            except OSError:
                return None
            rec = {"bytes": total, "read": rd, "write": wr}
            if l2w is not None:
                rec["l2_write"] = l2w
            return rec
    return None


# ------------------------------------------------------------------ GPU arm


def make_ops(sp, w, d, idx, args, outs):
    """The step as a list of (name, callable) over device tensors d."""
    ops = [("sort_rows", lambda: outs.__setitem__("row_idx", sp.sort_rows(d["ro"], nnz=w.nnz, index_dtype=idx))),
           ("plan", lambda: outs.__setitem__("plan", sp.plan_build(d["ro"], outs["row_idx"], d["col"], w.n)))]
    if "B" in d:
        ops.append(("spmm", lambda: outs.__setitem__(
            "C", sp.spmm(d["val"], d["ro"], outs["row_idx"], d["col"], d["B"], w.m, path=args.spmm_path,
                         plan=outs["plan"]))))
    if "A" in d:
        ops.append(("sddmm", lambda: outs.__setitem__(
            "G", sp.sddmm(d["ro"], outs["row_idx"], d["col"], d["A"], d["BT"], backend=args.sddmm_backend,
                          plan=outs["plan"]))))
    if "W" in d:
        ops.append(("csr_add", lambda: outs.__setitem__(
            "D", sp.csr_add(d["val"], d["ro"], outs["row_idx"], d["col"], d["W"]))))
    return ops


def run_step_forked(ops, stream, side, overlap=True):
    """The step on `stream` and the side streams, by data dependence: sort_rows first; with
    overlap, csr_add (which needs only row_idx) forks right after it, beside the plan, and after
    the plan sddmm forks while spmm runs on `stream`; everything joins back into `stream`.
    Without overlap the operators run one after the other (kept for comparisons)."""
    by = dict(ops)
    spare = list(side)
    joins = []

    def fork(f):
        s = spare.pop(0)
        e = torch.cuda.Event()
        e.record(stream)
        s.wait_event(e)
        with torch.cuda.stream(s):
            f()
            j = torch.cuda.Event()
            j.record(s)
        joins.append(j)

    by["sort_rows"]()
    if "csr_add" in by and overlap:
        fork(by["csr_add"])
    by["plan"]()
    if "sddmm" in by and "spmm" in by and overlap:
        fork(by["sddmm"])
        by["spmm"]()
    elif "sddmm" in by and "spmm" in by:
        by["spmm"]()
        by["sddmm"]()
    elif "sddmm" in by:
        by["sddmm"]()
    elif "spmm" in by:
        by["spmm"]()
    if "csr_add" in by and not overlap:
        by["csr_add"]()
    for j in joins:
        stream.wait_event(j)


def run_fixed_forked(ops, stream, side, overlap=True):
    """The step with the mask fixed: row_idx and the plan of the last full step are reused, so
    only the operators on values run, forked as in run_step_forked (csr_add and, with overlap,
    sddmm on the side streams, spmm on `stream`)."""
    by = dict(ops)
    spare = list(side)
    joins = []
    for name in ("csr_add", "sddmm"):
        if name in by and overlap and (name == "csr_add" or "spmm" in by):
            e = torch.cuda.Event()
            e.record(stream)
            s = spare.pop(0)
            s.wait_event(e)
            with torch.cuda.stream(s):
                by[name]()
                j = torch.cuda.Event()
                j.record(s)
            joins.append(j)
    if "spmm" in by:
        by["spmm"]()
    if "sddmm" in by and not ("spmm" in by and overlap):
        by["sddmm"]()
    if "csr_add" in by and not overlap:
        by["csr_add"]()
    for j in joins:
        stream.wait_event(j)


def host_inputs(w, idx):
    h = {"ro": w.row_offsets, "col": w.col_idx.to(idx), "val": w.values}
    for k in ("B", "A", "BT", "W"):
        t = getattr(w, k)
        if t is not None:
            h[k] = t
    return h


def config_dict(name, w, args):
    """The `config` object of the JSON line for workload `name` (the same on both arms)."""
    return {"workload": DESCRIPTION[name], "m": w.m, "n": w.n, "nnz": w.nnz,
            "N": int(w.meta["spec"].N) or None, "kd": int(w.meta["spec"].kd) or None,
            "index": "int16" if max(w.m, w.n) <= 32768 else "int32", "sddmm_backend": args.sddmm_backend,
            "spmm_path": args.spmm_path, "l2": "flushed before every step (256 MB write, outside step events)",
            "parallelism": "replicas (independent problems per GPU)"}


def workload_list(args):
    return list(wl.CONFIG_ORDER) + EXTRA_WORKLOADS if args.workload == "all" else [args.workload]


def headline_name(args):
    return HEADLINE if args.workload == "all" else args.workload


def measure(sp, lib, name, args, dev, ws, rank, local, flush):
    """Time one workload's step (CUDA graph replays, L2 flushed before each) and its
    operators one at a time; then the end-to-end leg, the next operators and, on rank 0 at
    N = 1, the oracle on a bounded sample. Returns the workload's JSON record."""
    w = wl.generate(name)
    acc = accounting(w)
    flops = step_flops(acc)
    idx = index_dtype(w)
    d = {k: v.to(dev) for k, v in host_inputs(w, idx).items()}
    outs = {}
    ops = make_ops(sp, w, d, idx, args, outs)
    stream = torch.cuda.Stream(device=dev)
    side = [torch.cuda.Stream(device=dev) for _ in range(2)]
    with torch.cuda.stream(stream):
        run_step_forked(ops, stream, side)
        torch.cuda.synchronize(dev)
        # the operators overlap on every workload: csr_add beside the plan takes the plan's
        # latency chain off the step (llama 427 -> 419 us, RoSA 83 -> 65 us), and SDDMM beside
        # SpMM shares the SMs between two tensor-core kernels or costs nothing measurable
        # where both are general row kernels (llama mask-fixed 387 vs 388 us)
        overlap = True
        for _ in range(max(args.warmup, 1)):
            run_step_forked(ops, stream, side, overlap)  # eager, on the streams the graph uses
            torch.cuda.synchronize(dev)
        pool = torch.cuda.graph_pool_handle()
        # the step on three streams by data dependence (fork / join inside one graph)
        step_graph = torch.cuda.CUDAGraph()
        launches0 = lib.spops_kernel_launches()
        with torch.cuda.graph(step_graph, stream=stream, pool=pool):
            run_step_forked(ops, stream, side, overlap)
        launches_per_step = lib.spops_kernel_launches() - launches0
        # one graph per operator, replayed in order, for the per-operator breakdown
        op_graphs = []
        for op_name, f in ops:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, pool=pool):
                f()
            op_graphs.append((op_name, g))
        # the mask-fixed step: the value operators on the row order and plan that the
        # operator graphs above leave in their buffers
        fixed_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(fixed_graph, stream=stream, pool=pool):
            run_fixed_forked(ops, stream, side, overlap)
        for _ in range(args.warmup):
            step_graph.replay()
            for _, g in op_graphs:
                g.replay()
        torch.cuda.synchronize(dev)

        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        sampler = ClockSampler(local, args.clock_log_dir)
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        sampler.start()
        time.sleep(0.2)
        t0 = time.perf_counter()
        for s in range(args.steps):
            flush.zero_()
            ev[s][0].record(stream)
            step_graph.replay()
            ev[s][1].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        if ws > 1:
            torch.distributed.barrier()
        clocks = sampler.stop()

        # per-operator breakdown: the same graphs one operator at a time, events between them
        nb = max(3, min(args.steps, args.breakdown_steps))
        nops = len(op_graphs)
        evb = [[torch.cuda.Event(enable_timing=True) for _ in range(nops + 1)] for _ in range(nb)]
        for s in range(nb):
            flush.zero_()
            evb[s][0].record(stream)
            for j, (_, g) in enumerate(op_graphs):
                g.replay()
                evb[s][j + 1].record(stream)
        torch.cuda.synchronize(dev)
        evf = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(nb)]
        for s in range(nb):
            flush.zero_()
            evf[s][0].record(stream)
            fixed_graph.replay()
            evf[s][1].record(stream)
        torch.cuda.synchronize(dev)

    step_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(args.steps)]
    op_ms = {op_name: [evb[s][j].elapsed_time(evb[s][j + 1]) for s in range(nb)]
             for j, (op_name, _) in enumerate(op_graphs)}
    total_ms = max_over_ranks(sum(step_ms), dev)
    ms_per_step = total_ms / args.steps
    value = ws * flops * args.steps / (total_ms * 1e-3) / 1e9
    fixed_ms = [evf[s][0].elapsed_time(evf[s][1]) for s in range(nb)]
    fixed_avg = sum(fixed_ms) / nb
    mask_fixed = {"ms_per_step": round(fixed_avg, 5), "ms_median": round(statistics.median(fixed_ms), 5),
                  "value": round(flops / (fixed_avg * 1e-3) / 1e9, 2), "unit": "GFLOP/s",
                  "ops": [o for o, _ in ops if o not in ("sort_rows", "plan")],
                  "note": "row_idx and the plan built once and reused (the mask does not change between steps); "
                          "forked like the full step; L2 flushed before each step"}
    del step_graph, op_graphs, fixed_graph

    e2e = run_e2e(sp, w, dev, idx, args, flops, ws)
    next_ops = time_next_ops(sp, w, d, idx, stream, pool, flush, nb) if not args.no_next_ops else None

    pk = peaks()
    per_op = {}
    for op_name, times in op_ms.items():
        t_avg = sum(times) / len(times)
        a = acc[op_name]
        per_op[op_name] = {"ms": round(t_avg, 5), "ms_median": round(statistics.median(times), 5),
                           "ms_min": round(min(times), 5),
                           "GFLOP/s": round(a["flops"] / (t_avg * 1e-3) / 1e9, 2) if a["flops"] else None,
                           "GB/s": round(a["bytes"] / (t_avg * 1e-3) / 1e9, 1),
                           "hbm_frac": round(a["bytes"] / (t_avg * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                           "algorithmic_bytes": int(a["bytes"])}
    dominant = max((k for k in per_op if k not in ("sort_rows", "plan")), key=lambda k: per_op[k]["ms"])
    dom_t = per_op[dominant]["ms"] * 1e-3
    achieved = acc[dominant]["bytes"] / dom_t / 1e9
    traffic = recorded_traffic(dominant, name)
    roofline = {"kernel": dominant, "bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                "traffic": traffic["bytes"] if traffic else None,
                "traffic_read": traffic["read"] if traffic else None,
                "traffic_write": traffic["write"] if traffic else None,
                "traffic_l2_write": traffic.get("l2_write") if traffic else None,
                "algorithmic_bytes": acc[dominant]["bytes"], "peak_source": pk["source"],
                "note": "achieved = algorithmic bytes of the operator / its mean event time in the per-operator "
                        "loop (L2 flushed before each step); traffic = ncu dram__bytes_read + dram__bytes_write "
                        "summed over the operator's kernels, from one capture per kernel; writes of an output "
                        "that stays in the write-back L2 during the capture are not in dram__bytes_write, so "
                        "traffic_l2_write gives the bytes the kernels wrote into L2 (lts__t_sectors_op_write x 32)"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, acc, seconds=args.cpu_seconds,
                           single_thread=name in SINGLE_THREAD_BASELINE and args.workload == "all")
    rec = {"value": round(value, 2), "unit": "GFLOP/s", "ms_per_step": round(ms_per_step, 5), "steps": args.steps,
           "dtype": w.dtype, "config": config_dict(name, w, args), "per_op": per_op, "roofline": roofline,
           "cpu_baseline": cpu, "e2e": e2e, "next_ops": next_ops, "mask_fixed": mask_fixed,
           "operators_overlap": overlap,
           "gpu_launches": int(launches_per_step) * args.steps, "launches_per_step": int(launches_per_step),
           "clocks": clocks, "breakdown_steps": nb,
           "step_ms_sum_of_ops": round(sum(v["ms"] for v in per_op.values()), 5),
           "wall_s_timed_region": round(wall, 4)}
    del d, outs, ops
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return rec


def run_gpu(args):
    import torch.distributed as dist

    import unstructured_sparse_linear_gb300 as sp

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    lib = sp._lib.load()

    head = headline_name(args)
    per_config = {}
    for name in workload_list(args):
        log(f"[bench] {name}")
        per_config[name] = measure(sp, lib, name, args, dev, ws, rank, local, flush)
    extra = time_fly_mlps(sp, dev, flush, args) if args.workload == "all" and not args.no_next_ops else None

    h = per_config[head]
    line = {
        "metric": METRIC, "value": h["value"], "unit": "GFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": h["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": h["dtype"], "data": "synthetic (seeded generators in the workloads package)",
        "config": h["config"], "per_op": h["per_op"], "roofline": h["roofline"], "cpu_baseline": h["cpu_baseline"],
        "e2e": h["e2e"], "gpu_launches": h["gpu_launches"], "clocks": h["clocks"], "mask_fixed": h["mask_fixed"],
        "headline": f"{head}: the step (sort_rows+plan+spmm+sddmm+csr_add where defined) on this workload; "
                    "per_config holds every configuration measured the same way",
        "per_config": {k: {kk: vv for kk, vv in v.items() if kk != "next_ops"} for k, v in per_config.items()},
        "next_ops": {k: v["next_ops"] for k, v in per_config.items() if v.get("next_ops")},
        "pixelfly_mlps": extra,
        "breakdown_steps": h["breakdown_steps"], "step_ms_sum_of_ops": h["step_ms_sum_of_ops"],
        "wall_s_timed_region": h["wall_s_timed_region"],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def time_next_ops(sp, w, d, idx, stream, pool, flush, reps):
    """The operators beyond the step, each as its own graph replayed `reps` times with an
    L2 flush before every replay: csr_transpose of the mask (structure and values), the
    value refresh through an existing transpose, dB = A^T dC with the transpose kept (the
    mask is fixed while its values train: permute values, sort_rows of A^T, SpMM of A^T),
    and one masked Adam step on the adapter's fp32 values."""
    pk = peaks()
    m, n, nnz = w.m, w.n, w.nnz
    b = w.values.element_size()
    ib = 2 if idx == torch.int16 else 4
    ro, col, val = d["ro"], d["col"], d["val"]
    ops, acc = [], {}
    with torch.cuda.stream(stream):
        t = sp.csr_transpose(val, ro, col, n)
        ops.append(("csr_transpose", lambda: sp.csr_transpose(val, ro, col, n)))
        acc["csr_transpose"] = (0, 4 * (m + 1) + nnz * (ib + b) + 4 * (n + 1) + nnz * (ib + b + 4))
        vt = torch.empty_like(val)
        ops.append(("permute_values", lambda: sp.permute_values(val, t, out=vt)))
        acc["permute_values"] = (0, nnz * (4 + 2 * b))
        if w.B is not None:
            N = int(w.B.shape[1])
            dC = torch.randn((m, N), device=val.device).to(val.dtype)
            active_rows = int((np.diff(w.row_offsets.numpy()) > 0).sum())
            ops.append(("spmm_grad_b", lambda: sp.spmm_grad_b(val, ro, col, dC, n, transpose=t)))
            acc["spmm_grad_b"] = (2 * nnz * N, nnz * (4 + 2 * b) + 4 * (n + 1) + ib * n + nnz * (ib + b)
                                  + active_rows * N * b + n * N * b)
        if w.B is not None and w.A is not None and w.dtype in ("f16", "bf16") and w.B.shape[1] == w.A.shape[1]:
            # the layer Y^T = W X^T (X^T = B: in x tokens) forward and backward with dY^T = A,
            # on the mask's values (structure, plans and transpose built once), against the
            # same layer with a dense weight on cuBLAS (three GEMMs)
            T = int(w.B.shape[1])
            Xt, dYt = d["B"], d["A"]
            ri = sp.sort_rows(ro, nnz=nnz, index_dtype=idx)
            pl = sp.plan_build(ro, ri, col, n)
            ri_t = sp.sort_rows(t.row_offsets, nnz=nnz, index_dtype=idx)
            pl_t = sp.plan_build(t.row_offsets, ri_t, t.col_idx, m)

            def layer_sparse():
                sp.spmm(val, ro, ri, col, Xt, m, plan=pl)
                sp.sddmm(ro, ri, col, dYt, Xt, plan=pl)
                sp.spmm(sp.permute_values(val, t), t.row_offsets, ri_t, t.col_idx, dYt, n, plan=pl_t)

            Wd = torch.zeros((m, n), dtype=val.dtype, device=val.device)
            rows_of = torch.repeat_interleave(torch.arange(m, device=val.device), torch.diff(ro.long()))
            Wd[rows_of, col.long()] = val

            def layer_dense():
                torch.matmul(Wd, Xt)
                torch.matmul(dYt, Xt.t())
                torch.matmul(Wd.t(), dYt)

            ops.append(("layer_fwd_bwd_sparse", layer_sparse))
            acc["layer_fwd_bwd_sparse"] = (3 * 2 * nnz * T, 0)
            ops.append(("layer_fwd_bwd_dense_cublas", layer_dense))
            acc["layer_fwd_bwd_dense_cublas"] = (3 * 2 * m * n * T, 0)
        if w.B is not None and w.B.shape[1] <= 16:
            # the SpMV end of the narrow-N range: one right-hand side
            ri1 = sp.sort_rows(ro, nnz=nnz, index_dtype=idx)
            pl1 = sp.plan_build(ro, ri1, col, n)
            b1 = d["B"][:, :1].contiguous()
            ops.append(("spmv_n1", lambda: sp.spmm(val, ro, ri1, col, b1, m, plan=pl1)))
            acc["spmv_n1"] = (2 * nnz, nnz * (ib + b) + 4 * (m + 1) + ib * m + n * b + m * b)
        P = torch.randn(nnz, device=val.device)
        M1 = torch.zeros(nnz, device=val.device)
        V1 = torch.zeros(nnz, device=val.device)
        G = torch.randn(nnz, device=val.device).to(val.dtype)
        ops.append(("masked_adam", lambda: sp.masked_adam(P, M1, V1, G, 10)))
        acc["masked_adam"] = (0, nnz * (24 + b))
        for _, f in ops:
            f()
        torch.cuda.synchronize()
        graphs = []
        for name, f in ops:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, pool=pool):
                f()
            graphs.append((name, g))
        for _, g in graphs:
            g.replay()
        torch.cuda.synchronize()
        ev = {name: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(reps)] for name, _ in graphs}
        for r in range(reps):
            for name, g in graphs:
                flush.zero_()
                ev[name][r][0].record(stream)
                g.replay()
                ev[name][r][1].record(stream)
        torch.cuda.synchronize()
    out = {}
    for name, _ in graphs:
        ts = [a.elapsed_time(e) for a, e in ev[name]]
        t_avg = sum(ts) / len(ts)
        fl, by = acc[name]
        out[name] = {"ms": round(t_avg, 5), "ms_min": round(min(ts), 5),
                     "GFLOP/s": round(fl / (t_avg * 1e-3) / 1e9, 2) if fl else None}
        if by:
            out[name].update({"GB/s": round(by / (t_avg * 1e-3) / 1e9, 1),
                              "hbm_frac": round(by / (t_avg * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                              "algorithmic_bytes": int(by)})
    if "layer_fwd_bwd_sparse" in out:
        out["layer_speedup_vs_dense"] = round(out["layer_fwd_bwd_dense_cublas"]["ms"] /
                                              out["layer_fwd_bwd_sparse"]["ms"], 3)
    return out


def time_fly_mlps(sp, dev, flush, args, iters: int = 100):
    """The two MLPs of the pixelfly issue's T4 comment ([16, 512, D] inputs, forward and
    backward repeated 100 times): each layer a SparseLinear on its butterfly mask (forward
    spmm; backward sddmm for dW, value refresh of the cached transpose and spmm for dX),
    against the same layers with dense weights on cuBLAS (six GEMMs per iteration). Both run
    as CUDA graphs replayed back to back (a training loop: no L2 flush between iterations).
    No activation function sits between the layers (only the linear layers are timed)."""
    out = {}
    stream = torch.cuda.Stream(device=dev)
    for mlp in wl.FLY_MLPS:
        names = wl.fly_layer_names(mlp)
        with torch.cuda.stream(stream):
            layers, dense_w = [], []
            for nm in names:
                w = wl.generate(nm, operands=())
                idx = index_dtype(w)
                L = sp.SparseLinear(w.row_offsets.to(dev), w.col_idx.to(idx).to(dev), w.values.to(dev), w.n)
                layers.append(L)
                Wd = torch.zeros((w.m, w.n), dtype=w.values.dtype, device=dev)
                rows_of = torch.repeat_interleave(torch.arange(w.m, device=dev), torch.diff(L.row_offsets.long()))
                Wd[rows_of, L.col_idx.long()] = L.values.detach()
                dense_w.append(Wd)
            T = wl.FLY_MLPS[mlp]["tokens"]
            g = torch.Generator(device="cpu").manual_seed(7)
            X = torch.randn((layers[0].in_features, T), generator=g).to(torch.bfloat16).to(dev)
            dY = torch.randn((layers[-1].out_features, T), generator=g).to(torch.bfloat16).to(dev)
            vals = [L.values.detach() for L in layers]
            vt = [torch.empty_like(v) for v in vals]

            def sparse_iter():
                acts = [X]
                for L, v in zip(layers, vals):
                    acts.append(sp.spmm(v, L.row_offsets, L.row_idx, L.col_idx, acts[-1], L.out_features,
                                        plan=L.plan))
                grad = dY
                for li in range(len(layers) - 1, -1, -1):
                    L = layers[li]
                    sp.sddmm(L.row_offsets, L.row_idx, L.col_idx, grad, acts[li], plan=L.plan)
                    sp.permute_values(vals[li], L.transpose, out=vt[li])
                    grad = sp.spmm(vt[li], L.transpose.row_offsets, L.row_idx_t, L.transpose.col_idx, grad,
                                   L.in_features, plan=L.plan_t)

            def dense_iter():
                acts = [X]
                for Wd in dense_w:
                    acts.append(torch.matmul(Wd, acts[-1]))
                grad = dY
                for li in range(len(dense_w) - 1, -1, -1):
                    torch.matmul(grad, acts[li].t())
                    grad = torch.matmul(dense_w[li].t(), grad)

            res = {}
            for kind, f in (("sparse", sparse_iter), ("dense_cublas", dense_iter)):
                for _ in range(3):
                    f()
                torch.cuda.synchronize(dev)
                gph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gph, stream=stream):
                    f()
                for _ in range(3):
                    gph.replay()
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(iters):
                    gph.replay()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                ms = e0.elapsed_time(e1)
                res[kind] = {"ms_per_iter": round(ms / iters, 5), f"s_for_{iters}_iters": round(ms * 1e-3, 5)}
                del gph
            nnz = sum(L.col_idx.numel() for L in layers)
            dense_macs = sum(Wd.numel() for Wd in dense_w)
            res["sparse"]["GFLOP/s"] = round(3 * 2 * nnz * T / (res["sparse"]["ms_per_iter"] * 1e-3) / 1e9, 1)
            res["dense_cublas"]["GFLOP/s"] = round(3 * 2 * dense_macs * T /
                                                   (res["dense_cublas"]["ms_per_iter"] * 1e-3) / 1e9, 1)
            res["speedup_vs_dense"] = round(res["dense_cublas"]["ms_per_iter"] / res["sparse"]["ms_per_iter"], 3)
            res["layers"] = [{"out": L.out_features, "in": L.in_features, "nnz": int(L.col_idx.numel()),
                              "density": round(L.col_idx.numel() / (L.out_features * L.in_features), 4)}
                             for L in layers]
            res["block"] = wl.FLY_MLPS[mlp]["block"]
            res["tokens"] = T
            out[mlp] = res
            del layers, dense_w, X, dY, vals, vt
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
    return out


def run_e2e(sp, w, dev, idx, args, flops, ws):
    """Same metric through the public calls, with every step's inputs copied from pinned host
    memory and its results copied back inside the timed region. The copies run on their own
    streams, two steps deep: step i's host-to-device copies overlap step i-1's operators and
    step i-2's result copies (events order each buffer's reuse), as a pipelined job would."""
    host = {k: v.contiguous().pin_memory() for k, v in host_inputs(w, idx).items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    shapes = {}
    if w.B is not None:
        shapes["C"] = (w.m, w.B.shape[1])
    if w.A is not None:
        shapes["G"] = (w.nnz,)
    if w.W is not None:
        shapes["D"] = (w.m, w.n)
    depth = 2
    res = [{k: torch.empty(sh, dtype=w.values.dtype).pin_memory() for k, sh in shapes.items()} for _ in range(depth)]
    d2h = sum(v.numel() * v.element_size() for v in res[0].values())
    dbuf = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(depth)]
    s_in, s_op, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    ev_in = [ev() for _ in range(depth)]      # inputs of the slot copied in
    ev_used = [ev() for _ in range(depth)]    # the slot's inputs consumed by the operators
    ev_op = [ev() for _ in range(depth)]      # the slot's results computed
    ev_out = [ev() for _ in range(depth)]     # the slot's results copied out
    for e in ev_used + ev_out:
        e.record(s_op)

    def step(i):
        k = i % depth
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_used[k])
            for name, t in host.items():
                dbuf[k][name].copy_(t, non_blocking=True)
            ev_in[k].record(s_in)
        with torch.cuda.stream(s_op):
            s_op.wait_event(ev_in[k])
            s_op.wait_event(ev_out[k])
            outs = {}
            for _, f in make_ops(sp, w, dbuf[k], idx, args, outs):
                f()
            ev_used[k].record(s_op)
            ev_op[k].record(s_op)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_op[k])
            for name, t in res[k].items():
                outs[name].record_stream(s_out)
                t.copy_(outs[name], non_blocking=True)
            ev_out[k].record(s_out)

    for i in range(max(2, args.warmup)):
        step(i)
    torch.cuda.synchronize(dev)
    steps = max(3, min(args.steps, 200))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_op.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(steps):
        step(i)
    s_in.wait_stream(s_out)
    s_in.wait_stream(s_op)
    e1.record(s_in)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    link = host_link_bound(dev, h2d, d2h, ms)
    return {"value": round(ws * flops / (ms * 1e-3) / 1e9, 2), "unit": "GFLOP/s", "ms_per_step": round(ms, 4),
            "steps": steps, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "link": link,
            "note": "pinned host buffers; copies on separate streams, two steps in flight"}


def host_link_bound(dev, h2d, d2h, ms):
    """The host link's own limit for the step's copies: pinned copy bandwidth measured here in
    each direction alone and in both at once (as the pipelined step runs them), and the step
    time those copies need at that rate: the end-to-end leg cannot beat it."""
    nb = 64 << 20
    hs, hd = torch.empty(nb, dtype=torch.uint8).pin_memory(), torch.empty(nb, dtype=torch.uint8).pin_memory()
    ds, dd = torch.empty(nb, dtype=torch.uint8, device=dev), torch.empty(nb, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def rate(h2d_on, d2h_on, reps=8):
        for r in range(reps + 2):
            if r == 2:
                torch.cuda.synchronize(dev)
                t0 = time.perf_counter()
            if h2d_on:
                with torch.cuda.stream(s1):
                    ds.copy_(hs, non_blocking=True)
            if d2h_on:
                with torch.cuda.stream(s2):
                    hd.copy_(dd, non_blocking=True)
        torch.cuda.synchronize(dev)
        return nb * reps / (time.perf_counter() - t0) / 1e9

    up, down, both = rate(True, False), rate(False, True), rate(True, True)
    common = min(h2d, d2h)  # bytes that move while the other direction is busy too
    bound_ms = (common / (both * 1e9) + (h2d - common) / (up * 1e9) + (d2h - common) / (down * 1e9)) * 1e3
    return {"h2d_gbs": round(up, 1), "d2h_gbs": round(down, 1), "both_ways_gbs_each": round(both, 1),
            "bound_ms_per_step": round(bound_ms, 4), "frac_of_bound": round(bound_ms / ms, 3) if ms > 0 else None}


# ------------------------------------------------------------------ CPU oracle


class OracleStep:
    """The step on the fp64 oracle, on all rows or on a row sample (bounded CPU time)."""

    def __init__(self, w, acc, target_gflop: float):
        import oracle as o
        o.build()
        self.o = o
        self.w = w
        self.ro, self.col = w.row_offsets.numpy(), w.col_idx.numpy()
        self.vals = w.values.double().numpy()
        self.dense = {k: getattr(w, k).double().numpy() for k in ("B", "A", "BT", "W") if getattr(w, k) is not None}
        lens = np.diff(self.ro)
        per_row = 2 * lens * ((w.B.shape[1] if w.B is not None else 0) + (w.A.shape[1] if w.A is not None else 0))
        total = float(per_row.sum())
        if total <= target_gflop * 1e9:
            self.rows = None
            self.flops = step_flops(acc)
            self.sample = "full workload"
        else:
            frac = target_gflop * 1e9 / total
            self.rows = np.sort(np.random.default_rng(0).choice(w.m, size=max(1, int(w.m * frac)), replace=False))
            self.flops = float(per_row[self.rows].sum())
            self.sample = f"{self.rows.size} random rows of {w.m} (all operators on those rows)"

    def __call__(self):
        o, d, r = self.o, self.dense, self.rows
        o.sort_rows(self.ro)
        if "B" in d:
            o.spmm(self.ro, self.col, self.vals, d["B"], rows=r)
        if "A" in d:
            o.sddmm(self.ro, self.col, d["A"], d["BT"], rows=r)
        if "W" in d:
            o.csr_add(self.ro, self.col, self.vals, d["W"], rows=r)


def _time_oracle(st, seconds):
    st()
    n, t0 = 0, time.perf_counter()
    while True:
        st()
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return (time.perf_counter() - t0) / n, n


def cpu_baseline(w, acc, seconds: float, single_thread: bool = False):
    """The oracle as it stands on the host cores (all of them, and one when single_thread)
    on a bounded sample of the workload (about 2 GFLOP per step)."""
    st = OracleStep(w, acc, target_gflop=2.0)
    dt, n = _time_oracle(st, seconds)
    out = {"value": round(st.flops / dt / 1e9, 3), "unit": "GFLOP/s", "cores": st.o.num_threads(), "kind": "oracle",
           "sample": f"{st.sample}; {n} step(s) of sort_rows+spmm+sddmm+csr_add in fp64",
           "ms_per_step": round(dt * 1e3, 2)}
    if single_thread:
        threads = st.o.num_threads()
        st.o.set_threads(1)
        try:
            dt1, n1 = _time_oracle(st, seconds)
        finally:
            st.o.set_threads(threads)
        out["single_thread"] = {"value": round(st.flops / dt1 / 1e9, 3), "cores": 1, "steps": n1,
                                "ms_per_step": round(dt1 * 1e3, 2)}
    return out


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    name = headline_name(args)
    w = wl.generate(name)
    acc = accounting(w)
    st = OracleStep(w, acc, target_gflop=2.0)
    for _ in range(min(args.warmup, 1)):
        st()
    steps = max(1, min(args.steps, args.ref_max_steps))
    t0 = time.perf_counter()
    for _ in range(steps):
        st()
    dt = (time.perf_counter() - t0) / steps
    value = round(st.flops / dt / 1e9, 3)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": ws, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generators in the workloads package)",
            "config": config_dict(name, w, args),
            "cpu_baseline": {"value": value, "unit": "GFLOP/s", "cores": st.o.num_threads(), "kind": "oracle",
                             "sample": f"{st.sample}, {steps} step(s)"},
            "e2e": {"value": value, "unit": "GFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="all", choices=["all"] + list(wl.SPECS),
                    help="all: every configuration, headline on the butterfly layer")
    ap.add_argument("--sddmm-backend", default="structure_aware", choices=["structure_aware", "general"])
    ap.add_argument("--spmm-path", default="auto", choices=["auto", "general"])
    ap.add_argument("--cpu-seconds", type=float, default=3.0)
    ap.add_argument("--breakdown-steps", type=int, default=200)
    ap.add_argument("--ref-max-steps", type=int, default=20)
    ap.add_argument("--no-next-ops", action="store_true", help="skip timing csr_transpose / dB / masked Adam")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-log-dir", default=None,
                    help="where the raw nvidia-smi clock samples go (default: the temp directory)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl != "reference":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
