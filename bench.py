"""Benchmark of the DSpark fused context-KV write on GB300.

One step = one dspark_ctx_kv_write call over one batch of the workload (all
layers, all heads, one kernel launch).  Default workload: long context
(65,536 tokens = 256 requests x 256 at random offsets below 131,072; 5 layers,
4 KV heads, rotary_dim 16, block size 128, bf16 cache), the largest
single-GPU workload, whose inputs (671 MB of all_kv) and written rows
(671 MB) both exceed the 129 MB L2.

Printed (rank 0, one JSON line): metric/value (compulsory GB/s of the whole
job), rows/s, the kernel's roofline against the measured HBM copy peak, an
end-to-end figure through the public API with host buffers (pinned host to
device copies of each step's inputs and a device to host read of the step's
error word inside the timed region), the CPU oracle as a baseline on a
bounded sample, and the SM clocks sampled during the timed region.

--impl reference times the CPU oracle (the reference arm of this build).
Multi-GPU (torchrun): every rank runs its own replica of the workload (the
write has no exchange step), so scaling is weak.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wk  # noqa: E402

METRIC = "context-KV write GB/s and rows/s on 1 GB300; % of HBM roofline"
UNIT = "GB/s"
# sources of the write kernels and of the host layer that picks one
KERNEL_SRCS = [os.path.join(ROOT, "speculative_decoding_draft_ctx_gb300", "csrc", f)
               for f in ("ctx_kv_tma.cu", "ctx_kv_kernel.cu", "ctx_kv_general.cu", "ctx_kv_warp.cu",
                         "ctx_kv_api.cpp", "ctx_kv_internal.h", "ctx_kv_device.cuh", "ctx_kv_pipe.cuh")]
QK_METRIC = "draft-token QK-norm/RoPE/KV-insert GB/s on 1 GB300; % of HBM roofline"
PROJ_METRIC = "fused context-KV projection + write TFLOP/s on 1 GB300; % of bf16 tensor roofline"
NORM_METRIC = "context-state Gemma RMSNorm GB/s on 1 GB300; % of HBM roofline"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="long_context",
                    choices=[w.name for w in wk.WORKLOADS] + [w.name for w in wk.GENERAL_WORKLOADS] +
                    [w.name for w in wk.QK_WORKLOADS] + [w.name for w in wk.PROJ_WORKLOADS] +
                    [w.name for w in wk.NORM_WORKLOADS],
                    help="a context-KV write workload (gen_*: a layout only the general write takes), a qk_* "
                         "workload of the draft-token QK insert, a proj_* workload of the projection with the "
                         "write fused into it, or an hn_* workload of the hidden-state norm")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--num-ctx", type=int, default=None,
                    help="run a smaller case of the workload (profiling captures): fewer tokens")
    ap.add_argument("--num-blocks", type=int, default=None, help="with --num-ctx: fewer cache blocks")
    ap.add_argument("--events", action="store_true",
                    help="context write: time each launch on its own between two CUDA events (isolated "
                         "launches, each paying its own ramp-up and drain) instead of replaying the timed "
                         "steps back to back from one CUDA graph")
    ap.add_argument("--graph", action="store_true", help="accepted for compatibility: the default")
    ap.add_argument("--layer-slots", type=int, default=0, metavar="G",
                    help="context write: layers split over G KV-cache groups, one slot mapping per group")
    return ap.parse_args(argv)


def select_workload(args) -> wk.Workload:
    """The named workload, or a smaller case of it with the same recipe."""
    wl = wk.WORKLOADS_BY_NAME.get(args.config) or wk.GENERAL_WORKLOADS_BY_NAME[args.config]
    if args.num_ctx is None and args.num_blocks is None:
        return wl
    T = args.num_ctx or wl.num_ctx
    over = {"num_ctx": T, "name": f"{wl.name}[num_ctx={T}"}
    if wl.requests:
        if T % wl.tokens_per_request:
            raise SystemExit("--num-ctx must be a multiple of the tokens per request")
        over["requests"] = T // wl.tokens_per_request
    over["pad_count"] = round(wl.pad_count * T / wl.num_ctx)
    if args.num_blocks:
        over["num_blocks"] = args.num_blocks
        over["name"] += f",num_blocks={args.num_blocks}"
    over["name"] += "]"
    return wl.with_(**over)


# ---------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, pg, device) -> float:
    """The largest `value` over all ranks (the job's time is its slowest rank's)."""
    if pg is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Units per second of the whole job: every rank processes its own replica
    of the workload each step (weak scaling), over the slowest rank's time."""
    return units_per_step * steps * world / (max_ms * 1e-3)


def replica_seed(wl: wk.Workload, rank: int, index: int = 0) -> int:
    """Seed of rank `rank`'s input set `index`: distinct data per replica."""
    return wl.seed + 1000 * rank + index


def measured_peaks(key: str = "hbm_gbs"):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}[key], "fallback"


def kernel_sha() -> str:
    """Hash of the kernel sources' code (comments and whitespace removed):
    recorded DRAM counters are only reported while it matches the one they
    were taken on."""
    import re

    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        with open(path, encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)  # block comments
        src = re.sub(r"//[^\n]*", " ", src)                 # line comments
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("kernel_sha") != kernel_sha():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            sel = str(device_index)
        self.cmd = ["nvidia-smi", "-i", sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "100"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sms.append(float(parts[0]))
                maxs.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs), "reasons": sorted(reasons),
                "samples": len(sms)}


def l2_bytes() -> int:
    try:
        return int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size)
    except Exception:
        return 129 * 2**20


def copy_same_bytes(step_bytes: int, dev, stream, launches: int = 50) -> float:
    """GB/s of a plain PyTorch elementwise copy kernel (dst = src * 1 in
    bf16, exact) when one launch moves the same number of bytes as one write
    step (half read, half written), replayed from one CUDA graph (no host
    gaps, even for a few-MB copy) on rotated buffers that together exceed L2:
    the streaming rate a single SM-kernel launch of this size reaches on this
    GPU, for context beside the long-copy peak.  (A Tensor.copy_ of
    contiguous same-dtype buffers is a memcpy, which a graph runs on a copy
    engine at about half the rate, so it is not used here.)"""
    half = max(16, (step_bytes // 2) // 16 * 16)
    n_sets = max(1, math.ceil(3 * l2_bytes() / (2 * half)))
    bufs = [(torch.empty(half // 2, dtype=torch.bfloat16, device=dev).fill_(1.0),
             torch.empty(half // 2, dtype=torch.bfloat16, device=dev)) for _ in range(n_sets)]
    for i in range(5):
        torch.mul(bufs[i % n_sets][0], 1, out=bufs[i % n_sets][1])
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for i in range(launches):
            src, dst = bufs[i % n_sets]
            torch.mul(src, 1, out=dst)
    stream.wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / launches
    del graph, bufs
    return 2 * half / (ms * 1e-3) / 1e9


# ---------------------------------------------------------------- CPU oracle

class OracleSample:
    """The oracle's write over the first `tokens` tokens of a workload, set
    up once and timed per run."""

    def __init__(self, inp: wk.Inputs, tokens: int):
        import oracle

        self.sub = wk.take_tokens(inp, tokens)
        self.p = oracle.problem_from_inputs(self.sub)
        p = self.p
        # host caches stay untouched except for the sampled rows (lazily backed)
        shape = (p.num_blocks, p.H, p.block_size, p.row)
        self.caches = [np.empty(shape, dtype=p.elem_dtype) for _ in range(p.L)]
        nv = self.sub.num_valid_tokens
        self.bytes = wk.compulsory_bytes(self.sub.workload, nv)
        self.rows = nv * p.L * p.H
        self.tokens = tokens

    def run(self) -> float:
        t0 = time.perf_counter()
        self.p.write(self.caches, alt_cap=1 << 20)
        return time.perf_counter() - t0


def calibrate_tokens(inp: wk.Inputs, seconds: float) -> int:
    probe = min(inp.workload.num_ctx, 256)
    s = OracleSample(inp, probe)
    s.run()
    per_tok = max(s.run() / probe, 1e-7)
    return int(max(1, min(inp.workload.num_ctx, seconds / per_tok)))


def cpu_baseline(inp: wk.Inputs, seconds: float):
    """The oracle on a bounded sample: one thread as it stands (the line's
    value), and the same sample split over every host core by token ranges
    (each thread the unchanged single-threaded write on its own tokens)."""
    n = calibrate_tokens(inp, seconds)
    s = OracleSample(inp, n)
    dt = s.run()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    t0 = time.perf_counter()
    s.p.write_threads(s.caches, cores)
    dt_all = time.perf_counter() - t0
    return {
        "value": s.bytes / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
        "rows_per_s": s.rows / dt, "seconds": dt,
        "sample": f"first {n} of {inp.workload.num_ctx} tokens ({s.rows} valid rows), one thread, plain C oracle",
        "all_cores": {"value": s.bytes / dt_all / 1e9, "unit": UNIT, "cores": cores, "seconds": dt_all,
                      "sample": "the same tokens split over every host core by token ranges"},
    }


def run_reference_qk(args):
    """The reference arm for a draft-token QK-insert workload: the oracle on a
    bounded sample (the first tokens of the call) per step."""
    import oracle

    wl = wk.QK_WORKLOADS_BY_NAME[args.config]
    inp = wk.generate_qk(wl)
    p = oracle.qk_problem_from_inputs(inp)
    per_step = 90.0 / max(1, args.steps + args.warmup)
    probe = min(wl.num_tokens, 14)
    t = time.perf_counter()
    p.run(cache=p.new_cache(), q_fp8=wl.q_fp8, t_end=probe)
    per_tok = max((time.perf_counter() - t) / probe, 1e-7)
    n = int(max(1, min(wl.num_tokens, per_step / per_tok)))
    nvalid = int((inp.slot_mapping[:n] >= 0).sum())
    sample_bytes = wk.qk_compulsory_bytes(wl, nvalid, num_tokens=n)
    cache = p.new_cache()
    for _ in range(args.warmup):
        p.run(cache=cache, q_fp8=wl.q_fp8, t_end=n)
    total = 0.0
    for _ in range(args.steps):
        t = time.perf_counter()
        p.run(cache=cache, q_fp8=wl.q_fp8, t_end=n)
        total += time.perf_counter() - t
    value = sample_bytes * args.steps / total / 1e9
    sample = f"first {n} of {wl.num_tokens} tokens per step, one thread, plain C oracle"
    line = {
        "impl": "reference", "metric": QK_METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": dict(wk.describe_qk(wl), sample_tokens=n),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    if args.config in wk.QK_WORKLOADS_BY_NAME:
        return run_reference_qk(args)
    if args.config in wk.PROJ_WORKLOADS_BY_NAME:
        return run_reference_proj(args)
    if args.config in wk.NORM_WORKLOADS_BY_NAME:
        return run_reference_norm(args)
    wl = select_workload(args)
    inp = wk.generate(wl)
    budget = 90.0  # seconds of oracle work for the whole run
    per_step = budget / max(1, args.steps + args.warmup)
    n = calibrate_tokens(inp, per_step)
    sample = OracleSample(inp, n)
    for _ in range(args.warmup):
        sample.run()
    total_t = sum(sample.run() for _ in range(args.steps))
    total_b = sample.bytes * args.steps
    total_r = sample.rows * args.steps
    value = total_b / total_t / 1e9
    sample = f"first {n} of {wl.num_ctx} tokens per step, one thread, plain C oracle"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": dict(wk.describe(wl), sample_tokens=n),
        "rows_per_s": total_r / total_t,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU

def run_ours(args):
    import speculative_decoding_draft_ctx_gb300 as dk

    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    dk.lib()

    wl = select_workload(args)
    base = wk.generate(wl, seed=replica_seed(wl, rank))
    fp8 = wl.kv_dtype == wk.KV_FP8
    nvalid = base.num_valid_tokens
    step_bytes = wk.compulsory_bytes(wl, nvalid)
    step_rows = nvalid * wl.num_layers * wl.num_kv_heads

    # input sets rotated across steps so that each step's reads and writes
    # miss L2 (one set when the workload alone is larger than L2)
    foot = base.all_kv.numel() * 2 + step_rows * wl.row_elems * wl.elem_size
    n_sets = max(1, math.ceil(3 * l2_bytes() / foot))
    sets = []
    for i in range(n_sets):
        inp = base if i == 0 else wk.generate(wl, seed=replica_seed(wl, rank, i))
        sets.append(inp.to(dev))
    k_scales = [sets[0].k_scale[l:l + 1].clone() for l in range(wl.num_layers)]
    v_scales = [sets[0].v_scale[l:l + 1].clone() for l in range(wl.num_layers)]
    caches = wk.make_caches(wl, device=dev, fill=None)
    general = not wk.pages_layout(wl)
    writer = dk.ContextKVWriter(caches, k_scales, v_scales, "fp8" if fp8 else "auto", general=general)
    stream = torch.cuda.current_stream()

    if args.layer_slots:
        for d in sets:
            ls = wk.layer_slot_mappings(d.to("cpu"), groups=args.layer_slots).to(dev)
            d.extra["slots"] = [ls[l] for l in range(wl.num_layers)]
        # every layer's rows are written at its own group's slots: the valid rows of each layer count
        step_rows = int(sum(int((s >= 0).sum()) for s in sets[0].extra["slots"])) * wl.num_kv_heads
        valid_layer_tokens = step_rows // wl.num_kv_heads
        step_bytes = (valid_layer_tokens * wl.num_kv_heads * (2 * wl.row_elems + wl.row_elems * wl.elem_size) +
                      wk.compulsory_bytes(wl, 0) + base.num_valid_tokens * (8 + 2 * wl.rotary_dim) +
                      8 * wl.num_ctx * (wl.num_layers - 1))

    # per-layer mappings: each input set has its own slot tensors, so its own
    # writer (and pointer table): nothing is rebuilt while a graph captures
    writers = ([dk.ContextKVWriter(caches, k_scales, v_scales, "fp8" if fp8 else "auto", general=general)
                for _ in range(n_sets)] if args.layer_slots else [writer])

    def step(i):
        d = sets[i % n_sets]
        slots = d.extra["slots"] if args.layer_slots else d.slot_mapping
        writers[i % len(writers)](d.all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, slots)

    for i in range(max(args.warmup, n_sets if args.layer_slots else 0)):
        step(i)
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    graph = None
    if not args.events:
        # the timed steps as one graph: one launch per step back to back, no
        # host gaps (each launch's prologue overlaps the previous one's drain,
        # as in a serving step); --events times isolated launches instead
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            # an eager call of every writer on the capture stream first: the
            # writer makes its work counters outside capture only
            for i in range(len(writers)):
                step(i)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for i in range(args.steps):
                step(i)
        stream.wait_stream(side)
        graph.replay()  # untimed warm replay
        torch.cuda.synchronize()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_begin.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(args.steps):
                starts[i].record(stream)
                step(i)
                ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    if pg:
        pg.barrier()
    total_ms = t_begin.elapsed_time(t_end)
    if graph is not None:
        launch_ms = [total_ms / args.steps]
    else:
        launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(total_ms, pg, dev)
    avg_launch_ms = sum(launch_ms) / len(launch_ms)
    value = whole_job_rate(step_bytes, args.steps, ws, total_ms) / 1e9
    rows_per_s = whole_job_rate(step_rows, args.steps, ws, total_ms)

    peak, peak_kind = measured_peaks()
    achieved = step_bytes / (avg_launch_ms * 1e-3) / 1e9
    traffic = None if args.layer_slots else recorded_traffic(wl.name)
    copy_gbs = copy_same_bytes(step_bytes, dev, stream)

    # end to end through the public API: pinned host inputs copied in, the
    # step's error word read back, every step
    e2e = None
    if not args.no_e2e:
        host = wk.generate(wl, seed=replica_seed(wl, rank))
        h_kv = host.all_kv.pin_memory()
        h_pos = host.positions.pin_memory()
        h_slot = host.slot_mapping.pin_memory()
        # two device input sets: step i+1's host-to-device copies (on a copy
        # stream) run while step i's write runs on the compute stream
        s0 = sets[0]
        bufs = [s0, sets[1] if n_sets > 1 else
                wk.Inputs(wl, s0.all_kv.clone(), s0.knorm_w, s0.positions.clone(), s0.slot_mapping.clone(),
                          s0.cos_sin, s0.k_scale, s0.v_scale, s0.eps)]
        copy_stream = torch.cuda.Stream()
        copied = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]
        flags = torch.zeros(1, dtype=torch.int32, device=dev)
        h_flags = torch.zeros(1, dtype=torch.int32).pin_memory()
        ne = max(1, args.e2e_steps)
        h2d_bytes = h_kv.numel() * 2 + h_pos.numel() * 8 + h_slot.numel() * 8

        def e2e_step(i):
            d = bufs[i % 2]
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(consumed[i % 2])  # the write two steps back is done with this set
                d.all_kv.copy_(h_kv, non_blocking=True)
                d.positions.copy_(h_pos, non_blocking=True)
                d.slot_mapping.copy_(h_slot, non_blocking=True)
                copied[i % 2].record(copy_stream)
            stream.wait_event(copied[i % 2])
            writer(d.all_kv, d.knorm_w, d.eps, d.positions, d.cos_sin, wl.rotary_dim, d.slot_mapping,
                   error_flags=flags)
            consumed[i % 2].record(stream)
            h_flags.copy_(flags, non_blocking=True)

        for e in consumed:
            e.record(stream)
        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        # the host-to-device rate alone, for context
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for i in range(3):
            bufs[i % 2].all_kv.copy_(h_kv, non_blocking=True)
        c1.record(stream)
        torch.cuda.synchronize()
        h2d_gbs = 3 * h_kv.numel() * 2 / (c0.elapsed_time(c1) * 1e-3) / 1e9
        if pg:
            pg.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_stream.wait_event(e0)
        for i in range(ne):
            e2e_step(i)
        stream.wait_stream(copy_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1), pg, dev)
        if int(h_flags.item()) != 0:
            raise RuntimeError(f"write reported error flags {int(h_flags.item())}")
        e2e = {"value": whole_job_rate(step_bytes, ne, ws, e_ms) / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": 4, "steps": ne, "ms_per_step": e_ms / ne,
               "h2d_gbs_alone": h2d_gbs, "overlap": "step i+1's copies on a copy stream during step i's write"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(base, args.cpu_seconds)

    if rank == 0:
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(wk.describe(wl), parallelism=f"replicas{ws}", input_sets=n_sets,
                           slot_mappings=(f"per layer, {args.layer_slots} KV-cache groups" if args.layer_slots
                                          else "shared"),
                           timing="one CUDA graph of all steps" if graph is not None else "CUDA events per launch",
                           l2=("inputs larger than L2" if n_sets == 1 else
                               f"{n_sets} input sets rotated, footprint > 3x L2")),
            "rows_per_s": rows_per_s,
            "bytes_per_step": step_bytes,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "peak_source": peak_kind,
                         "frac_of_8tbs": achieved / 8000.0,
                         "copy_same_bytes_gbs": copy_gbs, "frac_of_copy_same_bytes": achieved / copy_gbs},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clocks,
            "gpu_launches": args.steps,
            "kernel_avg_us": avg_launch_ms * 1e3,
            "kernel_median_us": statistics.median(launch_ms) * 1e3,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def run_qk(args):
    """The draft-token fused QK-norm / RoPE / KV insert: one launch per step
    over one draft batch, replayed from a CUDA graph (a launch-bound few-MB
    call) over rotated input sets whose footprint exceeds L2."""
    import speculative_decoding_draft_ctx_gb300 as dk

    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    dk.lib()
    wl = wk.QK_WORKLOADS_BY_NAME[args.config]
    base = wk.generate_qk(wl, seed=wl.seed + 1000 * rank)
    step_bytes = wk.qk_compulsory_bytes(wl, base.num_valid_tokens)
    foot = step_bytes
    n_sets = max(1, math.ceil(3 * l2_bytes() / foot))
    sets = [(base if i == 0 else wk.generate_qk(wl, seed=wl.seed + 1000 * rank + i)).to(dev) for i in range(n_sets)]
    caches = [wk.make_qk_cache(wl, device=dev, fill=0) for _ in range(n_sets)]
    qf = [torch.empty((wl.num_tokens, wl.num_heads * 128), dtype=torch.uint8, device=dev) if wl.q_fp8 else None
          for _ in range(n_sets)]
    ks = torch.tensor([base.k_scale], dtype=torch.float32, device=dev)
    vs = torch.tensor([base.v_scale], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        j = i % n_sets
        d = sets[j]
        dk.qknorm_rope_kv_insert(d.qkv, d.q_norm_w, d.k_norm_w, d.cos_sin, d.positions, wl.num_heads,
                                 wl.num_kv_heads, wl.rotary_dim, d.eps, slot_mapping=d.slot_mapping,
                                 kv_cache=caches[j], k_scale=ks, v_scale=vs, q_fp8_out=qf[j],
                                 q_fp8_scale=d.q_scale)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for i in range(args.steps):
            step(i)
    stream.wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0.record(stream)
        graph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
    if pg:
        pg.barrier()
    total_ms = max_over_ranks(t0.elapsed_time(t1), pg, dev)
    launch_ms = total_ms / args.steps
    value = whole_job_rate(step_bytes, args.steps, ws, total_ms) / 1e9
    peak, peak_kind = measured_peaks()
    achieved = step_bytes / (launch_ms * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        host = wk.generate_qk(wl, seed=wl.seed + 1000 * rank)
        h_qkv, h_pos, h_slot = host.qkv.pin_memory(), host.positions.pin_memory(), host.slot_mapping.pin_memory()
        d = sets[0]
        flags = torch.zeros(1, dtype=torch.int32, device=dev)
        h_flags = torch.zeros(1, dtype=torch.int32).pin_memory()
        h_q = torch.empty_like(d.qkv, device="cpu").pin_memory()
        ne = max(1, args.e2e_steps)

        def e2e_step():
            d.qkv.copy_(h_qkv, non_blocking=True)
            d.positions.copy_(h_pos, non_blocking=True)
            d.slot_mapping.copy_(h_slot, non_blocking=True)
            dk.qknorm_rope_kv_insert(d.qkv, d.q_norm_w, d.k_norm_w, d.cos_sin, d.positions, wl.num_heads,
                                     wl.num_kv_heads, wl.rotary_dim, d.eps, slot_mapping=d.slot_mapping,
                                     kv_cache=caches[0], k_scale=ks, v_scale=vs, q_fp8_out=qf[0],
                                     q_fp8_scale=d.q_scale, error_flags=flags)
            h_q.copy_(d.qkv, non_blocking=True)
            h_flags.copy_(flags, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(ne):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1), pg, dev)
        if int(h_flags.item()) != 0:
            raise RuntimeError(f"insert reported error flags {int(h_flags.item())}")
        e2e = {"value": whole_job_rate(step_bytes, ne, ws, e_ms) / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": h_qkv.numel() * 2 + h_pos.numel() * 8 + h_slot.numel() * 8,
               "d2h_bytes_per_step": h_q.numel() * 2 + 4, "steps": ne, "ms_per_step": e_ms / ne}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle

        p = oracle.qk_problem_from_inputs(base)
        cache = p.new_cache()
        t = time.perf_counter()
        p.run(cache=cache, q_fp8=wl.q_fp8)
        dt = time.perf_counter() - t
        cpu = {"value": step_bytes / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle", "seconds": dt,
               "sample": f"the whole call ({wl.num_tokens} tokens), one thread, plain C oracle"}
    if rank == 0:
        line = {
            "metric": QK_METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(wk.describe_qk(wl), parallelism=f"replicas{ws}", input_sets=n_sets,
                           timing="one CUDA graph of all steps",
                           l2=f"{n_sets} input sets rotated, footprint > 3x L2"),
            "bytes_per_step": step_bytes,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None, "peak_source": peak_kind,
                         "frac_of_8tbs": achieved / 8000.0},
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clk.summary(), "gpu_launches": args.steps,
            "kernel_avg_us": launch_ms * 1e3,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def run_proj(args):
    """The context-KV projection with the write fused into its epilogue: one
    tensor-core launch per step (all_kv never reaches HBM), input sets
    rotated so that each step's operands miss L2.  Beside it, timed the same
    way: the library's projection alone, PyTorch's (cuBLAS) matmul alone, and
    the unfused path a user would otherwise run (cuBLAS projection, then the
    library's write kernel)."""
    import speculative_decoding_draft_ctx_gb300 as dk

    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    dk.lib()
    wl = wk.PROJ_WORKLOADS_BY_NAME[args.config]
    b = wl.base
    flops = wk.proj_flops(wl)
    foot = (b.num_ctx + wl.n_out) * wl.hidden * 2
    n_sets = max(1, math.ceil(3 * l2_bytes() / foot))
    sets = [wk.generate_proj(wl, seed=b.seed + 500 + 1000 * rank + i).to(dev) for i in range(n_sets)]
    d0 = device_inputs_ctx(sets[0].ctx)
    fp8 = b.kv_dtype == wk.KV_FP8
    caches = wk.make_caches(b, device=dev, fill=None)
    writer = dk.ContextKVWriter(caches, d0["k_scales"], d0["v_scales"], "fp8" if fp8 else "auto")
    stream = torch.cuda.current_stream()
    all_kv = torch.empty((b.num_ctx, b.num_layers, 2, b.num_kv_heads, 128), dtype=torch.bfloat16, device=dev)

    def fused(i):
        s_ = sets[i % n_sets]
        c = s_.ctx
        writer.project_and_write(s_.x, s_.w_kv, c.knorm_w, c.eps, c.positions, c.cos_sin, b.rotary_dim,
                                 c.slot_mapping)

    def project_only(i):
        s_ = sets[i % n_sets]
        dk.project_context_kv(s_.x, s_.w_kv, b.num_layers, b.num_kv_heads, out=all_kv)

    def cublas_only(i):
        s_ = sets[i % n_sets]
        torch.matmul(s_.x, s_.w_kv.t(), out=all_kv.view(b.num_ctx, -1))

    def unfused(i):
        s_ = sets[i % n_sets]
        c = s_.ctx
        torch.matmul(s_.x, s_.w_kv.t(), out=all_kv.view(b.num_ctx, -1))
        writer(all_kv, c.knorm_w, c.eps, c.positions, c.cos_sin, b.rotary_dim, c.slot_mapping)

    def timed(fn, steps):
        for i in range(args.warmup):
            fn(i)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        t0.record(stream)
        for i, (a, z) in enumerate(ev):
            a.record(stream)
            fn(i)
            z.record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        per = sum(a.elapsed_time(z) for a, z in ev) / steps
        return max_over_ranks(t0.elapsed_time(t1), pg, dev), per

    with ClockSampler(local) as clk:
        total_ms, fused_ms = timed(fused, args.steps)
    side_steps = max(10, min(args.steps, 200))
    _, proj_ms = timed(project_only, side_steps)
    _, cublas_ms = timed(cublas_only, side_steps)
    _, unfused_ms = timed(unfused, side_steps)
    value = whole_job_rate(flops, args.steps, ws, total_ms) / 1e12
    # the timed loop is one launch after another: while the sampled clocks
    # show the power cap, the sustained cuBLAS figure is the fair peak, else
    # the burst one
    clocks = clk.summary()
    capped = "sw_power_cap" in (clocks or {}).get("reasons", [])
    peak, peak_kind = measured_peaks("bf16_tflops_sustained" if capped else "bf16_tflops")
    peak_kind += " sustained (power cap seen)" if capped else " burst"
    achieved = flops / (fused_ms * 1e-3) / 1e12

    e2e = None
    if not args.no_e2e:
        h_x = sets[0].x.cpu().pin_memory()
        d = sets[0]
        flags = torch.zeros(1, dtype=torch.int32, device=dev)
        h_flags = torch.zeros(1, dtype=torch.int32).pin_memory()
        ne = max(1, args.e2e_steps)

        def e2e_step():
            d.x.copy_(h_x, non_blocking=True)
            c = d.ctx
            writer.project_and_write(d.x, d.w_kv, c.knorm_w, c.eps, c.positions, c.cos_sin, b.rotary_dim,
                                     c.slot_mapping, error_flags=flags)
            h_flags.copy_(flags, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(ne):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1), pg, dev)
        if int(h_flags.item()) != 0:
            raise RuntimeError(f"projection write reported error flags {int(h_flags.item())}")
        e2e = {"value": whole_job_rate(flops, ne, ws, e_ms) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h_x.numel() * 2, "d2h_bytes_per_step": 4, "steps": ne,
               "ms_per_step": e_ms / ne}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        n = min(b.num_ctx, 16)
        dt = proj_oracle_sample(wl, n)
        cpu = {"value": 2 * n * wl.n_out * wl.hidden / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
               "kind": "oracle", "seconds": dt,
               "sample": f"first {n} of {b.num_ctx} tokens: fp64 numpy matmul (BLAS threads) + C write oracle"}
    if rank == 0:
        line = {
            "metric": PROJ_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(wk.describe(b), workload=wl.name, hidden=wl.hidden, n_out=wl.n_out,
                           parallelism=f"replicas{ws}", input_sets=n_sets, timing="CUDA events per launch",
                           l2=("inputs larger than L2" if n_sets == 1 else
                               f"{n_sets} input sets rotated, footprint > 3x L2")),
            "flops_per_step": flops,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": None, "peak_source": peak_kind},
            "compare_ms_per_step": {"fused_projection_write": fused_ms, "projection_alone": proj_ms,
                                    "cublas_matmul_alone": cublas_ms,
                                    "unfused_cublas_matmul_then_write": unfused_ms},
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks, "gpu_launches": args.steps,
            "kernel_avg_us": fused_ms * 1e3,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def run_norm(args):
    """The hidden-state Gemma RMSNorm of the context states: one launch per
    step, CUDA events per launch, input sets rotated past L2; beside it the
    unfused PyTorch composition (fp32 ops) timed the same way."""
    import speculative_decoding_draft_ctx_gb300 as dk

    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    dk.lib()
    wl = wk.NORM_WORKLOADS_BY_NAME[args.config]
    step_bytes = wk.norm_bytes(wl)
    n_sets = max(1, math.ceil(3 * l2_bytes() / step_bytes))
    sets = []
    for i in range(n_sets):
        x, w, eps = wk.generate_norm(wl, seed=wl.seed + 1000 * rank + i)
        sets.append((x.to(dev), w.to(dev), torch.empty_like(x, device=dev)))
    stream = torch.cuda.current_stream()

    def ours(i):
        x, w, o = sets[i % n_sets]
        dk.gemma_rms_norm(x, w, wl.eps, out=o)

    def unfused(i):
        x, w, o = sets[i % n_sets]
        xf = x.float()
        o.copy_((xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + wl.eps) * (1.0 + w.float())).to(torch.bfloat16))

    def timed(fn, steps):
        """The steps replayed from one CUDA graph (no host launch gaps:
        a 10 us launch is shorter than the host's launch path)."""
        for i in range(args.warmup):
            fn(i)
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for i in range(steps):
                fn(i)
        stream.wait_stream(side)
        graph.replay()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        t0.record(stream)
        graph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        ms = t0.elapsed_time(t1)
        del graph
        return max_over_ranks(ms, pg, dev), ms / steps

    with ClockSampler(local) as clk:
        total_ms, ours_ms = timed(ours, args.steps)
    _, unfused_ms = timed(unfused, max(10, min(args.steps, 200)))
    value = whole_job_rate(step_bytes, args.steps, ws, total_ms) / 1e9
    peak, peak_kind = measured_peaks()
    achieved = step_bytes / (ours_ms * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        hx = sets[0][0].cpu().pin_memory()
        ho = torch.empty_like(hx).pin_memory()
        x, w, o = sets[0]
        ne = max(1, args.e2e_steps)

        def e2e_step():
            x.copy_(hx, non_blocking=True)
            dk.gemma_rms_norm(x, w, wl.eps, out=o)
            ho.copy_(o, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(ne):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1), pg, dev)
        e2e = {"value": whole_job_rate(step_bytes, ne, ws, e_ms) / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": hx.numel() * 2, "d2h_bytes_per_step": ho.numel() * 2, "steps": ne,
               "ms_per_step": e_ms / ne}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle

        x, w, eps = wk.generate_norm(wl)
        n = min(wl.rows, 256)
        xb = x[:n].contiguous().view(torch.int16).numpy().view(np.uint16)
        t = time.perf_counter()
        oracle.gemma_norm_rows(xb, w.view(torch.int16).numpy().view(np.uint16), eps)
        dt = time.perf_counter() - t
        cpu = {"value": 4 * n * wl.hidden / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle", "seconds": dt,
               "sample": f"first {n} of {wl.rows} rows, one thread, plain C oracle"}
    if rank == 0:
        line = {
            "metric": NORM_METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.name, "rows": wl.rows, "hidden": wl.hidden, "parallelism": f"replicas{ws}",
                       "input_sets": n_sets, "timing": "one CUDA graph of all steps",
                       "l2": ("inputs larger than L2" if n_sets == 1 else
                              f"{n_sets} input sets rotated, footprint > 3x L2")},
            "bytes_per_step": step_bytes,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None, "peak_source": peak_kind},
            "compare_ms_per_step": {"fused_norm": ours_ms, "unfused_torch_fp32": unfused_ms},
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clk.summary(), "gpu_launches": args.steps,
            "kernel_avg_us": ours_ms * 1e3,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def proj_oracle_sample(wl, n: int) -> float:
    """Seconds the oracle takes for the projection and write of the first
    ``n`` tokens of a projection workload (fp64 BLAS matmul + C write)."""
    import oracle

    b = wl.base
    inp = wk.generate_proj(wl)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    c = inp.ctx
    sub_ctx = wk.Inputs(b.with_(num_ctx=n), c.all_kv, c.knorm_w, c.positions[:n].contiguous(),
                        c.slot_mapping[:n].contiguous(), c.cos_sin, c.k_scale, c.v_scale, c.eps)
    sub = wk.ProjInputs(wl.with_(base=b.with_(num_ctx=n)), inp.x[:n], inp.w_kv, sub_ctx)
    t = time.perf_counter()
    kv = oracle.project_context_kv(bits(sub.x), bits(sub.w_kv))
    pr = oracle.problem_from_inputs(wk.with_all_kv(sub, kv))
    pr.write(pr.new_caches())
    return time.perf_counter() - t


def run_reference_proj(args):
    """The reference arm of a projection workload: the oracle on the first
    tokens of the call per step (fp64 BLAS matmul + the C write oracle)."""
    wl = wk.PROJ_WORKLOADS_BY_NAME[args.config]
    b = wl.base
    per_step = 90.0 / max(1, args.steps + args.warmup)
    probe = proj_oracle_sample(wl, min(b.num_ctx, 4)) / min(b.num_ctx, 4)
    n = int(max(1, min(b.num_ctx, per_step / max(probe, 1e-7))))
    for _ in range(args.warmup):
        proj_oracle_sample(wl, n)
    total = sum(proj_oracle_sample(wl, n) for _ in range(args.steps))
    value = 2 * n * wl.n_out * wl.hidden * args.steps / total / 1e12
    sample = f"first {n} of {b.num_ctx} tokens per step: fp64 numpy matmul (BLAS threads) + C write oracle"
    line = {
        "impl": "reference", "metric": PROJ_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(wk.describe(b), workload=wl.name, hidden=wl.hidden, sample_tokens=n),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_norm(args):
    """The reference arm of a norm workload: the C oracle on the first rows
    of the call per step."""
    import oracle

    wl = wk.NORM_WORKLOADS_BY_NAME[args.config]
    x, w, eps = wk.generate_norm(wl)
    wb = w.view(torch.int16).numpy().view(np.uint16)
    per_step = 90.0 / max(1, args.steps + args.warmup)
    t = time.perf_counter()
    oracle.gemma_norm_rows(x[:8].contiguous().view(torch.int16).numpy().view(np.uint16), wb, eps)
    per_row = max((time.perf_counter() - t) / 8, 1e-7)
    n = int(max(1, min(wl.rows, per_step / per_row)))
    xb = x[:n].contiguous().view(torch.int16).numpy().view(np.uint16)
    for _ in range(args.warmup):
        oracle.gemma_norm_rows(xb, wb, eps)
    total = 0.0
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.gemma_norm_rows(xb, wb, eps)
        total += time.perf_counter() - t
    value = 4 * n * wl.hidden * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": NORM_METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "rows": wl.rows, "hidden": wl.hidden, "sample_rows": n},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"first {n} of {wl.rows} rows per step, one thread, plain C oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def device_inputs_ctx(ctx):
    """Per-layer fp32 scale tensors (one element each) of a device-side
    context-write input set, like the attention layers' k/v scales."""
    L = ctx.knorm_w.shape[0]
    return {"k_scales": [ctx.k_scale[l:l + 1].clone() for l in range(L)],
            "v_scales": [ctx.v_scale[l:l + 1].clone() for l in range(L)]}


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.config in wk.QK_WORKLOADS_BY_NAME:
        return run_qk(args)
    if args.config in wk.PROJ_WORKLOADS_BY_NAME:
        return run_proj(args)
    if args.config in wk.NORM_WORKLOADS_BY_NAME:
        return run_norm(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
