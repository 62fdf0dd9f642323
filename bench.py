"""Benchmark: BF16 x NVFP4 GEMM on the Llama-3-70B linear shapes.

One step = one pass of the hot path over one batch: the four linear layers of
a Llama-3-70B block (QKV 10240x8192, O 8192x8192, gate_up 57344x8192,
down 8192x28672; W stored [n, k]) at decode size m = 16, NVFP4 weights with
16-element E4M3 scales and global scale 1, A ~ N(0,1), W ~ N(0,0.02)
(synthetic, seeded).  Weights are quantised and repacked offline (before the
timed region).  Two weight sets (2 x 481 MB, more than 3x the 129 MB L2) are
used on alternate steps, so every weight byte comes from HBM.

value = algorithmic bytes (packed weights + scales + A + C) of all steps on
all ranks / max-over-ranks time, in GB/s.  A step is the four GEMM launches
back to back on one stream (programmatic dependent launch lets each kernel's
prologue overlap the previous one's tail; the host runs ahead of the GPU).
The headline is the median of 5 batches of `steps` steps, each batch
bracketed by a barrier and a device synchronisation and timed with CUDA
events.  Further passes replay, per shape, a graph of consecutive launches
that rotate through R = max(2, ceil(3 L2 / weight bytes)) weight copies, to
give each shape's steady-state launch duration.

--impl reference times the FP64 CPU oracle (dequantise + GEMM) on a bounded
sample of the same workload instead.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BF16×NVFP4 GEMM TFLOP/s & HBM GB/s (% roofline), Llama-3-70B shapes m=16/256"
SHAPES = [("qkv", 10240, 8192), ("o", 8192, 8192), ("gate_up", 57344, 8192), ("down", 8192, 28672)]
M_DECODE = 16
M_PREFILL = 256
BATCHES = 5          # the headline is the median of this many timed batches


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prefill", action="store_true")
    p.add_argument("--profile-only", action="store_true",
                   help="prepare one weight set and launch each decode GEMM once (for ncu captures)")
    p.add_argument("--profile-m", type=int, default=M_DECODE)
    p.add_argument("--profile-fmt", choices=["nvfp4", "mxfp4", "nvfp4_f16"], default="nvfp4",
                   help="weight format / activation type of the --profile-only launches")
    p.add_argument("--profile-moe", type=int, default=0, metavar="TOKENS",
                   help="with --profile-only: one MXFP4 MoE grouped GEMM (8 experts, top-2, "
                        "n=28672, k=4096) for TOKENS tokens instead of the four linears")
    p.add_argument("--tile", default=os.environ.get("PETIT_CONFIG", ""), metavar="BN,KU",
                   help="force the GEMM tile shape (activation rows per tile, 128-k chunks per "
                        "unit) for every launch; default: the planner's choice (env PETIT_CONFIG)")
    return p.parse_args()


def apply_tile(args, binding):
    """Forward --tile / PETIT_CONFIG to the library; returns the forced pair."""
    if not args.tile:
        return None
    bn, ku = (int(x) for x in args.tile.split(","))
    binding.set_tile_config(bn, ku)
    return [bn, ku]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, device):
    """The largest of x over all ranks of the process group (x itself when
    no group is initialised)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(step_bytes, steps, world, elapsed_max_ms):
    """Whole-job GB/s: the bytes every rank processed over the slowest rank's
    time (each replica runs the same step)."""
    return world * step_bytes * steps / (elapsed_max_ms * 1e-3) / 1e9


def algo_bytes(m, n, k, scale_group=16):
    """Packed FP4 weights + block scales + A + C bytes of one GEMM."""
    return n * k // 2 + n * k // scale_group + 2 * m * k + 2 * m * n


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def ncu_traffic(kernel_file):
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel source changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", kernel_file)
    src = os.path.join(ROOT, "fp4_weight_only_gb300", "csrc", "gemm.cu")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("-"):
                key, val = line.strip()[1:].split(":", 1)
                fields[key.strip()] = val.strip()
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if fields.get("gemm.cu sha256 prefix") != digest:
        return None
    try:
        return float(fields["dram bytes per launch (gate_up, scaled)"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples (200 ms period), read by a
    background thread as they arrive, each stamped with the host time."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        import threading
        self.proc = None
        self.rows = []            # (host time, sm MHz, max sm MHz, [reason flags])
        self.lock = threading.Lock()
        self.first = threading.Event()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            self.first.set()
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                row = (time.time(), float(parts[0]), float(parts[1]), parts[3:8])
            except ValueError:
                continue
            with self.lock:
                self.rows.append(row)
            self.first.set()
        self.first.set()

    def wait_first(self, timeout=10.0):
        """Block until the first sample has arrived (or nvidia-smi is gone)."""
        self.first.wait(timeout)

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.thread.join(timeout=5)

    def summary(self, windows):
        """Median SM clock over the samples taken inside any of the (t0, t1)
        host-time windows (all samples if none fell inside one), the largest
        max clock, and the throttle reasons seen active."""
        with self.lock:
            rows = list(self.rows)
        inside = [r for r in rows if any(t0 - 0.1 <= r[0] <= t1 + 0.1 for t0, t1 in windows)]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "samples_in_timed_region": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3][1:5]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside),
                "period_ms": 200}


def rotation_copies(weight_bytes, l2_bytes):
    """Weight copies to rotate through so that each launch reads its weights
    from HBM: R = max(2, ceil(3 * L2 / (W + S)))."""
    return max(2, -(-3 * int(l2_bytes) // int(weight_bytes)))


def l2_bytes(dev):
    props = torch.cuda.get_device_properties(dev)
    return int(getattr(props, "L2_cache_size", 0) or 129 * 2**20)


# --------------------------------------------------------------------- oracle
def oracle_sample(weights_cpu, acts_cpu, rows, min_seconds=0.0):
    """Time the FP64 oracle (dequant + GEMM) on the first `rows` rows of each
    weight matrix; quantisation is done first and not timed.  The timed pass
    over the four matrices repeats until `min_seconds` have elapsed.
    Returns (bytes, wall s, passes, process CPU s): the CPU time of all the
    process's threads over the wall time is how many cores the oracle kept
    busy (numpy's dequantise runs on one, its BLAS matrix product on a pool)."""
    from oracle import gemm as og
    from oracle import quantize as oq
    prepared = []
    for (name, n, k), w, a in zip(SHAPES, weights_cpu, acts_cpu):
        codes, scales = oq.nvfp4_quantize(w[:rows].float().numpy(), 1.0)
        prepared.append((a.float().numpy(), codes, scales, k))
    per_pass = sum(algo_bytes(M_DECODE, rows, k) for _, _, _, k in prepared)
    passes = 0
    c0 = time.process_time()
    t0 = time.perf_counter()
    while True:
        for a, codes, scales, k in prepared:
            og.gemm(a, og.dequantize(codes, scales, "nvfp4"), 1.0)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    return per_pass * passes, dt, passes, time.process_time() - c0


def busy_cores(cpu_s, wall_s):
    """Cores kept busy on average (at least 1), from process CPU and wall time."""
    return max(1, round(cpu_s / wall_s)) if wall_s > 0 else 1


def synth_inputs_cpu(rows):
    from fp4_weight_only_gb300 import synth
    ws = [synth.weights(rows, k, seed=100 + i) for i, (_, n, k) in enumerate(SHAPES)]
    acts = [synth.activations(M_DECODE, k, seed=200 + i) for i, (_, n, k) in enumerate(SHAPES)]
    return ws, acts


def decode_config(world):
    """The workload both arms report (the reference arm times a sample of it)."""
    return {"workload": "llama3-70b linears qkv/o/gate_up/down, NVFP4 decode m=16, g=1",
            "m": M_DECODE, "shapes_nk": [[n, k] for _, n, k in SHAPES],
            "parallelism": f"replicas x{world}"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    rows = 96
    ws, acts = synth_inputs_cpu(rows)
    for _ in range(max(args.warmup, 0)):
        oracle_sample(ws, acts, rows)
    total_b, total_t, total_c = 0, 0.0, 0.0
    for _ in range(args.steps):
        b, t, _, c = oracle_sample(ws, acts, rows)
        total_b += b
        total_t += t
        total_c += c
    value = total_b / total_t / 1e9
    cores = busy_cores(total_c, total_t)
    sample = (f"{rows} seeded N(0,0.02) rows for each of the 4 Llama-3-70B weight shapes, m={M_DECODE}; "
              "oracle NVFP4 dequantise + FP64 GEMM per step (quantisation untimed); "
              f"{total_c:.1f} s of CPU in {total_t:.1f} s on a {os.cpu_count()}-core host")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": decode_config(world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------------ GPU
def shape_durations(launchers, stream, reps, min_burst=8):
    """Steady-state duration (ms) of one launch of each shape.  launchers[i]
    holds one launch function per weight copy of shape i; a graph holds at
    least `min_burst` consecutive launches rotating through the copies (so
    each launch reads its weights from HBM, and programmatic dependent launch
    overlaps each prologue with the previous kernel's tail, as inside a step)
    and is replayed `reps` times between two stream events."""
    out = []
    for fns in launchers:                      # fns[w]: launch with weight copy w
        burst = len(fns) * max(1, -(-min_burst // len(fns)))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for b in range(burst):
                fns[b % len(fns)]()
        for _ in range(2):
            g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) / (reps * burst))
    return np.array(out)


def run_ours(args, rank, world, local):
    from fp4_weight_only_gb300 import binding, synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.load()
    tile = apply_tile(args, binding)
    peaks = load_peaks()
    stream = torch.cuda.Stream(dev)        # graphs are captured and replayed off the default stream
    torch.cuda.set_stream(stream)

    # offline preparation: quantise + repack on the GPU (not timed)
    sets = [[], []]
    acts, outs = [], []
    for i, (name, n, k) in enumerate(SHAPES):
        w = synth.weights(n, k, seed=100 + i, device=dev)
        fw = binding.FP4Weight(w, "nvfp4", 1.0)
        del w
        sets[0].append(fw)
        sets[1].append(fw.rep.clone())
        torch.cuda.synchronize()
        acts.append(synth.activations(M_DECODE, k, seed=200 + i, device=dev))
        outs.append(torch.empty((M_DECODE, n), dtype=torch.bfloat16, device=dev))
    ws = binding.Workspace(dev)
    for (name, n, k) in SHAPES:
        ws.ensure(binding.workspace_bytes(M_PREFILL, n, k))
    torch.cuda.synchronize()

    def launch(i, which, m=M_DECODE, a=None, c=None):
        fw = sets[0][i]
        rep = fw.rep if which == 0 else sets[1][i]
        binding.gemm(acts[i] if a is None else a, rep, fw.n, "nvfp4", 1.0, workspace=ws,
                     out=outs[i] if c is None else c)

    # a step: the four GEMMs launched back to back on one stream (each launch
    # carries programmatic dependent launch, so a kernel's prologue overlaps
    # the previous kernel's tail); the host enqueues far ahead of the GPU
    for i in range(len(SHAPES)):
        for which in (0, 1):
            launch(i, which)
    torch.cuda.synchronize()

    def step(s):
        for i in range(len(SHAPES)):
            launch(i, s & 1)

    l2 = l2_bytes(dev)

    def rotated(reps, weight_bytes):
        """`reps` extended by clones to the rotation count for its size."""
        r = rotation_copies(weight_bytes, l2)
        out = list(reps) + [reps[0].clone() for _ in range(r - len(reps))]
        # a GEMM reads its weights while the previous kernel is finishing:
        # the copies must be complete before the first launch that reads them
        torch.cuda.synchronize()
        return out

    # the clock sampler runs from before the warm-up to after the per-shape
    # passes, and the timed region starts only once it has produced a sample
    sampler = ClockSampler(local)
    sampler.wait_first()
    windows = []
    for s in range(args.warmup):
        step(s)
    # the headline: BATCHES batches of `steps` steps each, every batch
    # bracketed by a barrier and a device synchronisation and timed with CUDA
    # events on the launching stream; the median batch (of the max over ranks)
    # is reported
    batch_ms = []
    for _ in range(BATCHES):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        t_host0 = time.time()
        start.record(stream)
        for s in range(args.steps):
            step(s)
        end.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        windows.append((t_host0, time.time()))
        batch_ms.append(max_over_ranks(start.elapsed_time(end), dev))
    elapsed_max = statistics.median(batch_ms)
    # per-shape pass (after the timed region): steady-state launch durations,
    # each shape rotating through enough weight copies to defeat L2
    decode_reps = [rotated([sets[0][i].rep, sets[1][i]], n * k // 2 + n * k // 16)
                   for i, (_, n, k) in enumerate(SHAPES)]

    def launch_rep(i, rep):
        binding.gemm(acts[i], rep, SHAPES[i][1], "nvfp4", 1.0, workspace=ws, out=outs[i])
    t_shapes0 = time.time()
    per_kernel_ms = shape_durations(
        [[(lambda i=i, r=r: launch_rep(i, r)) for r in decode_reps[i]] for i in range(len(SHAPES))],
        stream, max(3, min(args.steps // 8, 50)))
    windows.append((t_shapes0, time.time()))

    step_bytes = sum(algo_bytes(M_DECODE, n, k) for _, n, k in SHAPES)
    step_flops = sum(2 * M_DECODE * n * k for _, n, k in SHAPES)
    ms_per_step = elapsed_max / args.steps
    value = job_gbs(step_bytes, args.steps, world, elapsed_max)
    shapes = {}
    for i, (name, n, k) in enumerate(SHAPES):
        t = per_kernel_ms[i] * 1e-3
        b = algo_bytes(M_DECODE, n, k)
        shapes[name] = {"n": n, "k": k, "us": round(t * 1e6, 2), "gbs": round(b / t / 1e9, 1),
                        "tflops": round(2 * M_DECODE * n * k / t / 1e12, 2),
                        "weight_gbs": round((n * k // 2 + n * k // 16) / t / 1e9, 1),
                        "frac_hbm": round(b / t / 1e9 / peaks["hbm_gbs"], 3),
                        "weight_copies": len(decode_reps[i])}
    del decode_reps
    # the timed region holds only gemm_kernel<NVFP4, BN=16> launches (4 per
    # step), so its average launch duration is elapsed / launches
    launches = len(SHAPES) * args.steps
    avg_launch_s = elapsed_max * 1e-3 / launches
    achieved = (step_bytes / len(SHAPES)) / avg_launch_s / 1e9
    traffic = ncu_traffic("gemm_nvfp4_decode_m16.txt")
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                "kernel": "gemm_kernel<NVFP4, BN=16, KU=2> (the only kernel in the timed region)",
                "per_launch": "average algorithmic bytes of the 4 launches of a step / "
                              "(median batch time / launches per batch)",
                "avg_launch_us": round(avg_launch_s * 1e6, 3),
                "peak_source": peaks["source"] + " hbm_gbs (copy bandwidth)"}

    # e2e: the public binding in a serving loop.  Every step copies its four
    # activation matrices in (one pinned host-to-device copy), runs the four
    # GEMMs and copies their results out (one device-to-host copy into pinned
    # memory), and the host reads each step's results.  Two buffer sets
    # alternate, so step s+1's input copy (copy-in stream) and step s-1's
    # result copy (copy-out stream) overlap step s's GEMMs, and the host
    # waits for step s-1's results while step s runs.
    a_sizes = [M_DECODE * k for _, _, k in SHAPES]
    c_sizes = [M_DECODE * n for _, n, _ in SHAPES]
    a_host_all = torch.cat([a.reshape(-1).cpu() for a in acts]).pin_memory()
    c_host = [torch.empty(sum(c_sizes), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    a_dev_all = [torch.empty(sum(a_sizes), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    c_dev_all = [torch.empty(sum(c_sizes), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    a_dev = [[v.view(M_DECODE, k) for v, (_, _, k) in zip(a_dev_all[b].split(a_sizes), SHAPES)]
             for b in range(2)]
    c_dev = [[v.view(M_DECODE, n) for v, (_, n, _) in zip(c_dev_all[b].split(c_sizes), SHAPES)]
             for b in range(2)]
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for b in range(2):   # every event starts recorded (buffers free)
        for e in (in_done[b], comp_done[b], out_done[b]):
            e.record(stream)
    e2e_steps = max(1, min(args.steps, 200))
    checksum = [0.0]

    def e2e_step(s):
        b = s & 1
        with torch.cuda.stream(cin):      # input copy once step s-2 has read buffer b
            cin.wait_event(comp_done[b])
            a_dev_all[b].copy_(a_host_all, non_blocking=True)
            in_done[b].record(cin)
        stream.wait_event(in_done[b])     # GEMMs once the input landed and step s-2's
        stream.wait_event(out_done[b])    # results left buffer b
        for i, (name, n, k) in enumerate(SHAPES):
            rep = sets[0][i].rep if b == 0 else sets[1][i]
            binding.gemm(a_dev[b][i], rep, n, "nvfp4", 1.0, workspace=ws, out=c_dev[b][i])
        comp_done[b].record(stream)
        with torch.cuda.stream(cout):
            cout.wait_event(comp_done[b])
            c_host[b].copy_(c_dev_all[b], non_blocking=True)
            out_done[b].record(cout)
        if s > 0:                         # the host reads step s-1's results
            out_done[b ^ 1].synchronize()
            checksum[0] += float(c_host[b ^ 1][0])

    for s in range(4):
        e2e_step(s)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(e2e_steps):
        e2e_step(s)
    out_done[(e2e_steps - 1) & 1].synchronize()
    e2e_t = time.perf_counter() - t0
    torch.cuda.synchronize()
    h2d = sum(2 * M_DECODE * k for _, _, k in SHAPES)
    d2h = sum(2 * M_DECODE * n for _, n, _ in SHAPES)
    e2e = {"value": round(world * step_bytes * e2e_steps / e2e_t / 1e9, 1), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "ms_per_step": round(1e3 * e2e_t / e2e_steps, 5),
           "path": "binding.gemm (ctypes -> C ABI) per layer; per step one pinned host-to-device "
                   "copy of the step's activations and one device-to-host copy of its results, "
                   "double-buffered on copy streams; the host reads every step's results one step "
                   "later; host wall clock over the steps"}

    # host cost of one GEMM call (enqueue only): the public binding call, timed
    # on the host over calls that do not fill the launch queue
    torch.cuda.synchronize()
    host_us = []
    for rnd in range(5):
        t_a = time.perf_counter()
        for r_ in range(32):
            binding.gemm(acts[1], sets[0][1].rep, SHAPES[1][1], "nvfp4", 1.0, workspace=ws, out=outs[1])
        host_us.append((time.perf_counter() - t_a) / 32 * 1e6)
        torch.cuda.synchronize()
    e2e["host_us_per_gemm_call"] = round(statistics.median(host_us), 2)

    # prefill m = 256 and the other per-shape lines: per-GEMM timing, each
    # shape rotating through R weight copies
    def prepared(fmt, seed0, gscale):
        """reps[i]: R copies of weight i in `fmt` (g = amax/(6*448) per matrix
        if gscale), with the global scales."""
        reps, gs = [], []
        for i, (name, n, k) in enumerate(SHAPES):
            w = synth.weights(n, k, seed=seed0 + i, device=dev)
            g = binding.nvfp4_global_scale(binding.absmax(w).item()) if gscale else 1.0
            fw = binding.FP4Weight(w, fmt, g)
            del w
            reps.append(rotated([fw.rep], fw.rep.numel()))
            gs.append(g)
        return reps, gs

    def shape_table(fmt, reps, gs, m, seed0, outliers=0.0, burst_reps=10):
        act = torch.float16 if fmt == "nvfp4_f16" else torch.bfloat16
        a = [synth.activations(m, k, seed=seed0 + i, device=dev, outlier_frac=outliers).to(act)
             for i, (_, n, k) in enumerate(SHAPES)]
        c = [torch.empty((m, n), dtype=act, device=dev) for _, n, _ in SHAPES]

        def fn(i, rep):
            binding.gemm(a[i], rep, SHAPES[i][1], fmt, gs[i], workspace=ws, out=c[i])
        for i in range(len(SHAPES)):
            ws.ensure(binding.workspace_bytes(m, SHAPES[i][1], SHAPES[i][2], fmt))
            fn(i, reps[i][0])
        torch.cuda.synchronize()
        ms = shape_durations([[(lambda i=i, r=r: fn(i, r)) for r in reps[i]] for i in range(len(SHAPES))],
                             stream, burst_reps)
        out = {}
        for i, (name, n, k) in enumerate(SHAPES):
            t = ms[i] * 1e-3
            b = algo_bytes(m, n, k, 32 if fmt == "mxfp4" else 16)
            tf = 2 * m * n * k / t / 1e12
            out[name] = {"us": round(t * 1e6, 2), "gbs": round(b / t / 1e9, 1), "tflops": round(tf, 2),
                         "frac_hbm": round(b / t / 1e9 / peaks["hbm_gbs"], 3),
                         "frac_bf16_peak": round(tf / peaks["bf16_tflops"], 3),
                         "weight_copies": len(reps[i])}
        out["step_us"] = round(float(ms.sum()) * 1e3, 2)
        return out

    prefill = None
    fp16_decode = None
    mxfp4 = None
    m_sweep = None
    cublas = None
    moe = None
    if not args.no_prefill:
        # NVFP4 prefill: m = 256, 0.1 % N(0,20) activation outliers, g = amax/(6*448)
        reps_g, gs_g = prepared("nvfp4", 500, True)
        prefill = shape_table("nvfp4", reps_g, gs_g, M_PREFILL, 300, outliers=0.001)
        del reps_g
        # MXFP4 decode variant at m in {1, 4, 8, 16}
        reps_mx, gs_mx = prepared("mxfp4", 600, False)
        mxfp4 = {f"m={m}": shape_table("mxfp4", reps_mx, gs_mx, m, 700 + m) for m in (1, 4, 8, 16, 256)}
        del reps_mx
        # FP16-activation variant, NVFP4 decode m = 16
        reps_h, gs_h = prepared("nvfp4_f16", 650, False)
        fp16_decode = shape_table("nvfp4_f16", reps_h, gs_h, M_DECODE, 660)
        del reps_h
        # NVFP4 m sweep at n = k = 8192, and m = n = k = 4096 (R weight copies)
        m_sweep = {}
        for (n, k, ms_list) in ((8192, 8192, (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024)), (4096, 4096, (4096,))):
            wsq = synth.weights(n, k, seed=800 + n, device=dev)
            f0 = binding.FP4Weight(wsq, "nvfp4", 1.0)
            del wsq
            rr = rotated([f0.rep], f0.rep.numel())
            for m in ms_list:
                a = synth.activations(m, k, seed=900 + m, device=dev)
                c = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
                ws.ensure(binding.workspace_bytes(m, n, k))

                def fn(rep, a=a, c=c, n=n):
                    binding.gemm(a, rep, n, "nvfp4", 1.0, workspace=ws, out=c)
                fn(rr[0])
                torch.cuda.synchronize()
                t = float(shape_durations([[lambda r=r: fn(r) for r in rr]], stream, 10)[0]) * 1e-3
                b = algo_bytes(m, n, k)
                tf = 2 * m * n * k / t / 1e12
                roof_t = max(b / (peaks["hbm_gbs"] * 1e9), 2 * m * n * k / (peaks["bf16_tflops"] * 1e12))
                m_sweep[f"m={m} n={n} k={k}"] = {
                    "us": round(t * 1e6, 2), "gbs": round(b / t / 1e9, 1), "tflops": round(tf, 1),
                    "bound": "hbm" if b / (peaks["hbm_gbs"] * 1e9) >= 2 * m * n * k / (peaks["bf16_tflops"] * 1e12)
                    else "tensor",
                    "frac_roofline": round(roof_t / t, 3), "weight_copies": len(rr)}
            del f0, rr
        # MoE grouped GEMM: 8 experts, top-2, Mixtral-8x7B-like gate_up
        # (n = 28672, k = 4096), MXFP4, seeded Zipf-like routing
        moe = {}
        E, n_e, k_e = 8, 28672, 4096
        ew = []
        n_sets = rotation_copies(E * n_e * k_e * 17 // 32, l2)
        for c in range(n_sets):
            reps_e = []
            for e in range(E):
                w = synth.weights(n_e, k_e, seed=1000 + 10 * c + e, device=dev)
                reps_e.append(binding.FP4Weight(w, "mxfp4").rep)
                del w
            ew.append(torch.cat(reps_e))
            del reps_e
        torch.cuda.synchronize()   # the concatenated weights are complete before any GEMM reads them
        for tokens in (16, 256):
            off = synth.moe_expert_offsets(tokens, E, 2, seed=tokens)
            a = synth.activations(off[-1], k_e, seed=1100 + tokens, device=dev)
            cm = torch.empty((off[-1], n_e), dtype=torch.bfloat16, device=dev)

            def fn(w, a=a, cm=cm, off=off):
                binding.moe_gemm(a, ew[w], off, n_e, "mxfp4", workspace=ws, out=cm)
            fn(0)
            torch.cuda.synchronize()
            t = float(shape_durations([[lambda w=w: fn(w) for w in range(n_sets)]], stream, 10)[0]) * 1e-3
            active = sum(1 for e in range(E) if off[e + 1] > off[e])
            b = active * n_e * k_e * 17 // 32 + 2 * off[-1] * (k_e + n_e)
            tf = 2 * off[-1] * n_e * k_e / t / 1e12
            moe[f"tokens={tokens} top2 rows={off[-1]}"] = {
                "us": round(t * 1e6, 2), "gbs": round(b / t / 1e9, 1), "tflops": round(tf, 1),
                "frac_hbm": round(b / t / 1e9 / peaks["hbm_gbs"], 3), "active_experts": active,
                "expert_rows": [off[e + 1] - off[e] for e in range(E)], "weight_copies": n_sets}
        del ew
        # context row: cuBLAS BF16 dense GEMM on the same shapes (BF16 weights are
        # 3.6x the NVFP4 bytes; R copies rotate so they come from HBM too)
        cublas = {}
        for i, (name, n, k) in enumerate(SHAPES):
            wb = [synth.weights(n, k, seed=950 + i + 10 * c, device=dev)
                  for c in range(rotation_copies(2 * n * k, l2))]
            row = {}
            for m in (M_DECODE, M_PREFILL):
                a = synth.activations(m, k, seed=960 + m, device=dev)
                fns = [lambda c=c, a=a: torch.matmul(a, wb[c].t()) for c in range(len(wb))]
                fns[0]()
                torch.cuda.synchronize()
                t = float(shape_durations([fns], stream, 10)[0]) * 1e-3
                ours = (per_kernel_ms[i] * 1e-3) if m == M_DECODE else prefill[name]["us"] * 1e-6
                row[f"m={m}"] = {"us": round(t * 1e6, 2), "tflops": round(2 * m * n * k / t / 1e12, 1),
                                 "ours_speedup": round(t / ours, 2), "weight_copies": len(wb)}
            cublas[name] = row
            del wb

    sampler.stop()
    clocks = sampler.summary(windows)
    # every GEMM of this run used `ws`: a bounded device wait that ran out
    # (or, in the bounds-checking build, a failed index check) would show here
    device_status = ws.status()
    if device_status != 0:
        raise RuntimeError(f"device status {binding.STATUS.get(device_status, device_status)} "
                           "after the benchmark: its numbers are not valid")

    cpu_baseline = None
    if rank == 0 and not args.no_cpu_baseline:
        rows = 512
        w_cpu = [synth.weights(n, k, seed=100 + i, device=dev)[:rows].cpu() for i, (_, n, k) in enumerate(SHAPES)]
        a_cpu = [a.cpu() for a in acts]
        nb, dt, passes, cpu_s = oracle_sample(w_cpu, a_cpu, rows, min_seconds=10.0)
        cpu_baseline = {"value": round(nb / dt / 1e9, 4), "unit": "GB/s", "cores": busy_cores(cpu_s, dt),
                        "kind": "oracle",
                        "sample": f"first {rows} rows of each of the 4 weight matrices (same seeded weights), "
                                  f"m={M_DECODE}; NVFP4 dequantise + FP64 GEMM with numpy (BLAS threads), "
                                  f"quantisation untimed; {passes} passes in {dt:.1f} s using {cpu_s:.1f} s "
                                  f"of CPU on a {os.cpu_count()}-core host (cores = CPU / wall time)"}

    if rank == 0:
        out = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights quantised to NVFP4 on the GPU)",
            "config": dict(decode_config(world), tile_override=tile,
                           l2="2 rotating weight sets of 481 MB each (> 3x the L2); per-shape lines "
                              "rotate R = max(2, ceil(3 L2 / weight bytes)) copies"),
            "timing": f"median of {BATCHES} batches of `steps` steps; each batch bracketed by a barrier and "
                      "a device synchronisation, CUDA events on the launching stream",
            "batch_ms": [round(b, 4) for b in batch_ms],
            "tflops": round(world * step_flops * args.steps / (elapsed_max * 1e-3) / 1e12, 2),
            "shapes": shapes, "roofline": roofline, "cpu_baseline": cpu_baseline, "e2e": e2e,
            "gpu_launches": BATCHES * len(SHAPES) * args.steps,
            "gpu_launches_per_batch": len(SHAPES) * args.steps, "clocks": clocks,
            "prefill_m256": prefill, "mxfp4_decode": mxfp4, "fp16_decode_m16": fp16_decode,
            "m_sweep": m_sweep,
            "moe_mxfp4_gate_up": moe, "cublas_bf16_context": cublas,
            "device_status": binding.STATUS.get(device_status, device_status),
        }
        print(json.dumps(out), flush=True)


def run_profile_only(args, local):
    """Quantise + repack the four weights, then launch each GEMM once:
    launch order qkv, o, gate_up, down (gemm_kernel launches 0..3)."""
    from fp4_weight_only_gb300 import binding, synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.load()
    apply_tile(args, binding)
    ws = binding.Workspace(dev)
    if args.profile_moe:
        # the bench's MoE line: 8 experts, top-2 seeded routing, MXFP4 gate_up
        E, n_e, k_e, tokens = 8, 28672, 4096, args.profile_moe
        reps_e = []
        for e in range(E):
            w = synth.weights(n_e, k_e, seed=1000 + e, device=dev)
            reps_e.append(binding.FP4Weight(w, "mxfp4").rep)
            del w
        rep = torch.cat(reps_e)
        torch.cuda.synchronize()   # complete before the GEMM reads it
        off = synth.moe_expert_offsets(tokens, E, 2, seed=tokens)
        a = synth.activations(off[-1], k_e, seed=1100 + tokens, device=dev)
        binding.moe_gemm(a, rep, off, n_e, "mxfp4", workspace=ws)
        torch.cuda.synchronize()
        assert ws.status() == 0
        print(f"profile-only: MoE tokens={tokens} rows={off[-1]} launched 1 grouped GEMM", flush=True)
        return
    m, fmt = args.profile_m, args.profile_fmt
    for i, (name, n, k) in enumerate(SHAPES):
        w = synth.weights(n, k, seed=100 + i, device=dev)
        fw = binding.FP4Weight(w, fmt, 1.0)
        del w
        a = synth.activations(m, k, seed=200 + i, device=dev)
        if fmt == "nvfp4_f16":
            a = a.to(torch.float16)
        fw(a, workspace=ws)
        torch.cuda.synchronize()
        del fw
    assert ws.status() == 0
    print(f"profile-only: {fmt} m={m} launched {len(SHAPES)} GEMMs", flush=True)


def main():
    args = parse()
    if args.profile_only:
        return run_profile_only(args, dist_env()[2])
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1 and args.impl != "reference":
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
