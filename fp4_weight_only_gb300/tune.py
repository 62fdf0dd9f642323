"""Tile tuning for one GEMM shape (Petit PyPI page, "Known limitations": the
tile parameters may need tuning for a given matrix size).

    python -m fp4_weight_only_gb300.tune --m 128 --n 8192 --k 8192 [--fmt nvfp4]
    python -m fp4_weight_only_gb300.tune --m 128 --n 8192 --k 8192 --plan-only --sms 152 --pairs 76

``--plan-only`` prints the planner's plan (no GPU needed with --sms and
--pairs).  Otherwise every tile shape (bn activation rows, ku 128-k chunks
per unit) and CTA-pair mode that applies is timed on the current GPU with
CUDA events, over enough weight copies that every launch reads its weights
from HBM, and printed fastest first beside the planner's own choice.  The
process-wide tile and pair settings are restored afterwards; pass the best
row's values to ``binding.set_tile_config`` / ``set_pair_mode`` (or
``petit_set_tile_config`` / ``petit_set_pair_mode``) to use it.
"""

import argparse
import json
import math

from . import binding

TILES = [(16, 1), (16, 2), (32, 1), (32, 2), (64, 1), (64, 2), (128, 1), (256, 1)]


def candidates(k):
    """(bn, ku) shapes that run as given for this k (ku = 2 needs an even
    number of 128-k chunks)."""
    return [(bn, ku) for bn, ku in TILES if ku == 1 or (k // 128) % 2 == 0]


def describe(p):
    pairs = "pairs" if p["cta_pairs"] else "single"
    return (f"bn={p['bn']} ku={p['ku']} {pairs} ranges={p['num_ranges']} ctas={p['num_ctas']} "
            f"units={p['units']} ({p['units_per_tile']}/tile) ws={p['workspace_bytes']} B")


def time_gemm(a, reps, n, fmt, ws, out, iters):
    """Mean launch time (us) of back-to-back GEMMs cycling through `reps`,
    the middle of three batches."""
    import torch
    stream = torch.cuda.current_stream()
    for j in range(2 * len(reps)):
        binding.gemm(a, reps[j % len(reps)], n, fmt, 1.0, workspace=ws, out=out)
    batches = []
    for _ in range(3):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for j in range(iters):
            binding.gemm(a, reps[j % len(reps)], n, fmt, 1.0, workspace=ws, out=out)
        e1.record(stream)
        torch.cuda.synchronize()
        batches.append(e0.elapsed_time(e1) * 1e3 / iters)
    return sorted(batches)[1]


def tune(m, n, k, fmt="nvfp4", iters=None):
    """Times every applicable (bn, ku, pair mode) for this shape on the
    current GPU; returns the rows (dicts) fastest first and the planner's
    own plan and time."""
    import torch
    from . import synth
    dev = torch.device("cuda", torch.cuda.current_device())
    w = synth.weights(n, k, seed=1, device=dev)
    fw = binding.FP4Weight(w, fmt, 1.0)
    del w
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 2**20)
    copies = max(2, math.ceil(3 * l2 / fw.rep.numel()))
    reps = [fw.rep] + [fw.rep.clone() for _ in range(copies - 1)]
    act = torch.float16 if fmt == "nvfp4_f16" else torch.bfloat16
    a = synth.activations(m, k, seed=2, device=dev).to(act)
    out = torch.empty((m, n), dtype=act, device=dev)
    ws = binding.Workspace(dev)
    iters = iters or max(40, 4 * copies)
    rows = []
    try:
        binding.set_tile_config(0, 0)
        binding.set_pair_mode(0)
        planned = binding.plan(m, n, k, fmt)
        planned_us = time_gemm(a, reps, n, fmt, ws, out, iters)
        for bn, ku in candidates(k):
            modes = (1, 2) if bn >= 128 and n % 256 == 0 else (1,)
            for mode in modes:
                binding.set_tile_config(bn, ku)
                binding.set_pair_mode(mode)
                p = binding.plan(m, n, k, fmt)
                us = time_gemm(a, reps, n, fmt, ws, out, iters)
                rows.append({"bn": bn, "ku": ku, "pair_mode": mode, "cta_pairs": p["cta_pairs"],
                             "num_ranges": p["num_ranges"], "us": round(us, 2),
                             "tflops": round(2 * m * n * k / us / 1e6, 1)})
    finally:
        binding.set_tile_config(0, 0)
        binding.set_pair_mode(0)
    status = ws.status()   # (reading clears it)
    if status != 0:
        raise RuntimeError(f"device status {binding.STATUS.get(status, status)} while tuning")
    rows.sort(key=lambda r: r["us"])
    return rows, planned, planned_us


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--m", type=int, required=True)
    ap.add_argument("--n", type=int, required=True)
    ap.add_argument("--k", type=int, required=True)
    ap.add_argument("--fmt", default="nvfp4", choices=sorted(binding.FORMATS))
    ap.add_argument("--plan-only", action="store_true", help="print the plan, time nothing")
    ap.add_argument("--sms", type=int, help="plan for this SM count (default: the current GPU's)")
    ap.add_argument("--pairs", type=int, help="plan for this CTA-pair capacity (default: the current GPU's)")
    ap.add_argument("--json", action="store_true", help="one JSON object instead of a table")
    args = ap.parse_args(argv)
    if args.plan_only:
        p = binding.plan(args.m, args.n, args.k, args.fmt, args.sms, args.pairs)
        print(json.dumps(p) if args.json else describe(p))
        return 0
    rows, planned, planned_us = tune(args.m, args.n, args.k, args.fmt)
    if args.json:
        print(json.dumps({"planned": planned, "planned_us": round(planned_us, 2), "rows": rows}))
        return 0
    print(f"m={args.m} n={args.n} k={args.k} {args.fmt}")
    print(f"  planner: {describe(planned)}: {planned_us:.2f} us")
    for r in rows:
        print(f"  bn={r['bn']:3d} ku={r['ku']} pair_mode={r['pair_mode']} "
              f"({'pairs' if r['cta_pairs'] else 'single'}, {r['num_ranges']} ranges): "
              f"{r['us']:8.2f} us  {r['tflops']:7.1f} TFLOP/s")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
