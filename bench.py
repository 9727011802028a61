#!/usr/bin/env python3
"""Benchmark of the NVFP4 block-scaled grouped GEMM on GB300.

One step = one grouped call (one persistent GEMM kernel) over the
workload's seeded synthetic inputs, resident in HBM, L2 flushed between timed
calls. Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload prefill]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample
  python bench.py --api device ...        # the device-resident group-table entry point
  python bench.py --op quantize ...       # quantise-and-pack of the workload's activations

N > 1 runs N independent replicas (one process per GPU under torchrun; the
path has no exchange step); value = all ranks' FLOPs / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "µs per grouped call and dense FP4 TFLOPS; % of roofline (1×GB300)"
FP4_OVER_BF16 = 13.5 / 2.25     # nominal dense FP4 : BF16 tensor rate on GB300
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

WORKLOAD_TEXT = {
    "tiny": "G=2: (128,128,256), (64,256,256)",
    "decode": "G=8 decode MoE: m_g~U[40,192], n=4096, k=7168",
    "prefill": "G=8 prefill: m_g=1024, n=4096, k=7168",
    "ragged": "G=4 ragged: m_g=(1,17,333,1000), n=7168, k=2048, B~N(0,0.02)+1% x50",
    "zipf64": "G=64 Zipf(1.2) routing of 16384 tokens (60 active, 4 idle), n=2048, k=7168",
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="prefill", choices=list(WORKLOAD_TEXT))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--tile-n", type=int, default=0, help="GEMM tile N (0 = library default)")
    ap.add_argument("--api", choices=["host", "device"], default="host",
                    help="host: nvfp4_grouped_gemm (group table from the host); device: "
                         "nvfp4_grouped_gemm_device (group table in device memory)")
    ap.add_argument("--problems", type=int, default=1,
                    help="P > 1: P independent copies of the workload (seeds seed..seed+P-1) in one "
                         "nvfp4_grouped_gemm_batched launch per step")
    ap.add_argument("--op", choices=["gemm", "quantize"], default="gemm",
                    help="gemm: the grouped GEMM (default); quantize: nvfp4_quantize_pack of the workload's "
                         "activations (all groups' rows stacked, bf16 [sum m, k])")
    ap.add_argument("--flush-mb", type=int, default=512, help="L2 flush buffer read between timed calls")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=1,
                    help="streams each e2e host<->device copy is split over (copy engines in parallel)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target wall time of the oracle sample")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ helpers

def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK), "fallback"


def roofline_terms(flops, nbytes, peaks):
    """Roofline of one grouped call: time = max(FLOPs at the FP4 peak, bytes at HBM)."""
    fp4_tflops = peaks["bf16_tflops"] * FP4_OVER_BF16
    t_flop = flops / (fp4_tflops * 1e12)
    t_mem = nbytes / (peaks["hbm_gbs"] * 1e9)
    return ("tensor" if t_flop >= t_mem else "hbm"), t_flop, t_mem, fp4_tflops


def kernel_code_digest(path) -> str:
    """sha256[:16] of a CUDA source with // comments and blank lines removed
    (an edit of comments alone does not change the kernel)."""
    import hashlib
    import re
    lines = []
    for line in Path(path).read_text().splitlines():
        line = re.sub(r"//.*$", "", line).rstrip()
        if line.strip():
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def profile_traffic(summary, source, expect=None):
    """DRAM bytes per launch from a committed ncu summary under profiles/, if it
    was taken on the kernel source as it is now and with the settings in
    `expect` (else None)."""
    summ = ROOT / "profiles" / summary
    if not summ.exists():
        return None
    digest = kernel_code_digest(ROOT / "nvfp4_block_scaled_grouped_gb300" / "csrc" / source)
    kv = {}
    for line in summ.read_text().splitlines():
        if ": " in line:
            k, v = line.split(": ", 1)
            kv[k.strip()] = v.strip()
    if kv.get(f"{source} code sha256[:16]", "").split(" ")[0] != digest:
        return None
    if any(kv.get(k) != v for k, v in (expect or {}).items()):
        return None
    try:
        return float(kv["dram bytes per launch"])
    except (KeyError, ValueError):
        return None


def stored_traffic(workload, tile_n):
    """The grouped GEMM kernel's DRAM bytes per launch for a workload."""
    return profile_traffic(f"gemm_kernel_{workload}.txt", "gemm.cu", {"tile_n": str(tile_n)})


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        for line in Path(self.path).read_text().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        smax = [num(r[1]) for r in rows if num(r[1]) is not None]
        pw = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower().startswith("active")})
        # samples under load: power above the run's midpoint between min and max
        if pw:
            mid = (min(pw) + max(pw)) / 2
            loaded = [float(r[0]) for r in rows if num(r[2]) is not None and num(r[2]) >= mid and num(r[0])]
        else:
            loaded = sm
        return {"sm_mhz": statistics.median(loaded or sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x; every rank calls it (one rank: x)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(work_per_rank: float, world: int, t_max_s: float) -> float:
    """Whole-job rate of N independent replicas: all ranks' work over the
    slowest rank's time."""
    return world * work_per_rank / t_max_s


def gpu_uuid(dev_index):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else f"GPU-{u}"
    except Exception:
        return str(dev_index)


# ------------------------------------------------------------------ the oracle legs (CPU)

def host_cores() -> int:
    """Host cores this process may run on (the oracle's thread count when all are used)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(prob, seconds, threads=0):
    """Time the CPU oracle on a column slice of every non-empty group, sized to
    take about `seconds` of wall time (`threads` OpenMP threads, 0 = all).
    Returns (flops, wall_s, threads_used, text, fraction of C's outputs)."""
    import numpy as np
    from oracle import oracle

    threads = threads or host_cores()
    groups = [(g, s) for g, s in enumerate(prob.problem_sizes) if s[0] > 0 and s[1] > 0 and s[2] > 0]
    outputs = sum(m * n for _, (m, n, _, _) in groups)

    def run(cols_per_group):
        flops, done = 0.0, 0
        t0 = time.perf_counter()
        for g, (m, n, k, _) in groups:
            c = min(cols_per_group, n)
            rows = np.repeat(np.arange(m, dtype=np.int32), c)
            cols = np.tile(np.arange(c, dtype=np.int32), m)
            oracle.gemm_sampled(m, n, k, prob.A[g], prob.B[g], prob.SFA[g], prob.SFB[g], rows, cols,
                                threads=threads)
            flops += 2.0 * m * c * k
            done += m * c
        return flops, time.perf_counter() - t0, done

    _, t0, _ = run(2)
    per_col = t0 / 2
    cols = int(max(2, min(max(s[1] for _, s in groups), seconds / max(per_col, 1e-9))))
    flops, wall, done = run(cols)
    frac = done / outputs
    text = (f"all rows x the first {cols} columns of each of the {len(groups)} non-empty groups "
            f"({flops / 2:.3g} multiply-adds, fp64, full k; {100 * frac:.3g}% of C's outputs) "
            f"on {threads} thread{'s' if threads > 1 else ''}")
    return flops, wall, threads, text, frac


def oracle_full(prob, threads):
    """Time the oracle's full C (every output of every group). Returns (flops, wall_s)."""
    from oracle import oracle
    t0 = time.perf_counter()
    oracle.grouped_gemm(prob.problem_sizes, prob.A, prob.B, prob.SFA, prob.SFB, threads=threads)
    return float(prob.flops()), time.perf_counter() - t0


def cpu_baseline_leg(prob, seconds):
    """The oracle as it stands on the host cores: full C when the slice rate
    says it ends within ~3x `seconds`, else a column slice (with the fraction
    of C it covers); plus single-thread figures on the two small task configs
    (the two-group tiny call in full, a slice of the ragged call)."""
    from nvfp4_block_scaled_grouped_gb300 import workloads
    from oracle import oracle

    cores = host_cores()
    f, w, _, text, frac = oracle_sample(prob, min(seconds, 3.0), threads=cores)
    full_est = w / max(frac, 1e-12)
    if full_est <= 3.0 * seconds:
        f, w = oracle_full(prob, cores)
        text, frac = f"full C ({f / 2:.3g} multiply-adds, fp64) on {cores} threads", 1.0
    elif seconds > 3.0:
        f, w, _, text, frac = oracle_sample(prob, seconds, threads=cores)
    single = {}
    tiny = workloads.make_problem("tiny", seed=0)
    tf, tw = oracle_full(tiny, 1)
    single["tiny"] = {"value": tf / tw / 1e12, "unit": "TFLOP/s", "wall_s": tw, "fraction_of_C": 1.0,
                      "sample": "full C of G=2: (128,128,256), (64,256,256), 1 thread"}
    rag = workloads.make_problem("ragged", seed=0)
    rf, rw, _, rtext, rfrac = oracle_sample(rag, 2.0, threads=1)
    single["ragged"] = {"value": rf / rw / 1e12, "unit": "TFLOP/s", "wall_s": rw, "fraction_of_C": rfrac,
                        "sample": rtext}
    return {"value": f / w / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": text,
            "wall_s": w, "fraction_of_C": frac, "full_C": frac == 1.0,
            "full_C_estimate_s": full_est if frac < 1.0 else w, "single_core": single}


def reference_arm(args, rank, world):
    """--impl reference: the CPU oracle, as it stands, on bounded samples."""
    if rank != 0:
        return 0
    from nvfp4_block_scaled_grouped_gb300 import workloads
    prob = workloads.make_problem(args.workload, seed=args.seed)
    per_step = max(0.5, min(3.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(prob, per_step)
    flops_l, wall_l = [], []
    text, cores = "", 0
    for _ in range(args.steps):
        f, w, cores, text, frac = oracle_sample(prob, per_step)
        flops_l.append(f)
        wall_l.append(w)
    value = sum(flops_l) / sum(wall_l) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(wall_l) / len(wall_l),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args, prob),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {text}", "fraction_of_C": frac},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(args, prob):
    extra = f" x {args.problems} independent problems in one launch" if args.problems > 1 else ""
    return {"workload": f"{args.workload}: {WORKLOAD_TEXT[args.workload]}{extra}",
            "group_count": prob.group_count,
            "problem_sizes": [list(s) for s in prob.problem_sizes],
            "sum_m": int(sum(s[0] for s in prob.problem_sizes)),
            "seed": args.seed,
            "l2": f"flushed between timed calls ({args.flush_mb} MB read)"}


# ------------------------------------------------------------------ the GPU arm

def gpu_arm(args, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist

    import nvfp4_block_scaled_grouped_gb300 as nv
    from nvfp4_block_scaled_grouped_gb300 import workloads
    from nvfp4_block_scaled_grouped_gb300.device import DeviceProblem

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    nv.lib()
    if args.tile_n:
        nv.set_tile_n(args.tile_n)
    probs = [workloads.make_problem(args.workload, seed=args.seed + i) for i in range(max(1, args.problems))]
    prob = probs[0]
    flops = sum(p.flops() for p in probs)
    nbytes = sum(p.algorithmic_bytes() for p in probs)

    stream = torch.cuda.current_stream(dev)
    dps = [DeviceProblem.upload(p, device=dev) for p in probs]   # uploads, then packs scales (library kernel)
    # The scale-layout pre-pass alone: the row-major scales of every operand
    # are resident, a spin keeps the GPU busy while the host queues the
    # launch, and events bracket only the one batched pack launch.
    sf_rows = [(torch.from_numpy(np.ascontiguousarray(sf)).to(dev), k)
               for p in probs for (m, n, k, _), sfa, sfb in zip(p.problem_sizes, p.SFA, p.SFB)
               for sf, rows in ((sfa, m), (sfb, n)) if rows > 0 and k > 0]
    nv.pack_scales_tensors(sf_rows)   # warm-up: its outputs' memory is then cached for the timed call
    torch.cuda.synchronize()
    t_pack0 = torch.cuda.Event(enable_timing=True)
    t_pack1 = torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(2_000_000)
    t_pack0.record(stream)
    packed = nv.pack_scales_tensors(sf_rows)
    t_pack1.record(stream)
    torch.cuda.synchronize()
    del sf_rows, packed
    dp = DeviceProblem(problem_sizes=[s for d in dps for s in d.problem_sizes], A=[t for d in dps for t in d.A],
                       B=[t for d in dps for t in d.B], SFA=[t for d in dps for t in d.SFA],
                       SFB=[t for d in dps for t in d.SFB], C=[t for d in dps for t in d.C])
    counts = [len(d.problem_sizes) for d in dps]

    def make_call(q):
        """The timed call on operands q (a DeviceProblem), through the chosen entry point."""
        ptr = lambda t: 0 if t.numel() == 0 else int(t.data_ptr())
        if len(counts) > 1:
            batch, at = [], 0
            for c in counts:
                sl = slice(at, at + c)
                batch.append((q.problem_sizes[sl], [ptr(t) for t in q.A[sl]], [ptr(t) for t in q.B[sl]],
                              [ptr(t) for t in q.SFA[sl]], [ptr(t) for t in q.SFB[sl]], [ptr(t) for t in q.C[sl]]))
                at += c
            return lambda: nv.grouped_gemm_batched(batch, stream)
        if args.api == "device":
            table = nv.DeviceGroupTable(len(q.problem_sizes), device=dev)
            table.set(q.problem_sizes, q.A, q.B, q.SFA, q.SFB, q.C)
            torch.cuda.synchronize()
            return lambda: table.run(stream)
        return lambda: q.run(stream)

    call = make_call(dp)

    # L2 flush: read a buffer 4x the 129 MB L2 (reads leave no dirty lines to write back)
    flush = torch.ones(args.flush_mb << 18, dtype=torch.int32, device=dev)
    # warm-up: the timed step sequence itself (flush, events, call), so that
    # every kernel and event the timed loop uses has been loaded and run once
    for _ in range(max(3, args.warmup)):
        flush.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda._sleep(1000)
    torch.cuda.synchronize()
    assert nv.device_status(stream) == 0, "a bounded wait gave up during warm-up"

    def barrier():
        if world > 1:
            dist.barrier()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(gpu_uuid(local_rank)) as clocks:
        barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        # keep the GPU busy while the host enqueues the steps, so no step's
        # events include time the GPU spent waiting for the host
        torch.cuda._sleep(2_000_000)
        for i in range(args.steps):
            flush.sum()                      # evict A/B/scales from L2 (outside the timed events)
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier()
        wall = time.perf_counter() - wall0
    times_ms = [a.elapsed_time(b) for a, b in ev]
    assert nv.device_status(stream) == 0, "a bounded wait gave up during the timed run"
    t_ms = statistics.fmean(times_ms)
    t_max = max_over_ranks(t_ms, world, dev)
    value = replica_throughput(flops, world, t_max * 1e-3) / 1e12

    # ---- e2e: host buffers in pinned memory, copies inside the timed region.
    # The inputs of a step live in one pinned host blob and the outputs come
    # back into another: one H2D and one D2H copy per step, the call on
    # device views of the blobs.
    e2e = None
    if not args.no_e2e:
        def blob(tensors):
            offs, pos = [], 0
            for t in tensors:
                offs.append(pos)
                pos += -(-t.numel() * t.element_size() // 256) * 256
            return offs, max(pos, 256)
        ins = [dp.A, dp.B, dp.SFA, dp.SFB]
        flat_in = [t for lst in ins for t in lst]
        in_offs, in_bytes = blob(flat_in)
        out_offs, out_bytes = blob(dp.C)
        d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        h_in = torch.empty(in_bytes, dtype=torch.uint8, pin_memory=True)
        d_out = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
        h_out = torch.empty(out_bytes, dtype=torch.uint8, pin_memory=True)

        def view(base, off, t):
            n = t.numel() * t.element_size()
            return base[off:off + n].view(t.dtype).view(t.shape)
        views = [view(d_in, o, t) for o, t in zip(in_offs, flat_in)]
        for v, t in zip(views, flat_in):
            v.copy_(t)
        h_in.copy_(d_in)
        it = iter(views)
        q = DeviceProblem(problem_sizes=dp.problem_sizes, A=[next(it) for _ in dp.A], B=[next(it) for _ in dp.B],
                          SFA=[next(it) for _ in dp.SFA], SFB=[next(it) for _ in dp.SFB],
                          C=[view(d_out, o, c) for o, c in zip(out_offs, dp.C)])
        call_e2e = make_call(q)
        h2d, d2h = in_bytes, out_bytes
        e2e_steps = max(3, min(args.steps, 10))
        side = [torch.cuda.Stream(dev) for _ in range(max(1, args.e2e_streams) - 1)]

        def copy(dst, src):
            # dst.copy_(src) in 256-byte-aligned contiguous pieces, one per
            # stream (the launching stream's own included), joined back on it
            n = len(side) + 1
            per = -(-dst.numel() // n)
            piece = -(-per // 256) * 256
            start = torch.cuda.Event()
            start.record(stream)
            joins = []
            for i, st in enumerate(side, 1):
                lo, hi = i * piece, min((i + 1) * piece, dst.numel())
                if lo >= hi:
                    break
                st.wait_event(start)
                with torch.cuda.stream(st):
                    dst[lo:hi].copy_(src[lo:hi], non_blocking=True)
                e = torch.cuda.Event()
                e.record(st)
                joins.append(e)
            dst[:piece].copy_(src[:piece], non_blocking=True)
            for e in joins:
                stream.wait_event(e)

        for _ in range(2):
            copy(d_in, h_in)
            call_e2e()
            copy(h_out, d_out)
        torch.cuda.synchronize()
        e_ms = []
        for _ in range(e2e_steps):
            flush.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            copy(d_in, h_in)
            call_e2e()
            copy(h_out, d_out)
            b.record(stream)
            b.synchronize()
            e_ms.append(a.elapsed_time(b))
        em = max_over_ranks(statistics.fmean(e_ms), world, dev)
        e2e = {"value": replica_throughput(flops, world, em * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": em, "steps": e2e_steps, "copy_streams": len(side) + 1}

    if rank != 0:
        return 0

    peaks, peak_src = measured_peaks()
    bound, t_flop, t_mem, fp4_peak = roofline_terms(flops, nbytes, peaks)
    t_s = t_ms * 1e-3
    tile_n = args.tile_n or 256
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": nbytes / t_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / t_s / 1e12, "peak": fp4_peak, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = stored_traffic(args.workload, tile_n)
    roof["peak_source"] = (f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback") + \
        ("" if bound == "hbm" else " bf16 burst x 6 (nominal FP4:BF16)")
    roof["kernel"] = "grouped_gemm_kernel (the only kernel of a grouped call; events around the call)"
    roof["roofline_us"] = max(t_flop, t_mem) * 1e6
    roof["frac_of_roofline_time"] = max(t_flop, t_mem) / t_s

    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline_leg(prob, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max, "us_per_call": t_max * 1e3,
        "us_per_call_p10_p50_p90": [float(v * 1e3) for v in _pcts(times_ms)],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 x e2m1, e4m3 per-16 scales) -> f32 acc -> f16",
        "data": "synthetic (seeded N(0,1) -> NVFP4 per-16 quantisation)",
        "config": dict(workload_config(args, prob), tile_n=tile_n, api=args.api, parallelism=f"replicas x{world}"),
        "flops_per_call": flops, "bytes_per_call": nbytes,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "scale_pack_us": 1e3 * t_pack0.elapsed_time(t_pack1),
        "clocks": clocks.summary(),
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ quantise-and-pack

def quantize_arm(args, rank, world, local_rank):
    """nvfp4_quantize_pack of the workload's stacked activations (bf16
    [sum m, k], seeded N(0, 1)); HBM-bound: bytes = 2 rows k in + rows k / 2
    codes + rows k / 16 scales."""
    import numpy as np
    import torch
    import torch.distributed as dist

    import nvfp4_block_scaled_grouped_gb300 as nv
    from nvfp4_block_scaled_grouped_gb300 import workloads

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    sizes = workloads.problem_sizes(args.workload, args.seed)
    rows, k = int(sum(s[0] for s in sizes)), int(max(s[2] for s in sizes))
    gen = torch.Generator().manual_seed(args.seed)
    x = torch.randn(rows, k, generator=gen).to(torch.bfloat16).to(dev)
    codes = torch.empty((rows, k // 2), dtype=torch.uint8, device=dev)
    sf = torch.empty(nv.scale_bytes(rows, k), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    call = lambda: nv.quantize_pack(x.data_ptr(), nv.DTYPE_BF16, rows, k, codes.data_ptr(), sf.data_ptr(), stream)
    nbytes = 2 * rows * k + rows * k // 2 + rows * k // 16
    flush = torch.ones(args.flush_mb << 18, dtype=torch.int32, device=dev)
    for _ in range(max(3, args.warmup)):
        flush.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda._sleep(1000)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(gpu_uuid(local_rank)) as clocks:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        torch.cuda._sleep(2_000_000)
        for i in range(args.steps):
            flush.sum()
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    times_ms = [a.elapsed_time(b) for a, b in ev]
    t_ms = max_over_ranks(statistics.fmean(times_ms), world, dev)
    # e2e: bf16 input from pinned host memory, codes and scales back
    hx = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    hx.copy_(x)
    hc = torch.empty(codes.shape, dtype=codes.dtype, pin_memory=True)
    hs = torch.empty(sf.shape, dtype=sf.dtype, pin_memory=True)
    e_ms = []
    for i in range(max(3, min(args.steps, 10)) + 1):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.sum()
        a.record(stream)
        x.copy_(hx, non_blocking=True)
        call()
        hc.copy_(codes, non_blocking=True)
        hs.copy_(sf, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i:
            e_ms.append(a.elapsed_time(b))
    em = max_over_ranks(statistics.fmean(e_ms), world, dev)   # every rank takes part
    if rank != 0:
        return 0
    peaks, peak_src = measured_peaks()
    t_s = t_ms * 1e-3
    roof = {"bound": "hbm", "achieved": nbytes / t_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = profile_traffic(f"quantize_pack_kernel_{args.workload}.txt", "quantize.cu",
                                      {"rows": str(rows), "k": str(k)})
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"
    roof["kernel"] = "quantize_pack_kernel (the only kernel of the call)"
    cpu = None
    if not args.no_cpu_baseline:
        from oracle import oracle
        xs = x[: max(1, min(rows, 64))].float().cpu().numpy()
        w0 = time.perf_counter()
        oracle.quantize(xs)
        w = time.perf_counter() - w0
        cpu = {"value": xs.size * 2 / w / 1e9, "unit": "GB/s of bf16 input", "cores": 1, "kind": "oracle",
               "sample": f"{xs.shape[0]} of {rows} rows", "wall_s": w}
    line = {
        "metric": "µs per quantise-and-pack call (bf16 activations -> NVFP4 codes + atom-layout scales)",
        "value": replica_throughput(nbytes, world, t_s) / 1e9, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_ms, "us_per_call": t_ms * 1e3,
        "us_per_call_p10_p50_p90": [float(v * 1e3) for v in _pcts(times_ms)],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 -> e2m1 + e4m3",
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": f"activations of {args.workload}: bf16 [{rows}, {k}]", "rows": rows, "k": k,
                   "l2": f"flushed between timed calls ({args.flush_mb} MB read)", "parallelism": f"replicas x{world}"},
        "bytes_per_call": nbytes, "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": replica_throughput(nbytes, world, em * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": em,
                "h2d_bytes_per_step": hx.numel() * 2, "d2h_bytes_per_step": hc.numel() + hs.numel()},
        "gpu_launches": args.steps, "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def _pcts(v):
    s = sorted(v)
    pick = lambda q: s[min(len(s) - 1, int(q * (len(s) - 1) + 0.5))]
    return pick(0.1), pick(0.5), pick(0.9)


def main(argv=None):
    args = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return reference_arm(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local_rank))
    try:
        if args.op == "quantize":
            return quantize_arm(args, rank, world, local_rank)
        return gpu_arm(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
