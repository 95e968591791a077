"""Benchmark of the tiled attention forward path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  * prefill: causal attention B=2, Hq=32, Hkv=8, N=8192, d=128 (the shape the headline
    TFLOP/s is quoted on), through attn_fwd (tile scheduler, TMA producer, tcgen05 MMA,
    softmax, epilogue);
  * decode: paged-KV decode, 32 sequences with contexts U[1024,16384], Hq=32, Hkv=8, d=128,
    pages of 64 at a permuted pool, through attn_fwd (split-KV + fused combine).
`value` is the prefill TFLOP/s (4*B*Hq*sum(visible pairs)*d / prefill time); the decode GB/s
(valid-token K+V bytes / decode time) is reported beside it. Inputs (335 MB prefill, 1.3 GB
decode) are larger than L2, so no flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
       python bench.py --suite [--steps K]   (every workload, one JSON line each)
For N > 1 it runs under torch.distributed.run, one rank per GPU, each rank an independent
replica of the step (the path has no exchange step); value sums all ranks' work over the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s & % BF16 peak (causal N=8192 d=128); decode GB/s % HBM"
PREFILL_NAME = "causal B2 Hq32 Hkv8 N8192 d128"
DECODE_NAME = "paged decode B32 L U[1024,16384] Hq32 Hkv8 d128 page64 (seeded permuted pool)"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def code_tokens(src: str) -> str:
    """C/C++/CUDA source with its comments removed and every run of whitespace made one space,
    so that editing a comment or re-wrapping lines leaves the hash of a kernel unchanged.
    String and character literals are kept as they are."""
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
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(names):
    """Hash of the code (not the comments) of the named files under csrc/."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "tiled_attention_gb300", "csrc", n), encoding="utf-8") as f:
            h.update(code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, sources):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this exact
    kernel code (comments aside); else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash(sources):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / power / throttle sampling while a timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def rows(self):
        """(sm MHz, max sm MHz, power W, [reason flags], utilization %) per sample."""
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                util = float(parts[9]) if parts[9] not in ("", "[N/A]") else 0.0
                power = float(parts[3]) if parts[3] not in ("", "[N/A]") else float("nan")
                rows.append((float(parts[1]), float(parts[2]), power, parts[5:9], util))
            except ValueError:
                continue
        return rows

    def summary(self):
        rows = self.rows()
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, _, r, _ in rows for i, v in enumerate(r)
                          if v.lower() == "active"})
        # Samples taken while the GPU was busy; the region may be shorter than one period,
        # in which case every sample is kept and the clock is the idle one.
        loaded = [r for r in rows if r[4] >= 50.0]
        use = loaded or rows
        out = {"sm_mhz": float(np.median([r[0] for r in use])), "sm_max_mhz": rows[0][1],
               "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded),
               "period_ms": self.period_ms}
        pw = [r[2] for r in use if np.isfinite(r[2])]
        if pw:
            out["power_w_median"] = float(np.median(pw))
            out["power_w_max"] = float(np.max(pw))
        return out


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of per-rank timings (the slowest rank sets the job time)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def replica_throughput(world: int, steps: int, units_per_step: float, seconds: float) -> float:
    """Whole-job throughput of `world` independent replicas: every rank processed
    units_per_step per step; the job took the slowest rank's time."""
    return world * steps * units_per_step / seconds


def cpu_baseline_sample(w, budget_s: float, seed: int, threads: int = 0):
    """Time the oracle on a random row sample sized for about budget_s seconds of work.
    Returns (rows_done, flops_done, seconds)."""
    import oracle
    rng = np.random.default_rng(seed)
    nrows = int(np.prod(w.lse_shape))

    def row_flops(rows):
        i = rows % w.N
        vis = (i + 1) if w.mask_kind == 1 else np.full_like(i, w.N)
        return 4.0 * w.d * float(vis.sum())

    probe = rng.choice(nrows, size=min(nrows, 64), replace=False)
    t0 = time.perf_counter()
    oracle.attention(w, rows=probe, threads=threads)
    dt = max(time.perf_counter() - t0, 1e-4)
    n = int(min(nrows, max(64, len(probe) * budget_s / dt)))
    rows = rng.choice(nrows, size=n, replace=False)
    t0 = time.perf_counter()
    oracle.attention(w, rows=rows, threads=threads)
    dt = time.perf_counter() - t0
    return n, row_flops(rows), dt


def step_config(world: int):
    """The workload description both arms report (the step: prefill, then paged decode)."""
    return {"workload": f"prefill {PREFILL_NAME} + {DECODE_NAME}",
            "prefill": PREFILL_NAME, "decode": DECODE_NAME,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (335 MB prefill, 1.3 GB decode), no flush"}


def reference_arm(args, rank: int):
    """The oracle (plain fp64 CPU) timed on the host cores: each step a bounded row sample."""
    if rank != 0:
        return
    import oracle
    from tiled_attention_gb300 import inputs as I
    w = I.config("3c")
    threads = oracle.max_threads()
    per_step_s = max(0.005, 90.0 / max(1, args.steps + args.warmup))
    rng = np.random.default_rng(77)
    nrows = int(np.prod(w.lse_shape))
    probe = rng.choice(nrows, size=32, replace=False)
    t0 = time.perf_counter()
    oracle.attention(w, rows=probe)
    dt = max(time.perf_counter() - t0, 1e-4)
    rows_per_step = int(max(8, 32 * per_step_s / dt))
    flops_total = 0.0
    t_total = 0.0
    for step in range(args.warmup + args.steps):
        rows = rng.choice(nrows, size=rows_per_step, replace=False)
        t0 = time.perf_counter()
        oracle.attention(w, rows=rows)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            t_total += dt
            i = rows % w.N
            flops_total += 4.0 * w.d * float((i + 1).sum())
    value = flops_total / t_total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(args.gpus),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows_per_step} random query rows of {PREFILL_NAME} per "
                                   "step, fp64, materialised scores"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure_ex2_rate(attn, torch, dev, stream, iters=4096):
    """Exp2 throughput ceiling of this GPU (exponentials per second): the library's MUFU probe
    with eight resident 256-thread CTAs per SM, best of five timed launches after two."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks = sms * 8
    out = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    for _ in range(2):
        assert attn.attn_bench_ex2(out, blocks, iters, stream) == 0, attn.last_error()
    best = 0.0
    for _ in range(5):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        assert attn.attn_bench_ex2(out, blocks, iters, stream) == 0, attn.last_error()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        best = max(best, blocks * 256 * 8 * iters / (e0.elapsed_time(e1) * 1e-3))
    assert bool(torch.isfinite(out).all())
    return best


def suite(args):
    """Time every specified workload and the mask variants one launch at a time (median of
    --steps launches after --warmup, L2 flushed before each launch by writing a 256 MB
    buffer), plus the two-stage paged decode (page gather, then decode on the dense copy)
    next to the fused paged decode. Prints one JSON line per workload."""
    import torch
    from tiled_attention_gb300 import attn, build
    from tiled_attention_gb300 import inputs as I
    from tiled_attention_gb300.runner import DeviceProblem
    build.build()
    attn.lib()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    peaks = load_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    tag = "of " + peaks["source"]
    ex2_ceiling = measure_ex2_rate(attn, torch, dev, stream)
    wanted = None if not args.workloads else set(args.workloads.split(","))

    def timed(fn, reps):
        times = []
        for k in range(args.warmup + reps):
            flush.fill_(k & 0xFF)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            rc = fn()
            e1.record(stream)
            assert rc == 0, attn.last_error()
            if k >= args.warmup:
                times.append((e0, e1))
        torch.cuda.synchronize(dev)
        assert attn.attn_get_status(stream) == 0
        return float(np.median([a.elapsed_time(b) for a, b in times]))

    def dec_bytes(w):
        return (w.kv_bytes_valid() + w.q.nbytes * 2 + w.B * w.Hq * 4 +
                (w.block_table.nbytes if w.block_table is not None else 0) +
                w.cu_seqlens.nbytes)

    def emit(w, ms, extra=None):
        line = {"suite": True, "workload": w.name, "mask_kind": w.mask_kind, "d": w.d,
                "ms": ms, "launches_timed": args.steps}
        if w.mask_kind in I.DECODE_KINDS:
            gbs = dec_bytes(w) / (ms * 1e-3) / 1e9
            line.update(value=gbs, unit="GB/s", frac=gbs / peaks["hbm_gbs"],
                        peak=f"HBM copy {tag}")
        else:
            tf = w.flops() / (ms * 1e-3) / 1e12
            exps = w.flops() / (4 * w.d) / (ms * 1e-3)  # one exponential per visible pair
            line.update(value=tf, unit="TFLOP/s", frac=tf / peaks["bf16_tflops"],
                        peak=f"bf16 burst {tag}", flops=w.flops(), exp2_per_s=exps,
                        exp2_frac_of_ceiling=exps / ex2_ceiling)
        if extra:
            line.update(extra)
        print(json.dumps(line), flush=True)

    for cfg in (1, 2, 3, "3c", "3c64", 4, "3b", "3p", "4b", "6", "6p64", 5, "5p16", "5b1", "5b4"):
        if wanted is not None and str(cfg) not in wanted:
            continue
        w = I.config(cfg)
        dp = DeviceProblem(w, device=dev, fill_outputs=0.0)
        emit(w, timed(lambda: dp.run(stream), args.steps))
        if cfg in ("5b1", "5b4"):
            # The allocation-free entry point on the same inputs: its tickets live in a zeroed
            # region of the library's scratch, so it issues no memset before the kernel.
            o_na, lse_na = torch.empty_like(dp.o), torch.empty_like(dp.lse)

            def noalloc():
                return attn.attn_paged_decode_noalloc(dp.q, dp.k, dp.v, o_na, lse_na, w.B, w.Hq,
                                                      w.Hkv, w.N, w.d, w.scale, dp.cu, dp.table,
                                                      w.page_size, dp.num_pages, stream)

            ms_na = timed(noalloc, args.steps)
            same = (torch.equal(o_na.view(torch.int16), dp.o.view(torch.int16)) and
                    torch.equal(lse_na, dp.lse))
            emit(w, ms_na, {"workload": w.name + " (allocation-free entry point)",
                            "bit_identical_to_attn_fwd": bool(same)})
        if cfg == 5:
            # Two-stage path of the paged-KV pattern: gather K and V pages into dense caches,
            # then the decode kernel reads the caches.
            max_pages = w.block_table.shape[1]
            L = max_pages * w.page_size
            kd = torch.empty((w.B, w.Hkv, L, w.d), dtype=torch.bfloat16, device=dev)
            vd = torch.empty_like(kd)
            o = torch.empty_like(dp.o)
            lse = torch.empty_like(dp.lse)
            nb = attn.attn_workspace_bytes(w.B, w.Hq, w.Hkv, L, w.d, attn.ATTN_MASK_DECODE, 0)
            ws = torch.empty(nb, dtype=torch.uint8, device=dev)
            pages = int(((np.diff(w.cu_seqlens) + w.page_size - 1) // w.page_size).sum())
            page_bytes = w.Hkv * w.page_size * w.d * 2

            def gather():
                rc = attn.attn_gather_pages(dp.k, kd, dp.table, w.B, max_pages, w.Hkv,
                                            w.page_size, w.d, dp.num_pages, stream)
                return rc | attn.attn_gather_pages(dp.v, vd, dp.table, w.B, max_pages, w.Hkv,
                                                   w.page_size, w.d, dp.num_pages, stream)

            def dense():
                return attn.attn_fwd(dp.q, kd, vd, o, lse, w.B, w.Hq, w.Hkv, L, w.d, w.scale,
                                     attn.ATTN_MASK_DECODE, 0, dp.cu, None, 0, 0, ws, stream)

            g_ms = timed(gather, args.steps)
            d_ms = timed(dense, args.steps)
            both_ms = timed(lambda: gather() | dense(), args.steps)
            g_bytes = 2 * 2 * pages * page_bytes  # K and V pages, read once and written once
            print(json.dumps({
                "suite": True, "workload": "two-stage paged decode (gather + dense decode) "
                "on " + w.name, "ms": both_ms, "launches_timed": args.steps,
                "gather_ms": g_ms, "gather_gbs": g_bytes / (g_ms * 1e-3) / 1e9,
                "gather_bytes": g_bytes, "dense_decode_ms": d_ms,
                "dense_decode_gbs": dec_bytes(w) / (d_ms * 1e-3) / 1e9,
                "bytes_moved": g_bytes + dec_bytes(w), "fused_bytes": dec_bytes(w),
                "unit": "GB/s (valid K+V per decode)",
                "value": dec_bytes(w) / (both_ms * 1e-3) / 1e9}), flush=True)
            del kd, vd, ws
        if cfg == "3c":
            # FP8 path on the same shape: Q and K block-quantized to E4M3 by the library (timed
            # on its own), then attention with S = Q K^T on the FP8 tensor cores. Half the
            # FLOPs (Q K^T) run at the FP8 rate, twice the bf16 one, so the peak for the whole
            # is 4/3 of the bf16 peak.
            B, Hq, Hkv, N, d = w.B, w.Hq, w.Hkv, w.N, w.d
            q8 = torch.empty((B, Hq, N, d), dtype=torch.uint8, device=dev)
            k8 = torch.empty((B, Hkv, N, d), dtype=torch.uint8, device=dev)
            qs = torch.empty((B * Hq, (N + 127) // 128), dtype=torch.float32, device=dev)
            ks = torch.empty((B * Hkv, (N + 127) // 128), dtype=torch.float32, device=dev)

            def quant():
                rc = attn.attn_quantize_fp8(dp.q, q8, qs, B * Hq, N, d, stream)
                return rc | attn.attn_quantize_fp8(dp.k, k8, ks, B * Hkv, N, d, stream)

            def fwd8():
                return attn.attn_fwd_fp8(q8, k8, dp.v, dp.o, dp.lse, qs, ks, B, Hq, Hkv, N, d,
                                         w.scale, w.mask_kind, w.window, stream)

            q_ms = timed(quant, args.steps)
            f_ms = timed(fwd8, args.steps)
            tf = w.flops() / (f_ms * 1e-3) / 1e12
            qbytes = (dp.q.numel() + dp.k.numel()) * 3 + (qs.numel() + ks.numel()) * 4
            print(json.dumps({
                "suite": True, "workload": "FP8 Q/K (E4M3, 128-row tile scales) " + w.name,
                "mask_kind": w.mask_kind, "d": d, "ms": f_ms, "launches_timed": args.steps,
                "value": tf, "unit": "TFLOP/s",
                "frac": tf / (peaks["bf16_tflops"] * 4 / 3),
                "peak": f"4/3 x bf16 burst {tag} (Q K^T at the FP8 rate, P V at bf16)",
                "frac_of_bf16_peak": tf / peaks["bf16_tflops"], "flops": w.flops(),
                "quantize_ms": q_ms,
                "quantize_gbs": qbytes / (q_ms * 1e-3) / 1e9}), flush=True)
            del q8, k8, qs, ks
        del dp
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="own", choices=["own", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--sustain-s", type=float, default=3.0,
                    help="seconds of back-to-back steps after the timed region, with the clocks "
                         "sampled under load (0 to skip)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the CPU baseline (rank 0, N=1 only)")
    ap.add_argument("--only", choices=["prefill", "decode"], default=None,
                    help="time one part of the step only (for profiler captures)")
    ap.add_argument("--suite", action="store_true",
                    help="time every workload one launch at a time (one JSON line each)")
    ap.add_argument("--workloads", default=None,
                    help="with --suite: comma-separated workload keys to time (e.g. 4,4b)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.suite:
        suite(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        reference_arm(args, rank)
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from tiled_attention_gb300 import attn, build
    from tiled_attention_gb300 import inputs as I
    from tiled_attention_gb300.runner import DeviceProblem
    build.build()
    attn.lib()

    do_p = args.only in (None, "prefill")
    do_d = args.only in (None, "decode")
    wp = I.config("3c")
    wd = I.config(5) if do_d else I.paged_decode_workload(5, 1, 64, 64, 32, 8, 128)
    pp = DeviceProblem(wp, device=dev, fill_outputs=0.0)
    pd = DeviceProblem(wd, device=dev, fill_outputs=0.0)
    stream = torch.cuda.current_stream(dev)
    launches_per_step = int(do_p) + int(do_d)

    def step(evs=None):
        rc = 0
        if evs:
            evs[0].record(stream)
        if do_p:
            rc |= pp.run(stream)
        if evs:
            evs[1].record(stream)
        if do_d:
            rc |= pd.run(stream)
        if evs:
            evs[2].record(stream)
        return rc

    for _ in range(args.warmup):
        assert step() == 0, attn.last_error()
    torch.cuda.synchronize(dev)
    assert attn.attn_get_status(stream) == 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index, period_ms=20) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for k in range(args.steps):
            step(evs[k])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    status = attn.attn_get_status(stream)
    assert status == 0, f"device status {status}"
    total_ms = t_start.elapsed_time(t_end)
    pre_ms = np.array([e[0].elapsed_time(e[1]) for e in evs])
    dec_ms = np.array([e[1].elapsed_time(e[2]) for e in evs])

    total_ms, pre_sum, dec_sum = max_over_ranks([total_ms, pre_ms.sum(), dec_ms.sum()], dist, dev)

    flops = wp.flops()
    kv_bytes = wd.kv_bytes_valid()
    # decode traffic that is not K/V: q, o (bf16), lse (fp32), table and lengths
    dec_bytes = kv_bytes + wd.q.nbytes * 2 + wd.B * wd.Hq * 4 + wd.block_table.nbytes + \
        wd.cu_seqlens.nbytes
    pre_sum = max(pre_sum, 1e-9)
    dec_sum = max(dec_sum, 1e-9)
    prefill_tflops = replica_throughput(world, args.steps, flops, pre_sum * 1e-3) / 1e12
    decode_gbs = replica_throughput(world, args.steps, dec_bytes, dec_sum * 1e-3) / 1e9
    peaks = load_peaks()
    pre_avg_s = pre_sum / args.steps * 1e-3
    dec_avg_s = dec_sum / args.steps * 1e-3
    tag = "of " + peaks["source"]
    roofline = {
        "bound": "tensor", "kernel": "prefill_kernel<128, causal>",
        "achieved": flops / pre_avg_s / 1e12, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
        "frac": flops / pre_avg_s / 1e12 / peaks["bf16_tflops"],
        "frac_of_sustained": flops / pre_avg_s / 1e12 / peaks["bf16_tflops_sustained"],
        "peak_source": f"bf16 burst {tag}",
        "traffic": recorded_traffic("prefill_causal_d128",
                                    ["prefill.cuh", "ptx.cuh", "sched.h", "tmem_io.inc"]),
        "algorithmic": f"4*B*Hq*sum(visible pairs)*d = {flops:.4e} FLOP per launch",
    }
    roofline_decode = {
        "bound": "hbm", "kernel": "decode_kernel<128, 4>",
        "achieved": dec_bytes / dec_avg_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
        "frac": dec_bytes / dec_avg_s / 1e9 / peaks["hbm_gbs"], "peak_source": f"HBM copy {tag}",
        "traffic": recorded_traffic("decode_d128_g4", ["decode.cuh", "ptx.cuh"]),
        "algorithmic": f"valid-token K+V + q/o/lse/table bytes = {dec_bytes:.4e} B per launch",
    }

    # ---- softmax exponentials against the measured exp2 ceiling
    softmax_exp = None
    if do_p:
        ceiling = measure_ex2_rate(attn, torch, dev, stream)
        n_exp = flops / (4 * wp.d)  # one exponential per visible (query, key) pair
        softmax_exp = {
            "achieved": n_exp / pre_avg_s, "ceiling": ceiling, "unit": "exp2/s",
            "frac": n_exp / pre_avg_s / ceiling,
            "algorithmic": f"B*Hq*sum(visible pairs) = {n_exp:.4e} exponentials per launch",
            "ceiling_source": "attn_bench_ex2 on this GPU (ex2.approx, 8 CTAs x 256 threads "
                              "per SM, 8 independent chains per thread), CUDA events"}

    # ---- end to end: host (pinned) buffers, copies inside the timed region
    e2e = None
    if args.e2e_steps > 0 and args.only is None:
        host = {}
        for name, dp in (("p", pp), ("d", pd)):
            for t_name in ("q", "k", "v", "o", "lse", "cu", "table"):
                tdev = getattr(dp, t_name)
                if tdev is not None:
                    host[name + t_name] = torch.empty(tdev.shape, dtype=tdev.dtype,
                                                      pin_memory=True)
                    host[name + t_name].copy_(tdev)
        h2d = d2h = 0
        for name, dp in (("p", pp), ("d", pd)):
            for t_name in ("q", "k", "v", "cu", "table"):
                if getattr(dp, t_name) is not None:
                    h2d += host[name + t_name].numel() * host[name + t_name].element_size()
            for t_name in ("o", "lse"):
                d2h += host[name + t_name].numel() * host[name + t_name].element_size()

        # Each part runs as a pipeline over three streams (host -> device copies, compute,
        # device -> host copies) with two device buffer sets, the way a serving loop feeds the
        # library: step k+1's inputs upload while step k computes and step k-1's results
        # download. Every step still copies its own inputs from pinned host memory and its O
        # and LSE back; the time is taken with CUDA events from the first upload to the last
        # download.
        def e2e_part(name, dp_a, in_names, steps):
            dps = [dp_a, DeviceProblem(dp_a.w, device=dev, fill_outputs=0.0)]
            s_in, s_cp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
            n = steps + 2
            ev_in = [torch.cuda.Event() for _ in range(n)]
            ev_cp = [torch.cuda.Event() for _ in range(n)]
            ev_out = [torch.cuda.Event() for _ in range(n)]
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            rc = 0
            for k in range(n):
                if k == 2:  # two untimed warm-up steps
                    s_in.wait_event(ev_out[1])
                    t0.record(s_in)
                dp = dps[k % 2]
                if k >= 2:
                    s_in.wait_event(ev_cp[k - 2])  # this set's previous step has read its inputs
                with torch.cuda.stream(s_in):
                    for t_name in in_names:
                        getattr(dp, t_name).copy_(host[name + t_name], non_blocking=True)
                ev_in[k].record(s_in)
                s_cp.wait_event(ev_in[k])
                if k >= 2:
                    s_cp.wait_event(ev_out[k - 2])  # and its previous results are downloaded
                rc |= dp.run(s_cp)
                ev_cp[k].record(s_cp)
                s_out.wait_event(ev_cp[k])
                with torch.cuda.stream(s_out):
                    host[name + "o"].copy_(dp.o, non_blocking=True)
                    host[name + "lse"].copy_(dp.lse, non_blocking=True)
                ev_out[k].record(s_out)
            t1.record(s_out)
            torch.cuda.synchronize(dev)
            assert rc == 0, attn.last_error()
            del dps[1]
            return t0.elapsed_time(t1)

        ep = e2e_part("p", pp, ("q", "k", "v"), args.e2e_steps)
        ed = e2e_part("d", pd, ("q", "k", "v", "cu", "table"), args.e2e_steps)
        assert attn.attn_get_status(stream) == 0
        ep, ed = max_over_ranks([ep, ed], dist, dev)
        e2e = {"value": replica_throughput(world, args.e2e_steps, flops, ep * 1e-3) / 1e12,
               "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": args.e2e_steps,
               "decode_gbs": replica_throughput(world, args.e2e_steps, dec_bytes, ed * 1e-3) / 1e9,
               "what": "per part of the step, pinned host -> device copies of its inputs, "
                       "attn_fwd, device -> pinned host copies of O and LSE, pipelined over "
                       "three streams with two device buffer sets; CUDA events from the first "
                       "upload to the last download"}

    # ---- sustained: the same step back to back for a few seconds, outside the timed steps,
    # with the clocks sampled under load (a long-running job settles at a lower SM clock
    # under the power cap than the short timed region above)
    sustained = None
    if args.sustain_s > 0 and args.only is None:
        chunk = 64
        t_wall = 0.0
        pre_s = dec_s = 0.0
        n_steps = 0
        torch.cuda.synchronize(dev)
        with ClockSampler(dev.index, period_ms=50) as sclk:
            w0 = time.perf_counter()
            while t_wall < args.sustain_s:
                cev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
                       for _ in range(chunk)]
                for k in range(chunk):
                    assert step(cev[k]) == 0, attn.last_error()
                torch.cuda.synchronize(dev)
                pre_s += sum(e[0].elapsed_time(e[1]) for e in cev) * 1e-3
                dec_s += sum(e[1].elapsed_time(e[2]) for e in cev) * 1e-3
                n_steps += chunk
                t_wall = time.perf_counter() - w0
        assert attn.attn_get_status(stream) == 0
        pre_s, dec_s = max_over_ranks([pre_s, dec_s], dist, dev)
        sc = sclk.summary()
        s_tf = replica_throughput(world, n_steps, flops, pre_s) / 1e12
        s_gbs = replica_throughput(world, n_steps, dec_bytes, dec_s) / 1e9
        mhz = sc.get("sm_mhz")
        sustained = {
            "seconds": t_wall, "steps": n_steps,
            "prefill_tflops": s_tf,
            "prefill_frac_of_sustained_peak": s_tf / world / peaks["bf16_tflops_sustained"],
            "prefill_frac_of_burst_peak": s_tf / world / peaks["bf16_tflops"],
            "decode_gbs": s_gbs, "decode_frac_hbm": s_gbs / world / peaks["hbm_gbs"],
            "clocks": sc,
            # time x clock: cycles per prefill launch at the median clock under load, against
            # the timed region's (comparable when the work per cycle is unchanged)
            "prefill_mcycles_per_launch": (pre_s / n_steps * mhz) if mhz else None,
            "prefill_mcycles_per_launch_timed_region":
                (pre_avg_s * clk.summary()["sm_mhz"]) if clk.summary().get("sm_mhz") else None,
            "peak": f"bf16 sustained {tag} ({peaks['bf16_tflops_sustained']} TFLOP/s: cuBLAS "
                    "bf16 GEMM looped for seconds under the power cap)"}

    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        import oracle
        n, f_done, dt = cpu_baseline_sample(wp, args.cpu_budget, seed=99)
        cpu = {"value": f_done / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
               "kind": "oracle",
               "sample": f"{n} random query rows of {PREFILL_NAME} ({f_done:.3e} FLOP, "
                         f"{dt:.1f} s), fp64 materialised scores"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": prefill_tflops, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": step_config(world),
            "prefill_frac_bf16_peak": prefill_tflops / world / peaks["bf16_tflops"],
            "decode": {"value": decode_gbs, "unit": "GB/s",
                       "frac_hbm": decode_gbs / world / peaks["hbm_gbs"]},
            "roofline": roofline,
            "roofline_decode": roofline_decode,
            "softmax_exp": softmax_exp,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "sustained": sustained,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
