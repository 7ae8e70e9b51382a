"""Benchmark of the software-pipelined GEMM (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--stages S] [--tile-n T]
                    [--no-sweep] [--no-e2e] [--no-cpu]

A step is one call of the GEMM over the workload's matrices (the whole hot
path: tile loop, N-stage ring, tcgen05 MMAs, epilogue).  The default workload
is C = A*B + C with M = N = K = 8192, bf16 inputs, fp32 accumulation and
fp32 C (beta = 1): A, B and C (805 MB) are larger than the 129 MB L2, so no
flush is needed between steps.  Inputs are seeded synthetic matrices.

Reported: TFLOP/s (2*M*N*K per step) over exactly K timed steps measured with
CUDA events on the launching stream; the dominant kernel's roofline (FLOPs
per launch / mean launch time against the measured dense bf16 peak); the
end-to-end number through the host-buffer entry point (host->device copies,
GEMM, device->host copy per step); the stage sweep; SM clocks sampled during
the timed region; and the CPU oracle timed on a bounded sample.

With N > 1 (torchrun, one rank per GPU) every rank runs an independent
replica of the same workload (the GEMM has no exchange step); value is the
sum over ranks of the work divided by the slowest rank's time.

--impl reference times the CPU oracle instead (fp64 triple loop on the host
cores), each step a bounded block of C of the same workload, sized so that
the whole run takes about two minutes; rank 0 alone runs it.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s & % of sm_103a MMA/FMA peak (bf16 8192³), vs pipeline stages"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "bf16_8192_beta1"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_tc_bf16_8192_traffic.txt")
SWEEP_PAUSE_S = 0.25   # idle time before each stage-sweep entry

KERNEL_SOURCES = ["stage_software_pipelining_gb300/csrc/gemm_tc_sm103a.cu",
                  "stage_software_pipelining_gb300/csrc/ptx.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--stages", type=int, default=0, help="0 = the workload's default")
    ap.add_argument("--tile", type=int, default=0,
                    help="tensor-core tile code: 0 auto, 128 (128x128), 256 (128x256), "
                         "512 (256x256 on a CTA pair), 1024 (256x512 on a CTA pair)")
    ap.add_argument("--schedule", type=int, default=0, choices=[0, 1, 2],
                    help="tensor-core tile schedule: 0 the library's automatic choice, "
                         "1 whole tiles, 2 stream-K tail")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_hash() -> str:
    """Hash of the kernel sources with comments and blank space removed, so
    that a comment edit does not disown the committed ncu traffic figures
    while any change to the code does."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


TILE_NAMES = {128: "128x128x64 (1 SM)", 256: "128x256x64 (1 SM)",
              512: "256x256x64 (CTA pair, cta_group::2)",
              1024: "256x512x64 (CTA pair, cta_group::2, two N=256 MMAs per K step)"}
# Every stage is a K slice of 64; the deepest ring each tile has room for.
TILE_MAX_STAGES = {128: 6, 256: 4, 512: 6, 1024: 4}
SCHEDULE_NAMES = {0: "automatic", 1: "whole tiles", 2: "stream-K tail"}
# Default ring depth per tile: the deepest ring that fits.
TILE_DEFAULT_STAGES = dict(TILE_MAX_STAGES)


def committed_traffic(workload: str, stages: int, tile: int):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source for this launch configuration."""
    try:
        fields = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if (fields.get("kernel_sha") == kernel_hash() and fields.get("workload") == workload
                and int(fields.get("stages", -1)) == stages
                and int(fields.get("tile", -1)) == tile):
            return float(fields["traffic_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (200 ms period)."""
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == len(self.FIELDS):
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        loaded = [s for s in sm if smax and s >= 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- ranks
def rank_max(value: float, device) -> float:
    """The largest `value` over all ranks (the slowest rank's time); `value`
    itself without a process group.  NCCL ranks pass their CUDA device, gloo
    ranks the CPU."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_rank_step: float, steps: int, world: int, slowest_s: float) -> float:
    """Units per second of the whole job: every rank does the same work per
    step (weak scaling), the job ends with the slowest rank."""
    return work_per_rank_step * steps * world / slowest_s


# ----------------------------------------------------------------------------- our arm
def run_ours(args):
    import torch

    from stage_software_pipelining_gb300 import gemm as G
    from stage_software_pipelining_gb300.workloads import BY_NAME, GEMM_F32, OUT_DTYPE, make_inputs

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    G.load_library()
    G.schedule_set(args.schedule)

    w = BY_NAME[args.workload]
    tile = args.tile
    if w.dtype == GEMM_F32:
        stages = args.stages or 2
    else:
        if tile == 0:   # the library's automatic choice (for the ring asked for, if any)
            tile = G.resolve_tile(w.M, w.N, w.K, w.dtype, stages=args.stages or 4)
        stages = args.stages or TILE_DEFAULT_STAGES[tile]
    inp = make_inputs(w)
    A = inp.A.to(dev)
    B = (inp.B.t().contiguous().t() if w.b_col_major else inp.B).to(dev)
    C = (inp.C0.to(dev) if inp.C0 is not None
         else torch.zeros(w.M, w.N, dtype=OUT_DTYPE[w.dtype], device=dev))
    stream = torch.cuda.current_stream(dev)

    def step(s=stages, t=tile):
        G.gemm(A, B, C, w.alpha, w.beta, stages=s, tile=t, stream=stream)

    G.gemm(A, B, C, w.alpha, w.beta, stages=stages, tile=tile, stream=stream, checked=True)
    for _ in range(args.warmup):
        step()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    visible = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    phys = int(visible[local]) if local < len(visible) and visible[local].isdigit() else local
    sampler = ClockSampler(phys)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # The tensor-core kernel's own SM clock: CTA 0 of each timed launch adds
    # its clock ticks and nanoseconds here (two atomics per launch).
    clk_log = torch.zeros(2, dtype=torch.int64, device=dev)
    G.clock_log(clk_log)
    sampler.start()
    barrier()
    t0.record(stream)
    # One kernel launch per step and nothing else on the stream: the events
    # bracket the whole region (events between the launches would leave gaps
    # as long as a small GEMM), and the mean launch time is the region / steps.
    for _ in range(args.steps):
        step()
    t1.record(stream)
    barrier()
    clocks = sampler.stop()
    G.clock_log(None)
    ticks, ns = (int(v) for v in clk_log.tolist())
    kernel_mhz = ticks * 1000.0 / ns if ns > 0 else None
    elapsed_ms = t0.elapsed_time(t1)
    launch_ms = elapsed_ms / args.steps
    elapsed_ms = rank_max(elapsed_ms, dev)
    flops_step = w.flops
    value = whole_job_rate(flops_step, args.steps, world, elapsed_ms * 1e-3) / 1e12

    # the stage sweep (same workload, same launch stream).  Each entry starts
    # after a short idle pause, so that no entry inherits the power state (and
    # clock) that the entries before it left behind.
    sweep = []
    if not args.no_sweep and w.dtype != GEMM_F32:
        for tn in (G.TILE_128x128, G.TILE_128x256, G.TILE_256x256_2SM, G.TILE_256x512_2SM):
            for s in range(1, TILE_MAX_STAGES[tn] + 1):
                reps = max(10, min(200, args.steps // 10))
                time.sleep(SWEEP_PAUSE_S)
                for _ in range(3):
                    step(s, tn)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize(dev)
                e0.record(stream)
                for _ in range(reps):
                    step(s, tn)
                e1.record(stream)
                torch.cuda.synchronize(dev)
                ms = e0.elapsed_time(e1) / reps
                sweep.append({"tile": TILE_NAMES[tn], "stages": s, "ms": round(ms, 4),
                              "tflops": round(flops_step / (ms * 1e-3) / 1e12, 1)})
    elif not args.no_sweep:
        for frag, frag_name in ((G.SIMT_FRAGMENTS_DOUBLE, "double-buffered register fragments"),
                                (G.SIMT_FRAGMENTS_SINGLE, "single register fragments")):
            for s in (1, 2, 3, 4):
                reps = max(10, min(200, args.steps // 10))
                time.sleep(SWEEP_PAUSE_S)
                for _ in range(3):
                    step(s, frag)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize(dev)
                e0.record(stream)
                for _ in range(reps):
                    step(s, frag)
                e1.record(stream)
                torch.cuda.synchronize(dev)
                ms = e0.elapsed_time(e1) / reps
                sweep.append({"fragments": frag_name, "stages": s, "ms": round(ms, 4),
                              "tflops": round(flops_step / (ms * 1e-3) / 1e12, 1)})

    # end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e:
        hA = inp.A.pin_memory()
        hB = (inp.B.t().contiguous().pin_memory().t() if w.b_col_major
              else inp.B.contiguous().pin_memory())
        hC = (inp.C0.clone() if inp.C0 is not None else torch.zeros_like(C, device="cpu"))
        hC = hC.pin_memory()
        e2e_steps = max(3, min(30, args.steps))
        G.gemm_host(hA, hB, hC, w.alpha, w.beta, stages=stages, tile=tile, stream=stream)
        barrier()
        h0 = time.perf_counter()
        for _ in range(e2e_steps):
            G.gemm_host(hA, hB, hC, w.alpha, w.beta, stages=stages, tile=tile, stream=stream)
        barrier()
        h_s = rank_max(time.perf_counter() - h0, dev)
        h2d = hA.numel() * hA.element_size() + hB.numel() * hB.element_size()
        if w.beta != 0.0:
            h2d += hC.numel() * hC.element_size()
        d2h = hC.numel() * hC.element_size()
        e2e = {"value": round(whole_job_rate(flops_step, e2e_steps, world, h_s) / 1e12, 2),
               "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": e2e_steps, "entry": "gemm_host (pinned host buffers)"}
        G.load_library().gemm_host_release()

    peaks, peak_kind = load_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    max_mhz = peaks.get("sm_max_mhz", 2070.0)
    if w.dtype == GEMM_F32:
        # FP32 FMA pipe: 128 lanes per SM, 2 FLOP per fused multiply-add.
        achieved = flops_step / (launch_ms * 1e-3) / 1e12
        peak = sms * 128 * 2 * max_mhz * 1e-6
        roof = {"bound": "alu", "achieved": round(achieved, 2), "peak": round(peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                "peak_kind": f"FP32 FMA pipe: {sms} SMs x 128 lanes x 2 FLOP x {max_mhz:g} MHz "
                             f"(max SM clock)",
                "algorithmic_flops_per_launch": flops_step,
                "algorithmic_bytes_per_launch": algorithmic_bytes(w),
                "kernel": "sgemm_simt_kernel", "mean_launch_ms": round(launch_ms, 4)}
        if clocks and clocks.get("sm_mhz"):
            pk = sms * 128 * 2 * clocks["sm_mhz"] * 1e-6
            roof["at_sampled_clock"] = {"sm_mhz": clocks["sm_mhz"], "peak": round(pk, 1),
                                        "frac": round(achieved / pk, 4)}
        if kernel_mhz:
            # the clock the kernel itself ran at (CTA 0's clock64 over globaltimer)
            pk = sms * 128 * 2 * kernel_mhz * 1e-6
            roof["per_clock"] = {"kernel_sm_mhz": round(kernel_mhz, 1),
                                 "peak_at_kernel_clock": round(pk, 1),
                                 "frac": round(achieved / pk, 4)}
        roof["model"] = roofline_model(w, flops_step, achieved, peak, peaks)
    else:
        sustained = elapsed_ms > 1000.0
        peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        achieved = flops_step / (launch_ms * 1e-3) / 1e12
        traffic = committed_traffic(w.name, stages, tile)
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_kind": f"{peak_kind} cuBLAS bf16 8192^3, "
                             f"{'sustained' if sustained else 'burst'}",
                "frac_of_burst": round(achieved / peaks["bf16_tflops"], 4),
                "algorithmic_flops_per_launch": flops_step,
                "algorithmic_bytes_per_launch": algorithmic_bytes(w),
                "kernel": "gemm_tc_kernel", "mean_launch_ms": round(launch_ms, 4)}
        # The per-SM tensor rate measured on this GPU (after the timed region):
        # the GEMM against SMs x that rate x the clock sampled under load.
        # The per-SM tensor rate of the instruction this tile issues: the
        # CTA-pair form for the 256-row tiles, the one-CTA form otherwise.
        pair_tile = tile in (G.TILE_256x256_2SM, G.TILE_256x512_2SM)
        rate = G.mma_rate(n_mma=8192, pair=pair_tile)
        per_clock = {"flop_per_clk_per_sm": round(rate["flop_per_clk_per_sm"], 1),
                     "probe": (f"{rate['ctas'] // 2} CTA pairs x {rate['n_mma']} tcgen05.mma."
                               f"cta_group::2 256x256x16" if pair_tile else
                               f"{rate['ctas']} CTAs x {rate['n_mma']} tcgen05.mma 128x256x16")
                              + f", SM clocks {rate['cycles_min']}..{rate['cycles_max']}",
                     "peak_at_max_clock": round(rate["flop_per_clk_per_sm"] * sms
                                                * max_mhz * 1e-6, 1)}
        per_clock["frac_at_max_clock"] = round(achieved / per_clock["peak_at_max_clock"], 4)
        per_clock["frac_of_nominal_dense"] = round(achieved / NOMINAL_DENSE_TFLOPS, 4)
        if kernel_mhz:
            # the clock the GEMM itself ran at (CTA 0's clock64 over globaltimer)
            pk = rate["flop_per_clk_per_sm"] * sms * kernel_mhz * 1e-6
            per_clock.update({"kernel_sm_mhz": round(kernel_mhz, 1),
                              "peak_at_kernel_clock": round(pk, 1),
                              "frac": round(achieved / pk, 4)})
        roof["per_clock"] = per_clock
        roof["model"] = roofline_model(w, flops_step, achieved, per_clock["peak_at_max_clock"],
                                       peaks)

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(inp, budget_s=12.0)

    if rank == 0:
        line = {
            "metric": METRIC if w.name == DEFAULT_WORKLOAD else f"GEMM TFLOP/s ({w.name})",
            "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if w.dtype == GEMM_F32 else ("f16" if w.dtype == 1 else "bf16"),
            "data": "synthetic (seeded)",
            "config": {"workload": describe(w), "M": w.M, "N": w.N, "K": w.K,
                       "alpha": w.alpha, "beta": w.beta, "stages": stages,
                       "schedule": SCHEDULE_NAMES[args.schedule],
                       "tile": "128x64x32 (SIMT)" if w.dtype == GEMM_F32
                       else TILE_NAMES[tile], "b_layout": "col" if w.b_col_major else "row",
                       "l2": f"inputs larger than L2 ({algorithmic_bytes(w) / 1e6:.0f} MB "
                             f"touched per step > 129 MB); no flush",
                       "parallelism": f"replicas x{world}"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps, "clocks": clocks, "stage_sweep": sweep,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


NOMINAL_HBM_GBS = 8000.0        # the "8 TB/s-class" HBM3e figure
NOMINAL_DENSE_TFLOPS = 2250.0   # GB300 dense bf16/fp16 tensor rate, nominal


def roofline_model(w, flops, achieved, compute_peak, peaks):
    """The roofline of the workload: min(compute peak, arithmetic intensity x
    HBM bandwidth), with the bandwidth both as measured (copy) and nominal."""
    b = algorithmic_bytes(w)
    ai = flops / b
    hbm_meas = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    out = {"arithmetic_intensity_flop_per_byte": round(ai, 1),
           "compute_peak_tflops": round(compute_peak, 1)}
    for key, bw in (("measured", hbm_meas), ("nominal_8tbs", NOMINAL_HBM_GBS)):
        hbm_bound = ai * bw / 1000.0
        roof = min(compute_peak, hbm_bound)
        out[key] = {"hbm_gbs": bw, "hbm_bound_tflops": round(hbm_bound, 1),
                    "roofline_tflops": round(roof, 1),
                    "bound": "compute" if compute_peak <= hbm_bound else "hbm",
                    "frac": round(achieved / roof, 4)}
    return out


def describe(w):
    from stage_software_pipelining_gb300.workloads import IN_DTYPE, OUT_DTYPE
    i = str(IN_DTYPE[w.dtype]).replace("torch.", "")
    o = str(OUT_DTYPE[w.dtype]).replace("torch.", "")
    return (f"{w.name}: C = {w.alpha:g}*A*B + {w.beta:g}*C, M={w.M} N={w.N} K={w.K}, "
            f"{i} inputs, fp32 accumulate, {o} output, B {'column' if w.b_col_major else 'row'}"
            f"-major")


def algorithmic_bytes(w) -> int:
    from stage_software_pipelining_gb300.workloads import IN_DTYPE, OUT_DTYPE
    import torch
    si = torch.tensor([], dtype=IN_DTYPE[w.dtype]).element_size()
    so = torch.tensor([], dtype=OUT_DTYPE[w.dtype]).element_size()
    b = (w.M * w.K + w.K * w.N) * si + w.M * w.N * so
    if w.beta != 0.0:
        b += w.M * w.N * so
    return int(b)


# ----------------------------------------------------------------------------- CPU oracle
def _oracle_block(inp, r0, r1, c0, c1, nthreads=0):
    """Time the oracle on the block C[r0:r1, c0:c1] of the workload
    (nthreads 0: every host core)."""
    import oracle
    w = inp.workload
    B = inp.B[:, c0:c1]
    C0 = inp.C0[:, c0:c1] if (w.beta != 0.0 and inp.C0 is not None) else None
    t = time.perf_counter()
    oracle.gemm(inp.A, B, C0, w.alpha, w.beta, rows=(r0, r1), nthreads=nthreads,
                with_abs=False)
    return time.perf_counter() - t


def _calibrate(inp, rows):
    """Seconds per column of C for `rows` rows (one row per thread)."""
    w = inp.workload
    cols = min(w.N, 256)
    return _oracle_block(inp, 0, rows, 0, cols) / cols


def cpu_baseline(inp, budget_s: float):
    """The oracle as it stands on the host cores, on a block sample of the workload."""
    import oracle
    w = inp.workload
    cores = oracle.max_threads()
    rows = max(1, min(w.M, cores))
    per_col = _calibrate(inp, rows)          # seconds per column for `rows` rows
    want_cols = budget_s / max(per_col, 1e-9)
    if want_cols <= w.N:
        cols = max(16, int(want_cols))
    else:                                    # whole rows: grow the row count instead
        cols = w.N
        rows = max(rows, min(w.M, rows * int(want_cols / w.N)))
    dt = _oracle_block(inp, 0, rows, 0, cols)
    flops = 2.0 * rows * cols * w.K
    out = {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": cores,
           "threads": cores, "kind": "oracle", "seconds": round(dt, 2),
           "sample": f"C[0:{rows}, 0:{cols}] of the {w.name} workload (K={w.K}) = "
                     f"{flops:.3e} FLOP, fp64 i-k-j loop, one row per OpenMP thread"}
    if w.name in SINGLE_THREAD_WORKLOADS:
        out["single_thread"] = cpu_single_thread(inp, budget_s=4.0)
    return out


# The three smaller workloads are also timed on one host thread.
SINGLE_THREAD_WORKLOADS = ("fp32_256", "fp32_2048", "fp16_2048")


def cpu_single_thread(inp, budget_s: float):
    """The oracle on ONE host thread, on whole rows of C (the whole problem
    when it fits the budget)."""
    w = inp.workload
    t1 = _oracle_block(inp, 0, 1, 0, w.N, nthreads=1)      # one row
    rows = int(max(1, min(w.M, budget_s / max(t1, 1e-9))))
    dt = _oracle_block(inp, 0, rows, 0, w.N, nthreads=1)
    flops = 2.0 * rows * w.N * w.K
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "threads": 1,
            "seconds": round(dt, 3),
            "sample": f"C[0:{rows}, 0:{w.N}] of the {w.name} workload (K={w.K}) = "
                      f"{flops:.3e} FLOP" + (" (the whole problem)" if rows == w.M else "")}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from stage_software_pipelining_gb300.workloads import BY_NAME, make_inputs
    w = BY_NAME[args.workload]
    inp = make_inputs(w)
    cores = oracle.max_threads()
    rows = max(1, min(w.M, cores))
    # size each step so that warmup + steps take about two minutes of CPU time
    per_col = _calibrate(inp, rows)
    total_steps = max(args.steps + args.warmup, 1)
    cols = max(16, min(w.N, int(120.0 / total_steps / max(per_col, 1e-9))))
    n_blocks = max(1, (w.M // rows) * (w.N // cols))

    def block(i):
        b = i % n_blocks
        r0 = (b % max(w.M // rows, 1)) * rows
        c0 = (b // max(w.M // rows, 1)) * cols
        return r0, min(r0 + rows, w.M), c0, min(c0 + cols, w.N)

    for i in range(args.warmup):
        _oracle_block(inp, *block(i))
    t = time.perf_counter()
    for i in range(args.steps):
        _oracle_block(inp, *block(args.warmup + i))
    el = time.perf_counter() - t
    flops = 2.0 * rows * cols * w.K * args.steps
    value = flops / el / 1e12
    line = {
        "impl": "reference", "metric": METRIC if w.name == DEFAULT_WORKLOAD
        else f"GEMM TFLOP/s ({w.name})",
        "value": round(value, 6), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": describe(w), "M": w.M, "N": w.N, "K": w.K,
                   "sample_block_per_step": [rows, cols], "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores,
                         "kind": "oracle",
                         "sample": f"a {rows}x{cols} block of C per step (K={w.K}), "
                                   f"fp64 i-k-j loop, one row per OpenMP thread"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


COPY_BYTES = 1 << 30


def run_copy(args):
    """The bandwidth-bound counter-example: a 1 GiB streaming copy through an
    N-stage shared-memory ring, swept over the stage count."""
    import torch

    from stage_software_pipelining_gb300 import gemm as G
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    G.load_library()
    gen = torch.Generator(device="cpu").manual_seed(20261202)
    src = torch.randint(0, 256, (COPY_BYTES,), generator=gen, dtype=torch.uint8).to(dev)
    dst = torch.empty_like(src)
    stream = torch.cuda.current_stream(dev)
    stages = args.stages or 2

    def timed(s, reps):
        for _ in range(3):
            G.pipelined_copy(dst, src, s, stream=stream)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            G.pipelined_copy(dst, src, s, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps

    for _ in range(args.warmup):
        G.pipelined_copy(dst, src, stages, stream=stream)
    visible = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    phys = int(visible[local]) if local < len(visible) and visible[local].isdigit() else local
    sampler = ClockSampler(phys)
    sampler.start()
    torch.cuda.synchronize(dev)
    ms = timed(stages, args.steps)
    clocks = sampler.stop()
    gbs = 2.0 * COPY_BYTES / (ms * 1e-3) / 1e9
    sweep = []
    if not args.no_sweep:
        for s in range(1, 9):
            m = timed(s, max(10, min(100, args.steps)))
            sweep.append({"stages": s, "ms": round(m, 4),
                          "gbs": round(2.0 * COPY_BYTES / (m * 1e-3) / 1e9, 1)})
    peaks, kind = load_peaks()
    line = {"metric": "pipelined streaming copy GB/s (1 GiB), vs pipeline stages",
            "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic (seeded)",
            "config": {"workload": "copy_1g: dst = src, 1 GiB, 8 KB bulk copies (TMA) in and "
                                   "out of an N-slot shared-memory ring per CTA, grid-stride",
                       "stages": stages,
                       "l2": "1 GiB read + 1 GiB written per step > 129 MB L2; no flush"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "traffic": None, "peak_kind": f"{kind} torch copy_ bandwidth",
                         "algorithmic_bytes_per_launch": 2 * COPY_BYTES,
                         "kernel": "pipelined_copy_kernel"},
            "gpu_launches": args.steps, "clocks": clocks, "stage_sweep": sweep,
            "cpu_baseline": None, "e2e": None}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.workload == "copy_1g":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the copy workload has no CPU arm; the oracle arm times the GEMM"}))
            return
        run_copy(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
