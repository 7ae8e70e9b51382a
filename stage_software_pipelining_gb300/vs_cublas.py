"""Side-by-side timing of this library's GEMM and cuBLAS (torch.matmul) on one
GPU, for the bf16 8192^3 problem.

Three arms, run back to back for a few seconds each so that the 1.4 kW power
cap has settled, then repeated in the same order:
  cublas       torch.matmul(A, B, out=C), bf16 in and out (beta = 0)
  ours_bf16    the same problem through gemm() (GEMM_BF16_BF16)
  ours_beta1   C = A*B + C with fp32 C (GEMM_BF16_F32, beta = 1)
For our arms the kernel's own mean SM clock (gemm_clock_log) is printed with
the rate.  The two bf16 outputs are compared element by element.

With --arm NAME --launches N only that arm runs, N times, with no timing:
the form to run under a profiler.

    python -m stage_software_pipelining_gb300.vs_cublas [--seconds 4] [--rounds 2]
    python -m stage_software_pipelining_gb300.vs_cublas --arm cublas --launches 8
"""
import argparse
import json
import os
import statistics
import subprocess
import time

import torch

from . import gemm as G

N = 8192
FLOPS = 2 * N ** 3


def make(seed: int = 0):
    gen = torch.Generator().manual_seed(seed)
    A = (torch.rand(N, N, generator=gen) * 2 - 1).to(torch.bfloat16).cuda()
    B = (torch.rand(N, N, generator=gen) * 2 - 1).to(torch.bfloat16).cuda()
    Cb = torch.empty(N, N, dtype=torch.bfloat16, device="cuda")
    Ct = torch.empty(N, N, dtype=torch.bfloat16, device="cuda")
    Cf = (torch.rand(N, N, generator=gen) * 2 - 1).cuda()
    return A, B, Cb, Ct, Cf


def arms(A, B, Cb, Ct, Cf):
    return {
        "cublas": lambda: torch.matmul(A, B, out=Ct),
        "ours_bf16": lambda: G.gemm(A, B, Cb, 1.0, 0.0),
        "ours_beta1": lambda: G.gemm(A, B, Cf, 1.0, 1.0),
    }


class SmClock:
    """nvidia-smi samples of the SM clock (MHz) every 200 ms while running."""

    def __init__(self):
        dev = torch.cuda.current_device()
        visible = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
        self.index = visible[dev] if dev < len(visible) else str(dev)
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.index, "--query-gpu=clocks.sm",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is not None:
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.samples = [float(x) for x in out.split() if x.replace(".", "", 1).isdigit()]

    def median(self):
        return statistics.median(self.samples) if self.samples else None


def timed(fn, seconds: float, ours: bool) -> dict:
    for _ in range(10):
        fn()
    torch.cuda.synchronize()
    log = torch.zeros(2, dtype=torch.int64, device="cuda") if ours else None
    if ours:
        G.clock_log(log)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with SmClock() as clk:
        t0 = time.time()
        e0.record()
        n = 0
        while time.time() - t0 < seconds:
            for _ in range(50):
                fn()
            n += 50
            torch.cuda.synchronize()
        e1.record()
        torch.cuda.synchronize()
    if ours:
        G.clock_log(None)
    ms = e0.elapsed_time(e1) / n
    out = {"launches": n, "ms": round(ms, 4), "tflops": round(FLOPS / (ms * 1e-3) / 1e12, 1),
           "smi_sm_mhz_median": clk.median()}
    if ours:
        ticks, ns = log.tolist()
        if ns > 0:
            out["kernel_sm_mhz"] = round(ticks * 1000.0 / ns, 1)
    return out


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--seconds", type=float, default=4.0)
    ap.add_argument("--rounds", type=int, default=2)
    ap.add_argument("--arm", choices=["cublas", "ours_bf16", "ours_beta1"])
    ap.add_argument("--launches", type=int, default=0)
    args = ap.parse_args()
    G.load_library()
    A, B, Cb, Ct, Cf = make()
    fns = arms(A, B, Cb, Ct, Cf)
    if args.arm:
        for _ in range(max(1, args.launches)):
            fns[args.arm]()
        torch.cuda.synchronize()
        print(json.dumps({"arm": args.arm, "launches": max(1, args.launches)}))
        return
    fns["cublas"]()
    fns["ours_bf16"]()
    torch.cuda.synchronize()
    same = bool(torch.equal(Cb, Ct))
    diff = (Cb.float() - Ct.float()).abs().max().item()
    print(json.dumps({"bf16_outputs_identical": same, "max_abs_difference": diff}))
    for r in range(args.rounds):
        for name, fn in fns.items():
            res = timed(fn, args.seconds, ours=name != "cublas")
            print(json.dumps({"round": r, "arm": name, **res}), flush=True)
            time.sleep(1.0)


if __name__ == "__main__":
    main()
