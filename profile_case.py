"""Run one operation of the library a few times on synthetic inputs, for
profilers (ncu) and quick timing.  Prints per-launch device times from the
library's own launch profiler.

    python profile_case.py mlp --T 2048 --reps 2
    python profile_case.py glu --T 2048 --reps 1
    python profile_case.py ce --T 1024 --reps 2
    python profile_case.py matmul --M 4096 --K 4096 --N 4096
    python profile_case.py sustained --N 8192 --seconds 3

`sustained` runs the library's bf16 GEMM Y = A B (N x N x N, fp32 Y, CTA
pairs and one-CTA tiles) and torch.matmul (cuBLAS, bf16 out) back to back,
each in a loop of about `--seconds` seconds, sampling the SM clock and the
board power with nvidia-smi, and prints TFLOP/s, the medians, TFLOP/s per
kW and per GHz for each.

Each run does one untimed warm-up call, then `--reps` calls.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from backward_tcgen05_tma_gemms_gb300 import api, inputs  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["mlp", "glu", "ce", "matmul", "sustained"])
    ap.add_argument("--seconds", type=float, default=3.0)
    ap.add_argument("--T", type=int, default=2048)
    ap.add_argument("--d", type=int, default=4096)
    ap.add_argument("--F", type=int, default=14336)
    ap.add_argument("--V", type=int, default=128256)
    ap.add_argument("--tp", type=int, default=8)
    ap.add_argument("--M", type=int, default=4096)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--N", type=int, default=4096)
    ap.add_argument("--axis", default="inner")
    ap.add_argument("--reps", type=int, default=2)
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
    if a.op == "sustained":
        sustained(a, dev)
        return
    if a.op == "mlp":
        X, W1, W2, GY = (t.to(dev) for t in inputs.mlp_case(0, a.T, a.d, a.F, torch.bfloat16))
        call = lambda: api.mlp_fwd_bwd(X, W1, W2, GY, a.tp, "gelu_tanh", "in_out")
    elif a.op == "glu":
        X, Wg, Wu, W2, GY = (t.to(dev) for t in inputs.glu_case(0, a.T, a.d, a.F, torch.bfloat16))
        call = lambda: api.glu_mlp_fwd_bwd(X, Wg, Wu, W2, GY, a.tp, "silu", "in_out")
    elif a.op == "ce":
        h, W, labels = (t.to(dev) for t in inputs.ce_case(0, a.T, a.d, a.V, torch.bfloat16))
        call = lambda: api.vocab_ce_fwd_bwd(h, W, labels, a.tp)
    else:
        A, B, G = (t.to(dev) for t in inputs.matmul_case(0, a.M, a.K, a.N, torch.bfloat16))
        call = lambda: api.matmul_fwd_bwd(A, B, G, a.tp, a.axis)
    call()
    torch.cuda.synchronize()
    with api.profile() as p:
        for _ in range(a.reps):
            call()
        torch.cuda.synchronize()
    rc = api.last_device_error()
    out = {k: dict(v, ms_per_launch=v["ms"] / v["launches"],
                   tflops=(v["flops"] / (v["ms"] * 1e-3) / 1e12) if v["flops"] else None,
                   gbs=(v["bytes"] / (v["ms"] * 1e-3) / 1e9) if v["bytes"] else None)
           for k, v in p.summary.items()}
    print(json.dumps({"op": a.op, "args": vars(a), "device_error": rc, "launches": out}, indent=1))
    if rc != 0:
        raise SystemExit(f"device error {rc}")


def _sample_loop(fn, seconds, dev):
    """Run fn in a loop for about `seconds`, sampling clock and power."""
    lines = []
    smi = subprocess.Popen(["nvidia-smi", "--query-gpu=clocks.sm,power.draw", "--format=csv,noheader,nounits",
                            "-lms", "100", "-i", str(dev.index or 0)], stdout=subprocess.PIPE,
                           stderr=subprocess.DEVNULL, text=True)
    reader = threading.Thread(target=lambda: [lines.append(x) for x in smi.stdout], daemon=True)
    reader.start()
    for _ in range(5):
        fn()
    torch.cuda.synchronize(dev)
    time.sleep(0.3)
    skip = len(lines)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0, n = time.time(), 0
    e0.record()
    while time.time() - t0 < seconds:
        for _ in range(10):
            fn()
        n += 10
        torch.cuda.synchronize(dev)
    e1.record()
    torch.cuda.synchronize(dev)
    smi.terminate()
    reader.join(timeout=2)
    vals = [x.strip().split(",") for x in lines[skip:] if x.strip()]
    clk = statistics.median(float(v[0]) for v in vals) if vals else float("nan")
    pw = statistics.median(float(v[1]) for v in vals) if vals else float("nan")
    return e0.elapsed_time(e1) / n, clk, pw


def sustained(a, dev):
    N = a.N
    gen = torch.Generator(device="cpu").manual_seed(0)
    A = (torch.randn(N, N, generator=gen) * 0.05).to(torch.bfloat16).to(dev)
    B = (torch.randn(N, N, generator=gen) * 0.05).to(torch.bfloat16).to(dev)
    Y = torch.empty(N, N, device=dev, dtype=torch.float32)
    C = torch.empty(N, N, device=dev, dtype=torch.bfloat16)
    lib = api.library()
    ta, tb, ty = api._tt(A), api._tt(B), api._tt(Y)

    def ours():  # Y only: the forward GEMM of tps_matmul_fwd_bwd
        rc = lib.tps_matmul_fwd_bwd(api._ref(ta), api._ref(tb), api._ref(ta), 1, 0, api._ref(ty), None, None,
                                    api._stream(dev))
        if rc != 0:
            raise RuntimeError(f"tps_matmul_fwd_bwd returned {rc}")

    res = {}
    for name in ("tps_cta_pair", "tps_one_cta", "cublas"):
        if name == "cublas":
            fn = lambda: torch.matmul(A, B, out=C)
        else:
            os.environ["TPS_GEMM_KERNEL"] = "2" if name == "tps_cta_pair" else "1"
            fn = ours
        ms, clk, pw = _sample_loop(fn, a.seconds, dev)
        tf = 2.0 * N ** 3 / (ms * 1e-3) / 1e12
        res[name] = dict(tflops=round(tf, 1), sm_mhz=clk, power_w=round(pw, 1),
                         tflops_per_kw=round(tf / pw * 1e3, 1), tflops_per_ghz=round(tf / clk * 1e3, 1))
        time.sleep(2)
    os.environ.pop("TPS_GEMM_KERNEL", None)
    if api.last_device_error() != 0:
        raise SystemExit("device error")
    print(json.dumps({"op": "sustained", "N": N, "seconds": a.seconds, "results": res}, indent=1))


if __name__ == "__main__":
    main()
