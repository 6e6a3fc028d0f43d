"""Run one operation of the library a few times on synthetic inputs, for
profilers (ncu) and quick timing.  Prints per-launch device times from the
library's own launch profiler.

    python -m backward_tcgen05_tma_gemms_gb300.profile_case mlp --T 2048 --reps 2
    python -m backward_tcgen05_tma_gemms_gb300.profile_case glu --T 2048 --reps 1
    python -m backward_tcgen05_tma_gemms_gb300.profile_case ce --T 1024 --reps 2
    python -m backward_tcgen05_tma_gemms_gb300.profile_case matmul --M 4096 --K 4096 --N 4096

Each run does one untimed warm-up call, then `--reps` calls.
"""
import argparse
import json

import torch

from . import api, inputs


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["mlp", "glu", "ce", "matmul"])
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


if __name__ == "__main__":
    main()
