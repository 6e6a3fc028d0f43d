"""GPU parity of tps_mlp_fwd_bwd against the float64 oracle.

Column-then-row MLP of "多卡张量：拆开计算，再合回同一结果" (01 / COLUMN THEN ROW,
02 / BACKWARD) and "第 6 课：张量并行 TP" (core concept 2.A; reference answer
tp_mlp with x (2, 8, 64), w1 (256, 64), w2 (64, 256), tp=4, exact GELU)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from backward_tcgen05_tma_gemms_gb300 import api, inputs
from parity import assert_close

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ACTS = {"gelu_erf": oracle.ACT_GELU_ERF, "gelu_tanh": oracle.ACT_GELU_TANH, "tanh": oracle.ACT_TANH,
        "silu": oracle.ACT_SILU}


def oracle_io(W, layout):
    """Weights in (in, out) layout for the oracle."""
    w = inputs.as_f64(W)
    return w if layout == "in_out" else w.T


def run_and_check(orc, X, W1, W2, GY, tp, act, layout, bf16, what=""):
    Y, dX, dW1, dW2 = api.mlp_fwd_bwd(X.cuda(), W1.cuda(), W2.cuda(), GY.cuda(), tp, act, layout)
    assert api.last_device_error() == 0
    d = X.shape[-1]
    x, gy = inputs.as_f64(X).reshape(-1, d), inputs.as_f64(GY).reshape(-1, d)
    rY, rdX, rdW1, rdW2 = orc.mlp(x, oracle_io(W1, layout), oracle_io(W2, layout), gy, ACTS[act])
    if layout == "out_in":
        rdW1, rdW2 = rdW1.T, rdW2.T
    assert_close(Y.cpu().reshape(-1, d), rY, bf16, f"{what} Y")
    assert_close(dX.cpu().reshape(-1, d), rdX, bf16, f"{what} dX")
    assert_close(dW1.cpu(), rdW1, bf16, f"{what} dW1")
    assert_close(dW2.cpu(), rdW2, bf16, f"{what} dW2")
    return Y, dX, dW1, dW2


def test_lesson_exercise_fp32(orc):
    x, w1, w2, gy, tp = inputs.lesson_mlp_case()
    Y, *_ = run_and_check(orc, x, w1, w2, gy, tp, "gelu_erf", "out_in", False, "lesson")
    assert Y.shape == x.shape
    # and within the lesson's own check against the unsharded MLP
    tol = json.load(open(os.path.join(GOLDEN, "tp_mlp_tolerances.json")))["tp_mlp"]
    ref = torch.nn.functional.gelu(x.double() @ w1.double().T) @ w2.double().T
    torch.testing.assert_close(Y.cpu().double(), ref, atol=tol["atol"], rtol=tol["rtol"])


@pytest.mark.parametrize("tp", [1, 3, 8, 300])
def test_fp32_uneven_and_empty_shards(orc, tp):
    X, W1, W2, GY = inputs.mlp_case(tp, 24, 40, 256, torch.float32, w_std=0.2)
    run_and_check(orc, X, W1, W2, GY, tp, "gelu_tanh", "in_out", False, f"tp{tp}")


@pytest.mark.parametrize("act", list(ACTS))
@pytest.mark.parametrize("layout", ["in_out", "out_in"])
def test_bf16_tensor_core(orc, act, layout, gemm_kernel):
    T, d, F = 300, 192, 520
    X, W1, W2, GY = inputs.mlp_case(17, T, d, F, torch.bfloat16, w_std=0.05, layout=layout)
    with api.profile() as p:
        run_and_check(orc, X, W1, W2, GY, 3, act, layout, True, f"{act}/{layout}")
    assert {k.split(":")[0] for k in p.summary} == {"gemm_tc"}, p.summary
    assert p.launches == 6


def test_bf16_multi_wave(orc, gemm_kernel):
    T, d, F = 1024, 512, 2048
    X, W1, W2, GY = inputs.mlp_case(23, T, d, F, torch.bfloat16)
    run_and_check(orc, X, W1, W2, GY, 8, "gelu_tanh", "in_out", True, "1024x512x2048")


def test_llama_shape_sampled(orc):
    """The Llama-3-8B-shaped MLP (T=8192, d=4096, F=14336, tp=8, tanh-GELU,
    bf16) at full size, in the benchmark's launch configuration; the oracle
    recomputes 8 rows of Y and dX and 8 columns of dW1 / rows of dW2."""
    cfg = inputs.LLAMA_MLP
    X, W1, W2, GY = inputs.mlp_case(0, cfg["T"], cfg["d"], cfg["F"], torch.bfloat16)
    Y, dX, dW1, dW2 = api.mlp_fwd_bwd(X.cuda(), W1.cuda(), W2.cuda(), GY.cuda(), cfg["tp"], "gelu_tanh", "in_out")
    assert api.last_device_error() == 0
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(cfg["T"], 8, replace=False))
    # columns spread over every rank's shard, including both ends
    off = api.plan_shards(cfg["F"], cfg["tp"])
    cols = np.array([off[r] + (r * 97) % (off[r + 1] - off[r]) for r in range(cfg["tp"])] + [0, cfg["F"] - 1])
    x, w1, w2, gy = (inputs.as_f64(t) for t in (X, W1, W2, GY))
    rY, rdX = orc.mlp_rows(x, w1, w2, gy, oracle.ACT_GELU_TANH, rows)
    rdW1, rdW2 = orc.mlp_cols(x, w1, w2, gy, oracle.ACT_GELU_TANH, cols)
    assert_close(Y[rows].cpu(), rY, True, "Y rows")
    assert_close(dX[rows].cpu(), rdX, True, "dX rows")
    assert_close(dW1[:, cols].cpu(), rdW1, True, "dW1 cols")
    assert_close(dW2[cols].cpu(), rdW2, True, "dW2 rows")
    for t in (Y, dX, dW1, dW2):
        assert torch.isfinite(t).all()
