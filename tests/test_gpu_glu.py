"""GPU parity of tps_glu_mlp_fwd_bwd (the gated column-then-row MLP,
SwiGLU for SiLU) against the float64 oracle.

"第 6 课：张量并行 TP", reference answer Q1 (gate/up projections and the
activation in the column-parallel layer, the down projection row-parallel)
and core concept 2.A (element-wise functions stay shard-local)."""
import numpy as np
import pytest
import torch

import oracle
from backward_tcgen05_tma_gemms_gb300 import api, inputs
from parity import assert_close

pytestmark = pytest.mark.gpu
ACTS = {"silu": oracle.ACT_SILU, "gelu_tanh": oracle.ACT_GELU_TANH, "gelu_erf": oracle.ACT_GELU_ERF,
        "tanh": oracle.ACT_TANH}


def io(W, layout):
    w = inputs.as_f64(W)
    return w if layout == "in_out" else w.T


def run_and_check(orc, X, Wg, Wu, W2, GY, tp, act, layout, bf16, what=""):
    out = api.glu_mlp_fwd_bwd(X.cuda(), Wg.cuda(), Wu.cuda(), W2.cuda(), GY.cuda(), tp, act, layout)
    assert api.last_device_error() == 0
    Y, dX, dWg, dWu, dW2 = (t.cpu() for t in out)
    d = X.shape[-1]
    x, gy = inputs.as_f64(X).reshape(-1, d), inputs.as_f64(GY).reshape(-1, d)
    rY, rdX, rdWg, rdWu, rdW2 = orc.glu(x, io(Wg, layout), io(Wu, layout), io(W2, layout), gy, ACTS[act])
    if layout == "out_in":
        rdWg, rdWu, rdW2 = rdWg.T, rdWu.T, rdW2.T
    assert_close(Y.reshape(-1, d), rY, bf16, f"{what} Y")
    assert_close(dX.reshape(-1, d), rdX, bf16, f"{what} dX")
    assert_close(dWg, rdWg, bf16, f"{what} dWg")
    assert_close(dWu, rdWu, bf16, f"{what} dWu")
    assert_close(dW2, rdW2, bf16, f"{what} dW2")


@pytest.mark.parametrize("tp", [1, 3, 8, 300])
def test_fp32_uneven_and_empty_shards(orc, tp):
    X, Wg, Wu, W2, GY = inputs.glu_case(tp, 24, 40, 256, torch.float32, w_std=0.2)
    run_and_check(orc, X, Wg, Wu, W2, GY, tp, "silu", "in_out", False, f"tp{tp}")


def test_fp32_torch_layout_3d_input(orc):
    X, Wg, Wu, W2, GY = inputs.glu_case(5, 16, 64, 96, torch.float32, w_std=0.2, layout="out_in")
    run_and_check(orc, X.reshape(2, 8, 64), Wg, Wu, W2, GY.reshape(2, 8, 64), 4, "silu", "out_in", False, "3d")


@pytest.mark.parametrize("act", list(ACTS))
@pytest.mark.parametrize("layout", ["in_out", "out_in"])
def test_bf16_fused_gate_up(orc, act, layout):
    """Ragged everywhere: T=300 (one full and one partial 256-row pair tile),
    F=520 (four 128-unit gated tiles and an 8-unit tail), tp=3."""
    T, d, F = 300, 192, 520
    X, Wg, Wu, W2, GY = inputs.glu_case(17, T, d, F, torch.bfloat16, w_std=0.05, layout=layout)
    with api.profile() as p:
        run_and_check(orc, X, Wg, Wu, W2, GY, 3, act, layout, True, f"{act}/{layout}")
    assert {k.split(":")[0] for k in p.summary} == {"gemm_tc"}, p.summary
    assert "gemm_tc:glu_gate_up" in p.summary and p.launches == 7, p.summary


def test_bf16_multi_wave(orc):
    T, d, F = 1024, 512, 2048
    X, Wg, Wu, W2, GY = inputs.glu_case(23, T, d, F, torch.bfloat16)
    run_and_check(orc, X, Wg, Wu, W2, GY, 8, "silu", "in_out", True, "1024x512x2048")


def test_bf16_unfusable_up_weight(orc):
    """An up weight whose strides differ from the gate's cannot share the
    gate's tensor map: the gate and up projections then run as two GEMMs
    (the second forms the gating in its epilogue), and dX's two branches,
    whose B operands no longer share a contiguous dimension, go to the
    SIMT kernel.  Results must not change."""
    X, Wg, Wu, W2, GY = inputs.glu_case(29, 200, 128, 384, torch.bfloat16, w_std=0.05)
    Wu_t = Wu.t().contiguous().t()          # same values, column-major storage
    with api.profile() as p:
        run_and_check(orc, X, Wg, Wu_t, W2, GY, 4, "silu", "in_out", True, "unfused")
    assert "gemm_tc:glu_up" in p.summary and "gemm_tc:glu_gate_up" not in p.summary, p.summary


def test_llama_shape_sampled(orc):
    """Llama-3-8B-shaped SwiGLU MLP (T=8192, d=4096, F=14336, tp=8, bf16) at
    full size; the oracle recomputes 8 rows of Y and dX and 10 hidden units'
    columns of dWg, dWu and rows of dW2."""
    cfg = inputs.LLAMA_MLP
    X, Wg, Wu, W2, GY = inputs.glu_case(0, cfg["T"], cfg["d"], cfg["F"], torch.bfloat16)
    out = api.glu_mlp_fwd_bwd(X.cuda(), Wg.cuda(), Wu.cuda(), W2.cuda(), GY.cuda(), cfg["tp"], "silu")
    assert api.last_device_error() == 0
    Y, dX, dWg, dWu, dW2 = out
    rng = np.random.default_rng(2)
    rows = np.sort(rng.choice(cfg["T"], 8, replace=False))
    off = api.plan_shards(cfg["F"], cfg["tp"])
    cols = np.array([off[r] + (r * 131) % (off[r + 1] - off[r]) for r in range(cfg["tp"])] + [0, cfg["F"] - 1])
    x, wg, wu, w2, gy = (inputs.as_f64(t) for t in (X, Wg, Wu, W2, GY))
    rY, rdX = orc.glu_rows(x, wg, wu, w2, gy, oracle.ACT_SILU, rows)
    rdWg, rdWu, rdW2 = orc.glu_cols(x, wg, wu, w2, gy, oracle.ACT_SILU, cols)
    assert_close(Y[rows].cpu(), rY, True, "Y rows")
    assert_close(dX[rows].cpu(), rdX, True, "dX rows")
    assert_close(dWg[:, cols].cpu(), rdWg, True, "dWg cols")
    assert_close(dWu[:, cols].cpu(), rdWu, True, "dWu cols")
    assert_close(dW2[cols].cpu(), rdW2, True, "dW2 rows")
    for t in out:
        assert torch.isfinite(t).all()


@pytest.mark.parametrize("T", [0, 1, 5])
def test_bf16_few_tokens(orc, T):
    """A single pair tile that is almost (or wholly) outside the token range;
    with no tokens every weight gradient is an exact zero."""
    X, Wg, Wu, W2, GY = inputs.glu_case(31 + T, max(T, 1), 64, 256, torch.bfloat16, w_std=0.1)
    X, GY = X[:T].contiguous(), GY[:T].contiguous()
    run_and_check(orc, X, Wg, Wu, W2, GY, 2, "silu", "in_out", True, f"T={T}")
