"""GPU parity of tps_matmul_fwd_bwd against the float64 oracle.

"Sharded GEMM与Backprop：行、列、内维三种切分": the M=3 K=5 N=4 parts=2 case
and the 1000-case random sweep of section 手动走一遍 (fp32, every axis,
parts up to 20 so that parts > dim gives empty shards), plus bf16 operands
on the tcgen05 tensor-core kernel at multi-tile sizes with ragged tails, in
every operand layout."""
import numpy as np
import pytest
import torch

from backward_tcgen05_tma_gemms_gb300 import api, inputs
from parity import assert_close

pytestmark = pytest.mark.gpu


def gpu_mm(A, B, G, parts, axis, out=None):
    Y, dA, dB = api.matmul_fwd_bwd(A.cuda(), B.cuda(), G.cuda(), parts, axis, out=out)
    assert api.last_device_error() == 0
    return Y.cpu(), dA.cpu(), dB.cpu()


def check(orc, A, B, G, parts, axis, bf16=False, what=""):
    ref = orc.matmul(inputs.as_f64(A), inputs.as_f64(B), inputs.as_f64(G))
    got = gpu_mm(A, B, G, parts, axis)
    for name, g, r in zip(("Y", "dA", "dB"), got, ref):
        assert_close(g, r, bf16, f"{what} {axis} {name}")


def test_plan_shards_bit_exact(orc):
    for dim in [0, 1, 5, 17, 14336, 128256]:
        for parts in [1, 2, 3, 7, 8, 20, 300]:
            assert api.plan_shards(dim, parts) == list(orc.plan_shards(dim, parts))


@pytest.mark.parametrize("axis", inputs.AXES)
def test_worked_case(orc, axis):
    A, B, G, parts = inputs.worked_matmul_case()
    check(orc, A, B, G, parts, axis, what="M3K5N4")


def test_sweep_1000_cases_three_axes(orc):
    for seed in range(1000):
        A, B, G, parts = inputs.sweep_case(seed)
        ref = orc.matmul(A.double().numpy(), B.double().numpy(), G.double().numpy())
        for axis in inputs.AXES:
            got = gpu_mm(A, B, G, parts, axis)
            for name, g, r in zip(("Y", "dA", "dB"), got, ref):
                assert_close(g, r, False, f"seed {seed} {axis} {name}")


# (4808, 384, 712): 19 pair rows walked in raster groups of 16 and a ragged 3,
# with a ragged last column tile
TC_SHAPES = [(128, 64, 256), (300, 200, 520), (1, 64, 8), (257, 1000, 136), (520, 72, 264), (1024, 512, 768),
             (4808, 384, 712)]


@pytest.mark.parametrize("M,K,N", TC_SHAPES)
def test_bf16_tensor_core(orc, M, K, N, gemm_kernel):
    A, B, G = inputs.matmul_case(M * 7 + K, M, K, N, torch.bfloat16)
    with api.profile() as p:
        check(orc, A, B, G, 3, "inner", bf16=True, what=f"{M}x{K}x{N}")
    kinds = {k.split(":")[0] for k in p.summary}
    assert kinds == {"gemm_tc"}, p.summary     # all three GEMMs on the tensor cores


@pytest.mark.parametrize("axis", ["rows", "columns"])
@pytest.mark.parametrize("parts", [3, 8])
def test_bf16_tensor_core_row_and_column_splits(orc, axis, parts, gemm_kernel):
    """Row and column splits on the tensor cores: one operand's gradient is
    the rank sum, accumulated in the contraction loop, the other is the
    concatenation of the shards' results."""
    A, B, G = inputs.matmul_case(parts * 11 + len(axis), 600, 320, 776, torch.bfloat16)
    with api.profile() as p:
        check(orc, A, B, G, parts, axis, bf16=True, what=f"600x320x776 p{parts}")
    assert {k.split(":")[0] for k in p.summary} == {"gemm_tc"}, p.summary


def test_bf16_unaligned_strides_use_simt(orc):
    A, B, G = inputs.matmul_case(5, 37, 13, 29, torch.bfloat16)
    with api.profile() as p:
        check(orc, A, B, G, 4, "rows", bf16=True, what="37x13x29")
    assert {k.split(":")[0] for k in p.summary} == {"gemm_simt"}


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_transposed_views_and_column_major_outputs(orc, dtype, gemm_kernel):
    M, K, N = 136, 192, 264
    A, B, G = inputs.matmul_case(11, M, K, N, dtype)
    At = A.t().contiguous().cuda().t()      # A viewed column-major
    Bt = B.t().contiguous().cuda().t()
    Yc = torch.empty(N, M, device="cuda").t()
    dAc = torch.empty(K, M, device="cuda").t()
    dBc = torch.empty(N, K, device="cuda").t()
    got = api.matmul_fwd_bwd(At, Bt, G.cuda(), 2, "columns", out=(Yc, dAc, dBc))
    assert api.last_device_error() == 0
    ref = orc.matmul(inputs.as_f64(A), inputs.as_f64(B), inputs.as_f64(G))
    for name, g, r in zip(("Y", "dA", "dB"), got, ref):
        assert_close(g.cpu(), r, dtype == torch.bfloat16, f"views {name}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_empty_contraction_and_empty_outputs(orc, dtype):
    # K = 0: Y is the zero matrix, dA and dB are empty.
    A, B, G = torch.zeros(4, 0, dtype=dtype), torch.zeros(0, 8, dtype=dtype), torch.ones(4, 8, dtype=dtype)
    Y, dA, dB = gpu_mm(A, B, G, 3, "inner")
    assert Y.shape == (4, 8) and not Y.any() and dA.shape == (4, 0) and dB.shape == (0, 8)
    # M = 0 with K > 0: dB is zero (sum over no rows), Y and dA empty.
    A, B, G = torch.zeros(0, 16, dtype=dtype), torch.ones(16, 8, dtype=dtype), torch.zeros(0, 8, dtype=dtype)
    Y, dA, dB = gpu_mm(A, B, G, 5, "rows")
    assert Y.shape == (0, 8) and dA.shape == (0, 16) and dB.shape == (16, 8) and not dB.any()


def test_more_ranks_than_rows(orc):
    A, B, G = inputs.matmul_case(3, 5, 9, 6)
    for axis in inputs.AXES:
        check(orc, A, B, G, 20, axis, what="parts>dim")


def test_sharded_outputs_are_ranges_of_one_buffer(orc):
    """Concatenated results: each logical rank's slice (array_split plan) of
    Y and dA under the rows split equals that rank's own product."""
    A, B, G = inputs.matmul_case(9, 50, 24, 40)
    Y, dA, _ = gpu_mm(A, B, G, 7, "rows")
    off = api.plan_shards(50, 7)
    for r in range(7):
        a = inputs.as_f64(A)[off[r]:off[r + 1]]
        g = inputs.as_f64(G)[off[r]:off[r + 1]]
        assert_close(Y[off[r]:off[r + 1]], a @ inputs.as_f64(B), False, f"rank {r} Y")
        assert_close(dA[off[r]:off[r + 1]], g @ inputs.as_f64(B).T, False, f"rank {r} dA")


@pytest.mark.parametrize("env", [{"TPS_GEMM_L2_HINTS": "21"}, {"TPS_GEMM_L2_HINTS": "12"},
                                 {"TPS_GEMM_L2_HINTS": "1"}, {"TPS_GEMM_GROUP": "4"}, {"TPS_GEMM_GROUP": "64"}],
                         ids=["hints21", "hints12", "hints1", "group4", "group64"])
def test_tuning_switches_keep_results_bit_identical(env, gemm_kernel, monkeypatch):
    """L2 eviction hints on the operand loads and the raster group size
    change which pair computes a tile and how its operands are cached, not
    the arithmetic: every output is bit-identical to the default launch."""
    A, B, G = (t.cuda() for t in inputs.matmul_case(5, 2600, 448, 1000, torch.bfloat16))
    base = api.matmul_fwd_bwd(A, B, G, 4, "inner")
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    tuned = api.matmul_fwd_bwd(A, B, G, 4, "inner")
    assert api.last_device_error() == 0
    for x, y in zip(base, tuned):
        assert torch.equal(x, y)
