"""Pins for the oracle's sharded-GEMM definition (CPU only).

"Sharded GEMM与Backprop：行、列、内维三种切分": L = <G, AB> (题意与假设),
dA = G B^T and dB = A^T G (解题路线 step 1), and each split -- rows, columns,
inner -- must equal the unsharded result (解题路线 steps 2-4, 手动走一遍).
The sharded forms below are the page's per-rank formulas (concatenate the
sharded results, sum the partial products) written with numpy; the oracle
itself computes only the unsharded definition."""
import numpy as np
import pytest
import torch

from backward_tcgen05_tma_gemms_gb300 import inputs


def sharded_numpy(A, B, G, parts, axis):
    """Per-rank simulation: concat for sharded results, sum for partials."""
    if axis == "rows":
        As, Gs = np.array_split(A, parts, 0), np.array_split(G, parts, 0)
        Y = np.concatenate([a @ B for a in As], 0)
        dA = np.concatenate([g @ B.T for g in Gs], 0)
        dB = sum((a.T @ g for a, g in zip(As, Gs)), np.zeros_like(B))
    elif axis == "columns":
        Bs, Gs = np.array_split(B, parts, 1), np.array_split(G, parts, 1)
        Y = np.concatenate([A @ b for b in Bs], 1)
        dA = sum((g @ b.T for b, g in zip(Bs, Gs)), np.zeros_like(A))
        dB = np.concatenate([A.T @ g for g in Gs], 1)
    else:
        As, Bs = np.array_split(A, parts, 1), np.array_split(B, parts, 0)
        Y = sum((a @ b for a, b in zip(As, Bs)), np.zeros_like(G))
        dA = np.concatenate([G @ b.T for b in Bs], 1)
        dB = np.concatenate([a.T @ G for a in As], 0)
    return Y, dA, dB


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def test_unsharded_equals_numpy_matmul(orc):
    rng = np.random.default_rng(0)
    for M, K, N in [(3, 5, 4), (1, 1, 1), (7, 1, 9), (16, 16, 16), (33, 17, 5)]:
        A, B, G = _rand(rng, M, K), _rand(rng, K, N), _rand(rng, M, N)
        Y, dA, dB = orc.matmul(A, B, G)
        np.testing.assert_allclose(Y, A @ B, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(dA, G @ B.T, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(dB, A.T @ G, rtol=1e-13, atol=1e-13)


def test_empty_contraction_gives_zeros(orc):
    A, B, G = np.zeros((3, 0)), np.zeros((0, 4)), np.ones((3, 4))
    Y, dA, dB = orc.matmul(A, B, G)
    assert Y.shape == (3, 4) and not Y.any()
    assert dA.shape == (3, 0) and dB.shape == (0, 4)


def test_finite_differences(orc):
    """L is bilinear, so the central difference is exact up to rounding:
    (L(A + hE) - L(A - hE)) / 2h = <dA, E>, likewise for B."""
    rng = np.random.default_rng(3)
    M, K, N = 6, 5, 7
    A, B, G = _rand(rng, M, K), _rand(rng, K, N), _rand(rng, M, N)
    _, dA, dB = orc.matmul(A, B, G)
    L = lambda a, b: float(np.sum(G * orc.matmul(a, b, G)[0]))
    h = 1e-3
    for _ in range(5):
        E = _rand(rng, M, K)
        fd = (L(A + h * E, B) - L(A - h * E, B)) / (2 * h)
        assert abs(fd - np.sum(dA * E)) <= 1e-9 * max(1.0, abs(fd))
        E = _rand(rng, K, N)
        fd = (L(A, B + h * E) - L(A, B - h * E)) / (2 * h)
        assert abs(fd - np.sum(dB * E)) <= 1e-9 * max(1.0, abs(fd))
    # single-entry probes catch a transposed index that a random E might hide
    for (i, j) in [(0, 1), (2, 4), (5, 0)]:
        E = np.zeros((M, K)); E[i, j] = 1.0
        fd = (L(A + h * E, B) - L(A - h * E, B)) / (2 * h)
        assert abs(fd - dA[i, j]) <= 1e-9 * max(1.0, abs(fd))


def test_worked_case_against_torch_autograd(orc):
    A, B, G, parts = inputs.worked_matmul_case()
    a = A.double().requires_grad_(); b = B.double().requires_grad_()
    y = a @ b
    (y * G.double()).sum().backward()
    Y, dA, dB = orc.matmul(A.numpy(), B.numpy(), G.numpy())
    np.testing.assert_allclose(Y, y.detach().numpy(), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(dA, a.grad.numpy(), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(dB, b.grad.numpy(), rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("axis", inputs.AXES)
def test_sweep_sharded_equals_unsharded(orc, axis):
    """The sweep of section 手动走一遍 (first 200 seeds here; all 1000 run in
    the GPU parity test), including parts > dim."""
    for seed in range(200):
        A, B, G, parts = inputs.sweep_case(seed)
        A, B, G = (t.double().numpy() for t in (A, B, G))
        ref = orc.matmul(A, B, G)
        got = sharded_numpy(A, B, G, parts, axis)
        for r, s in zip(ref, got):
            scale = max(1.0, np.abs(r).max(initial=0.0))
            assert np.abs(r - s).max(initial=0.0) <= 1e-12 * scale


def test_rows_split_needs_the_db_sum(orc):
    """Negative test (手动走一遍): with the rows split, the per-rank dB_r must
    be summed; keeping one rank's dB_r (a replica that was never reduced)
    does not match the unsharded gradient."""
    A, B, G, _ = inputs.worked_matmul_case()
    A, B, G = (t.double().numpy() for t in (A, B, G))
    _, _, dB = orc.matmul(A, B, G)
    As, Gs = np.array_split(A, 2, 0), np.array_split(G, 2, 0)
    for r in range(2):
        assert np.abs(As[r].T @ Gs[r] - dB).max() > 1e-3
    # dividing the sum by the rank count (averaging) is also wrong
    assert np.abs(sum(a.T @ g for a, g in zip(As, Gs)) / 2 - dB).max() > 1e-3
