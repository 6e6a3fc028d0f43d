"""Pins for the oracle's activations (CPU only).

GELU (erf form) is torch's default gelu, used by "第 6 课：张量并行 TP"
(reference answer, tp_mlp / reference_mlp); the tanh form is the common
approximation; tanh with derivative 1 - H^2 is what "多卡张量：拆开计算，
再合回同一结果", section 02 / BACKWARD, writes."""
import math

import numpy as np
import pytest
import torch

import oracle

KINDS = [oracle.ACT_GELU_ERF, oracle.ACT_GELU_TANH, oracle.ACT_TANH, oracle.ACT_SILU]
XS = np.linspace(-6.0, 6.0, 241)


def test_gelu_matches_torch(orc):
    x = torch.tensor(XS, dtype=torch.float64)
    np.testing.assert_allclose(orc.act(oracle.ACT_GELU_ERF, XS),
                               torch.nn.functional.gelu(x).numpy(), rtol=0, atol=1e-15)
    np.testing.assert_allclose(orc.act(oracle.ACT_GELU_TANH, XS),
                               torch.nn.functional.gelu(x, approximate="tanh").numpy(), rtol=0, atol=1e-15)
    np.testing.assert_allclose(orc.act(oracle.ACT_TANH, XS), np.tanh(XS), rtol=0, atol=1e-15)
    np.testing.assert_allclose(orc.act(oracle.ACT_SILU, XS), torch.nn.functional.silu(x).numpy(), rtol=0,
                               atol=1e-15)


@pytest.mark.parametrize("kind", KINDS)
def test_grad_matches_autograd(orc, kind):
    x = torch.tensor(XS, dtype=torch.float64, requires_grad=True)
    if kind == oracle.ACT_GELU_ERF:
        y = torch.nn.functional.gelu(x)
    elif kind == oracle.ACT_GELU_TANH:
        y = torch.nn.functional.gelu(x, approximate="tanh")
    elif kind == oracle.ACT_SILU:
        y = torch.nn.functional.silu(x)
    else:
        y = torch.tanh(x)
    y.sum().backward()
    np.testing.assert_allclose(orc.act_grad(kind, XS), x.grad.numpy(), rtol=0, atol=1e-14)


@pytest.mark.parametrize("kind", KINDS)
def test_grad_finite_difference(orc, kind):
    h = 1e-5
    fd = (orc.act(kind, XS + h) - orc.act(kind, XS - h)) / (2 * h)
    np.testing.assert_allclose(orc.act_grad(kind, XS), fd, rtol=0, atol=1e-9)


def test_gelu_closed_forms(orc):
    # GELU(0) = 0;  x Phi(x) - (-x) Phi(-x) = x (Phi(x) + Phi(-x)) = x
    assert orc.act(oracle.ACT_GELU_ERF, 0.0) == 0.0
    np.testing.assert_allclose(orc.act(oracle.ACT_GELU_ERF, XS) - orc.act(oracle.ACT_GELU_ERF, -XS), XS,
                               rtol=0, atol=1e-14)
    # GELU(1) = Phi(1) = 0.5 (1 + erf(1/sqrt 2))
    assert abs(orc.act(oracle.ACT_GELU_ERF, 1.0) - 0.5 * (1 + math.erf(1 / math.sqrt(2)))) < 1e-16
    # the tanh approximation stays within 1e-3 of the erf form on [-3, 3]
    x = np.linspace(-3, 3, 601)
    assert np.max(np.abs(orc.act(oracle.ACT_GELU_TANH, x) - orc.act(oracle.ACT_GELU_ERF, x))) < 1e-3


def test_silu_closed_forms(orc):
    # SiLU(0) = 0, SiLU'(0) = 1/2, x s(x) - (-x) s(-x) = x (s(x) + s(-x)) = x,
    # SiLU(x) -> x for large x and -> 0 for very negative x
    assert orc.act(oracle.ACT_SILU, 0.0) == 0.0
    assert orc.act_grad(oracle.ACT_SILU, 0.0) == 0.5
    np.testing.assert_allclose(orc.act(oracle.ACT_SILU, XS) - orc.act(oracle.ACT_SILU, -XS), XS, rtol=0, atol=1e-14)
    assert abs(orc.act(oracle.ACT_SILU, 40.0) - 40.0) < 1e-12 and abs(orc.act(oracle.ACT_SILU, -40.0)) < 1e-15
    assert abs(orc.act(oracle.ACT_SILU, 1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16


def test_activation_does_not_commute_with_partial_sum(orc):
    """Negative test: "Sharded GEMM与Backprop", 解题路线 step 5 and
    "第 6 课", core concept 2.A.6: GELU(sum partial) != sum GELU(partial)."""
    lhs = orc.act(oracle.ACT_GELU_ERF, 1.0 + 2.0)
    rhs = orc.act(oracle.ACT_GELU_ERF, 1.0) + orc.act(oracle.ACT_GELU_ERF, 2.0)
    assert abs(lhs - rhs) > 0.19
