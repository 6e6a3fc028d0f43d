"""Pins for the oracle's column-then-row MLP (CPU only).

Forward: "多卡张量：拆开计算，再合回同一结果", section 01 / COLUMN THEN ROW, and
"第 6 课：张量并行 TP", core concept 2.A and the reference answer (tp_mlp,
reference_mlp).  Backward: "多卡张量", section 02 / BACKWARD, which also says
every weight and input gradient can be checked by finite differences."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from backward_tcgen05_tma_gemms_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
KINDS = [oracle.ACT_GELU_ERF, oracle.ACT_GELU_TANH, oracle.ACT_TANH]


def torch_act(kind, x):
    if kind == oracle.ACT_GELU_ERF:
        return torch.nn.functional.gelu(x)
    if kind == oracle.ACT_GELU_TANH:
        return torch.nn.functional.gelu(x, approximate="tanh")
    return torch.tanh(x)


@pytest.mark.parametrize("kind", KINDS)
def test_lesson_mlp_against_autograd(orc, kind):
    x, w1, w2, gy, tp = inputs.lesson_mlp_case()
    X = x.reshape(-1, 64).double().requires_grad_()
    W1 = w1.double().requires_grad_()      # torch (out, in) = (256, 64)
    W2 = w2.double().requires_grad_()      # (64, 256)
    G = gy.reshape(-1, 64).double()
    Y = torch_act(kind, X @ W1.T) @ W2.T
    (Y * G).sum().backward()
    oY, odX, odW1, odW2 = orc.mlp(X.detach().numpy(), W1.detach().numpy().T, W2.detach().numpy().T,
                                  G.numpy(), kind)
    scale = lambda t: max(1.0, float(np.abs(t).max()))
    for got, ref in [(oY, Y.detach().numpy()), (odX, X.grad.numpy()),
                     (odW1.T, W1.grad.numpy()), (odW2.T, W2.grad.numpy())]:
        assert np.abs(got - ref).max() <= 1e-12 * scale(ref)


@pytest.mark.parametrize("kind", KINDS)
def test_finite_differences(orc, kind):
    rng = np.random.default_rng(7)
    T, d, F = 5, 4, 6
    X, W1, W2, G = (rng.standard_normal(s) for s in [(T, d), (d, F), (F, d), (T, d)])
    _, dX, dW1, dW2 = orc.mlp(X, W1, W2, G, kind)
    L = lambda x, w1, w2: float(np.sum(G * orc.mlp_rows(x, w1, w2, G, kind)[0]))
    h = 1e-6
    for name, base, grad in [("X", X, dX), ("W1", W1, dW1), ("W2", W2, dW2)]:
        for idx in [(0, 0), (1, 2), (base.shape[0] - 1, base.shape[1] - 1)]:
            E = np.zeros_like(base); E[idx] = 1.0
            args_p = [X, W1, W2]; args_m = [X, W1, W2]
            i = ["X", "W1", "W2"].index(name)
            args_p[i] = base + h * E; args_m[i] = base - h * E
            fd = (L(*args_p) - L(*args_m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_page_example_inputs_finite_differences(orc):
    """The two-rank example's printed X and G with phi = tanh (whose
    derivative the page writes as 1 - H^2).  Its weights are not printed, so
    seeded weights stand in: parity of this example is pinned only through
    finite differences."""
    g = json.load(open(os.path.join(GOLDEN, "mlp_worked_inputs.json")))
    X, G = np.array(g["X"]), np.array(g["G"])
    rng = np.random.default_rng(11)
    W1, W2 = rng.standard_normal((2, 4)), rng.standard_normal((4, 2))
    kind = oracle.ACT_TANH
    _, dX, dW1, dW2 = orc.mlp(X, W1, W2, G, kind)
    L = lambda x, w1, w2: float(np.sum(G * orc.mlp_rows(x, w1, w2, G, kind)[0]))
    h = 1e-6
    for i, (base, grad) in enumerate([(X, dX), (W1, dW1), (W2, dW2)]):
        for idx in np.ndindex(base.shape):
            E = np.zeros_like(base); E[idx] = 1.0
            a_p, a_m = [X, W1, W2], [X, W1, W2]
            a_p[i], a_m[i] = base + h * E, base - h * E
            fd = (L(*a_p) - L(*a_m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(fd))


@pytest.mark.parametrize("tp", [1, 2, 3, 4, 7, 300])
def test_tp_sum_equals_unsharded(orc, tp):
    """The lesson's tp_mlp: each rank computes phi(X W1_r) W2_r and the
    outputs are summed once; equals the unsharded MLP for any tp, including
    uneven (array_split) and empty shards."""
    x, w1, w2, gy, _ = inputs.lesson_mlp_case()
    X = x.reshape(-1, 64).double().numpy()
    W1, W2 = w1.double().numpy().T, w2.double().numpy().T   # (in, out)
    oY, _ = orc.mlp_rows(X, W1, W2, gy.reshape(-1, 64).double().numpy(), oracle.ACT_GELU_ERF)
    Y = 0
    for cols in np.array_split(np.arange(256), tp):
        H = X @ W1[:, cols]
        Y = Y + orc.act(oracle.ACT_GELU_ERF, H) @ W2[cols, :]
    assert np.abs(Y - oY).max() <= 1e-12 * np.abs(oY).max()


def test_row_then_column_order_is_wrong(orc):
    """Negative test ("第 6 课", core concept 2.A.6): with the first layer split
    by rows, applying the activation to each partial product before the sum
    changes the result."""
    x, w1, w2, gy, _ = inputs.lesson_mlp_case()
    X = x.reshape(-1, 64).double().numpy()
    W1, W2 = w1.double().numpy().T, w2.double().numpy().T
    oY, _ = orc.mlp_rows(X, W1, W2, gy.reshape(-1, 64).double().numpy(), oracle.ACT_GELU_ERF)
    wrong = 0
    for rows in np.array_split(np.arange(64), 4):
        wrong = wrong + orc.act(oracle.ACT_GELU_ERF, X[:, rows] @ W1[rows, :])
    wrong = wrong @ W2
    assert np.abs(wrong - oY).max() > 1e-2 * np.abs(oY).max()


def test_sampled_rows_and_cols_match_full(orc):
    rng = np.random.default_rng(5)
    T, d, F = 9, 6, 11
    X, W1, W2, G = (rng.standard_normal(s) for s in [(T, d), (d, F), (F, d), (T, d)])
    Y, dX, dW1, dW2 = orc.mlp(X, W1, W2, G, oracle.ACT_GELU_TANH)
    rows = np.array([8, 0, 3])
    cols = np.array([10, 2])
    sY, sdX = orc.mlp_rows(X, W1, W2, G, oracle.ACT_GELU_TANH, rows)
    sdW1, sdW2 = orc.mlp_cols(X, W1, W2, G, oracle.ACT_GELU_TANH, cols)
    np.testing.assert_array_equal(sY, Y[rows]); np.testing.assert_array_equal(sdX, dX[rows])
    np.testing.assert_array_equal(sdW1, dW1[:, cols]); np.testing.assert_array_equal(sdW2, dW2[cols])
