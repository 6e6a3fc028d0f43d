"""Pins for the oracle's gated column-then-row MLP (CPU only).

"第 6 课：张量并行 TP", reference answer Q1 (gate/up projections and the
activation column-parallel, the down projection row-parallel) and core
concept 2.A (element-wise functions pass through the column split; SiLU is
one it names).  The gating product is the usual gated linear unit; these
pins tie it to torch autograd, to finite differences, to the ungated MLP
oracle when the up branch is constant, and to the lesson's per-rank sum."""
import numpy as np
import pytest
import torch

import oracle
from test_oracle_mlp import torch_act as _torch_act

KINDS = [oracle.ACT_SILU, oracle.ACT_GELU_ERF, oracle.ACT_GELU_TANH, oracle.ACT_TANH]


def torch_act(kind, x):
    return torch.nn.functional.silu(x) if kind == oracle.ACT_SILU else _torch_act(kind, x)


def rand_case(seed, T, d, F):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal(s) for s in [(T, d), (d, F), (d, F), (F, d), (T, d)]]


@pytest.mark.parametrize("kind", KINDS)
def test_against_autograd(orc, kind):
    X, Wg, Wu, W2, G = rand_case(1, 13, 8, 19)
    tX, tWg, tWu, tW2 = (torch.tensor(a, requires_grad=True) for a in (X, Wg, Wu, W2))
    Y = (torch_act(kind, tX @ tWg) * (tX @ tWu)) @ tW2
    (Y * torch.tensor(G)).sum().backward()
    got = orc.glu(X, Wg, Wu, W2, G, kind)
    ref = [Y.detach().numpy(), tX.grad.numpy(), tWg.grad.numpy(), tWu.grad.numpy(), tW2.grad.numpy()]
    for name, a, b in zip(["Y", "dX", "dWg", "dWu", "dW2"], got, ref):
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(b).max()), name


def test_finite_differences(orc):
    X, Wg, Wu, W2, G = rand_case(2, 5, 4, 6)
    kind = oracle.ACT_SILU
    grads = orc.glu(X, Wg, Wu, W2, G, kind)[1:]
    L = lambda *a: float(np.sum(G * orc.glu_rows(*a, G, kind)[0]))
    h = 1e-6
    base = [X, Wg, Wu, W2]
    for i, grad in enumerate(grads[:3] + (grads[3],)):
        for idx in [(0, 0), (1, 2), (base[i].shape[0] - 1, base[i].shape[1] - 1)]:
            E = np.zeros_like(base[i]); E[idx] = 1.0
            p, m = list(base), list(base)
            p[i], m[i] = base[i] + h * E, base[i] - h * E
            fd = (L(*p) - L(*m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (i, idx, fd, grad[idx])


@pytest.mark.parametrize("kind", KINDS)
def test_constant_up_branch_is_the_plain_mlp(orc, kind):
    """With a last input feature of ones and Wu selecting only it, U = 1 and
    the gated MLP is the ungated one with W1 = Wg; Y, dWg, dW2 and the other
    columns of dX must agree with the ungated oracle."""
    X, Wg, _, W2, G = rand_case(3, 11, 6, 9)
    X[:, -1] = 1.0
    Wu = np.zeros_like(Wg); Wu[-1, :] = 1.0
    Y, dX, dWg, _, dW2 = orc.glu(X, Wg, Wu, W2, G, kind)
    pY, pdX, pdW1, pdW2 = orc.mlp(X, Wg, W2, G, kind)
    scale = lambda t: max(1.0, float(np.abs(t).max()))
    for a, b in [(Y, pY), (dX[:, :-1], pdX[:, :-1]), (dWg, pdW1), (dW2, pdW2)]:
        assert np.abs(a - b).max() <= 1e-12 * scale(b)


@pytest.mark.parametrize("tp", [1, 3, 4, 7, 40])
def test_tp_sum_equals_unsharded(orc, tp):
    """Each rank gates its own column shard of Hg and U and multiplies by its
    row shard of W2; the rank outputs are summed once (the lesson's tp_mlp
    with the gate/up pair in the column layer)."""
    X, Wg, Wu, W2, G = rand_case(4, 10, 8, 33)
    kind = oracle.ACT_SILU
    oY, odX = orc.glu_rows(X, Wg, Wu, W2, G, kind)
    Y, dX = 0, 0
    for cols in np.array_split(np.arange(33), tp):
        hg, u = X @ Wg[:, cols], X @ Wu[:, cols]
        Y = Y + (orc.act(kind, hg) * u) @ W2[cols, :]
        dA = G @ W2[cols, :].T
        dX = dX + (dA * u * orc.act_grad(kind, hg)) @ Wg[:, cols].T + (dA * orc.act(kind, hg)) @ Wu[:, cols].T
    assert np.abs(Y - oY).max() <= 1e-12 * np.abs(oY).max()
    assert np.abs(dX - odX).max() <= 1e-12 * np.abs(odX).max()


def test_sampled_rows_and_cols_match_full(orc):
    X, Wg, Wu, W2, G = rand_case(5, 9, 6, 11)
    kind = oracle.ACT_SILU
    Y, dX, dWg, dWu, dW2 = orc.glu(X, Wg, Wu, W2, G, kind)
    rows, cols = np.array([8, 0, 3]), np.array([10, 2])
    sY, sdX = orc.glu_rows(X, Wg, Wu, W2, G, kind, rows)
    sdWg, sdWu, sdW2 = orc.glu_cols(X, Wg, Wu, W2, G, kind, cols)
    np.testing.assert_array_equal(sY, Y[rows]); np.testing.assert_array_equal(sdX, dX[rows])
    np.testing.assert_array_equal(sdWg, dWg[:, cols]); np.testing.assert_array_equal(sdWu, dWu[:, cols])
    np.testing.assert_array_equal(sdW2, dW2[cols])
