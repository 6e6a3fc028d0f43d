"""Pins for the oracle's vocabulary-sharded cross-entropy (CPU only).

"多卡张量：拆开计算，再合回同一结果", section 04 / VOCABULARY SHARDS: per-shard
max and sum-exp combined into a global log-sum-exp, L = log s - sum_r t_r,
dL/dz_j = e^{z_j - m}/s - 1[j = y]; the shared hidden's gradient is summed
over the vocabulary shards; shifting all logits changes neither the loss nor
the probabilities.  The page's worked example prints only its six logits."""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def worked_logits():
    return np.array(json.load(open(os.path.join(GOLDEN, "ce_worked_logits.json")))["logits"])


def ce_on_logits(orc, z, y, parts=1):
    """Run the oracle's full CE with h = z and W = identity, so the logits are z."""
    V = len(z)
    loss, dlog, dh, own = orc.ce_tokens(np.array([z]), np.eye(V), np.array([y]), parts)
    return loss[0], dlog[0], dh[0], own[0]


def test_worked_example_closed_form(orc):
    z = worked_logits()
    assert z.max() == 2.0
    den = sum(math.exp(v) for v in z)
    p = np.array([math.exp(v) / den for v in z])
    assert abs(p.sum() - 1.0) < 1e-15
    for y in range(6):
        loss, dlog, dh, _ = ce_on_logits(orc, z, y)
        assert abs(loss - (math.log(den) - z[y])) < 1e-14
        onehot = np.eye(6)[y]
        np.testing.assert_allclose(dlog, p - onehot, rtol=0, atol=1e-15)
        assert abs(dlog.sum()) < 1e-15
        np.testing.assert_allclose(dh, dlog, rtol=0, atol=1e-15)   # W = I


@pytest.mark.parametrize("c", [-3.0, 0.5, 100.0, 700.0])
def test_shift_invariance(orc, c):
    z = worked_logits()
    for y in range(6):
        l0, g0, _, _ = ce_on_logits(orc, z, y)
        l1, g1, _, _ = ce_on_logits(orc, z + c, y)
        assert abs(l0 - l1) < 1e-12
        np.testing.assert_allclose(g0, g1, rtol=0, atol=1e-14)


@pytest.mark.parametrize("parts", [1, 2, 3, 4, 5, 6, 7, 9])
def test_sharded_form_equals_unsharded(orc, parts):
    z = worked_logits()
    for y in range(6):
        L, m_r, s_r, t_r = orc.ce_sharded_one(z, y, parts)
        loss, _, _, own = ce_on_logits(orc, z, y, parts)
        assert abs(L - loss) < 1e-14
        off = orc.plan_shards(6, parts)
        owners = [r for r in range(parts) if off[r] <= y < off[r + 1]]
        assert own == owners[0]
        assert np.count_nonzero(t_r) <= 1 and abs(t_r.sum() - (z[y] - 2.0)) < 1e-15
        empty = np.diff(off) == 0
        assert np.all(np.isneginf(m_r[empty])) and np.all(s_r[empty] == 0)


def test_two_shard_statistics(orc):
    z = worked_logits()
    _, m_r, s_r, _ = orc.ce_sharded_one(z, 2, 2)
    assert list(m_r) == [2.0, 1.4]
    assert abs(s_r[0] - sum(math.exp(v - 2.0) for v in z[:3])) < 1e-15
    assert abs(s_r[1] - sum(math.exp(v - 2.0) for v in z[3:])) < 1e-15


def test_random_against_torch(orc):
    rng = np.random.default_rng(2)
    T, d, V = 7, 5, 23
    h, W = rng.standard_normal((T, d)), rng.standard_normal((d, V))
    y = rng.integers(0, V, size=T)
    H = torch.tensor(h, requires_grad=True)
    Z = (H @ torch.tensor(W)).detach().requires_grad_()
    loss = torch.nn.functional.cross_entropy(Z, torch.tensor(y), reduction="none")
    loss.sum().backward()
    dH = Z.grad @ torch.tensor(W).T
    oloss, odlog, odh, own = orc.ce_tokens(h, W, y, 4)
    np.testing.assert_allclose(oloss, loss.detach().numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(odlog, Z.grad.numpy(), rtol=0, atol=1e-14)
    np.testing.assert_allclose(odh, dH.numpy(), rtol=1e-12, atol=1e-13)
    off = orc.plan_shards(V, 4)
    assert list(own) == [int(np.searchsorted(off, v, side="right") - 1) for v in y]


def test_finite_difference_on_logits(orc):
    z = np.random.default_rng(4).standard_normal(11)
    y = 6
    _, g, _, _ = ce_on_logits(orc, z, y)
    h = 1e-6
    for j in range(11):
        e = np.zeros(11); e[j] = h
        fd = (ce_on_logits(orc, z + e, y)[0] - ce_on_logits(orc, z - e, y)[0]) / (2 * h)
        assert abs(fd - g[j]) < 1e-8


def test_no_division_by_shard_count(orc):
    """The hidden gradient is the plain sum over vocabulary shards ("多卡张量",
    04: 不能重复除以并行数): it does not depend on the shard count."""
    rng = np.random.default_rng(9)
    h, W = rng.standard_normal((3, 4)), rng.standard_normal((4, 10))
    y = np.array([0, 5, 9])
    a = orc.ce_tokens(h, W, y, 1)
    b = orc.ce_tokens(h, W, y, 4)
    np.testing.assert_array_equal(a[2], b[2])
    np.testing.assert_array_equal(a[0], b[0])


def test_label_out_of_range(orc):
    with pytest.raises(ValueError, match="label"):
        orc.ce_tokens(np.ones((1, 2)), np.ones((2, 3)), np.array([3]), 1)
