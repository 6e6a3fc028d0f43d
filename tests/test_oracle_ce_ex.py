"""Pins for the oracle's extended cross-entropy (CPU only): vocabulary
padding, ignore_index and the loss denominator.

"多卡张量：拆开计算，再合回同一结果", section 04 (a real implementation also
handles vocabulary padding and ignore_index) and "Sharded GEMM与Backprop",
section 易错点与追问 (a loss denominator consistent across ranks whose batches
have uneven masks)."""
import numpy as np
import pytest
import torch

IGN = -100


def torch_ref(h, W, y, vr, reduction, denominator=0.0):
    H = torch.tensor(h, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    z = H @ Wt
    zr = z[:, :vr]
    per = torch.nn.functional.cross_entropy(zr, torch.tensor(y), ignore_index=IGN, reduction="none")
    if reduction == "none":
        out = per.sum()
    elif reduction == "sum":
        out = per.sum()
    else:
        n = int((torch.tensor(y) != IGN).sum())
        out = per.sum() / (denominator if denominator > 0 else max(n, 1))
    z.retain_grad()
    out.backward()
    return per.detach().numpy(), float(out), z.grad.numpy(), H.grad.numpy(), Wt.grad.numpy()


@pytest.mark.parametrize("reduction,code", [("none", 0), ("sum", 1), ("mean", 2)])
@pytest.mark.parametrize("vr", [37, 40])
def test_against_torch(orc, reduction, code, vr):
    rng = np.random.default_rng(3)
    T, d, V = 11, 6, 40
    h, W = rng.standard_normal((T, d)), rng.standard_normal((d, V))
    y = rng.integers(0, vr, size=T)
    y[[2, 7]] = IGN
    loss, red, dlog, dh, dw, own = orc.ce_ex(h, W, y, 4, IGN, vr, code)
    per, out, gz, gh, gw = torch_ref(h, W, y, vr, reduction)
    np.testing.assert_allclose(loss, per, rtol=1e-12, atol=1e-13)
    if code:
        assert abs(red - out) < 1e-12 * max(1.0, abs(out))
    np.testing.assert_allclose(dlog, gz, rtol=0, atol=1e-14)
    np.testing.assert_allclose(dh, gh, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dw, gw, rtol=1e-12, atol=1e-13)
    assert list(own[[2, 7]]) == [-1, -1]
    assert not dlog[[2, 7]].any() and not dlog[:, vr:].any()


def test_global_denominator(orc):
    """Two 'ranks' with uneven masks: the mean over the whole job equals
    the sum of each rank's partial sums divided by the job's total count,
    which each rank receives as `denominator`."""
    rng = np.random.default_rng(4)
    d, V = 5, 30
    W = rng.standard_normal((d, V))
    h1, h2 = rng.standard_normal((7, d)), rng.standard_normal((4, d))
    y1 = rng.integers(0, V, 7); y1[[0, 2]] = IGN          # 5 valid here, 4 on the other rank
    y2 = rng.integers(0, V, 4)
    total = int((y1 != IGN).sum() + (y2 != IGN).sum())
    _, r1, g1, _, _, _ = orc.ce_ex(h1, W, y1, 3, IGN, 0, 2, float(total))
    _, r2, g2, _, _, _ = orc.ce_ex(h2, W, y2, 3, IGN, 0, 2, float(total))
    _, rall, gall, _, _, _ = orc.ce_ex(np.vstack([h1, h2]), W, np.concatenate([y1, y2]), 3, IGN, 0, 2)
    assert abs((r1 + r2) - rall) < 1e-12
    np.testing.assert_allclose(np.vstack([g1, g2]), gall, rtol=0, atol=1e-15)
    # dividing each rank by its own count is the plausible mistake: it differs
    _, l1, _, _, _, _ = orc.ce_ex(h1, W, y1, 3, IGN, 0, 2)
    _, l2, _, _, _, _ = orc.ce_ex(h2, W, y2, 3, IGN, 0, 2)
    assert abs((l1 + l2) / 2 - rall) > 1e-3


def test_reduces_to_plain_ce(orc):
    rng = np.random.default_rng(5)
    T, d, V = 6, 4, 17
    h, W = rng.standard_normal((T, d)), rng.standard_normal((d, V))
    y = rng.integers(0, V, T)
    loss, _, dlog, dh, _, own = orc.ce_ex(h, W, y, 3)
    l0, g0, dh0, own0 = orc.ce_tokens(h, W, y, 3)
    np.testing.assert_array_equal(loss, l0)
    np.testing.assert_array_equal(dlog, g0)
    np.testing.assert_allclose(dh, dh0, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(own, own0)


def test_padding_equals_truncated_head(orc):
    rng = np.random.default_rng(6)
    T, d, V, vr = 5, 4, 24, 19
    h, W = rng.standard_normal((T, d)), rng.standard_normal((d, V))
    y = rng.integers(0, vr, T)
    loss, _, dlog, dh, _, _ = orc.ce_ex(h, W, y, 2, IGN, vr, 0)
    lt, gt, dht, _ = orc.ce_tokens(h, W[:, :vr], y, 2)
    np.testing.assert_allclose(loss, lt, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dlog[:, :vr], gt, rtol=0, atol=1e-15)
    np.testing.assert_allclose(dh, dht, rtol=1e-12, atol=1e-13)


def test_all_ignored_and_bad_label(orc):
    h, W = np.ones((3, 2)), np.ones((2, 5))
    y = np.full(3, IGN)
    loss, red, dlog, dh, dw, own = orc.ce_ex(h, W, y, 2, IGN, 0, 2)
    assert red == 0.0 and not loss.any() and not dlog.any() and not dw.any() and list(own) == [-1] * 3
    with pytest.raises(ValueError, match="label"):
        orc.ce_ex(h, W, np.array([0, 4, 1]), 2, IGN, 4, 0)     # 4 is padding
