"""Vocabulary CE with more tokens than one launch's grid.y holds (65,535):
the cluster and two-pass kernels then run in slabs of tokens, and the
extended form's finalize must see every slab's count.  Checked against the
float64 oracle ("多卡张量：拆开计算，再合回同一结果", section 04 / VOCABULARY
SHARDS)."""
import numpy as np
import pytest
import torch

from backward_tcgen05_tma_gemms_gb300 import api, inputs
from parity import assert_close

pytestmark = pytest.mark.gpu
T = 70001
IGN = -100


@pytest.mark.parametrize("tp,V", [(3, 96), (9, 90)], ids=["cluster", "two_pass"])
def test_fp32_token_slabs(orc, tp, V):
    h, W, labels = inputs.ce_case(11 + tp, T, 8, V, torch.float32, w_std=0.5)
    loss, dlog, dh, own = api.vocab_ce_fwd_bwd(h.cuda(), W.cuda(), labels.cuda(), tp)
    assert api.last_device_error() == 0
    toks = np.array([0, 1, 65534, 65535, 65536, 65537, T - 1])
    rl, rdl, rdh, rown = orc.ce_tokens(inputs.as_f64(h), inputs.as_f64(W), labels.numpy(), tp, toks)
    assert_close(loss[toks].cpu(), rl, False, "loss")
    assert_close(dlog[toks].cpu(), rdl, False, "dlogits")
    assert_close(dh[toks].cpu(), rdh, False, "dHidden")
    off = np.array(api.plan_shards(V, tp))
    assert np.array_equal(own.cpu().numpy(), np.searchsorted(off, labels.numpy(), side="right") - 1)
    assert torch.isfinite(loss).all()


@pytest.mark.parametrize("dtype,V,tp,d", [(torch.float32, 96, 3, 8), (torch.bfloat16, 512, 4, 16)],
                         ids=["fp32_two_pass", "bf16_fused"])
def test_extended_mean_over_slabs(orc, dtype, V, tp, d):
    """ignore_index on every seventh token, vocabulary padding and a mean
    over all supervised tokens of all slabs; everything is compared."""
    h, W, labels = inputs.ce_case(5, T, d, V, dtype, w_std=0.2)
    vr = V - 5
    y = labels.numpy() % vr
    y[::7] = IGN
    y = torch.from_numpy(y)
    loss, red, dlog, dh, dw, own = api.vocab_ce_fwd_bwd_ex(h.cuda(), W.cuda(), y.cuda(), tp, ignore_index=IGN,
                                                           vocab_size=vr, reduction="mean", want_dwhead=True)
    assert api.last_device_error() == 0
    rl, rred, rdl, rdh, rdw, rown = orc.ce_ex(inputs.as_f64(h), inputs.as_f64(W), y.numpy(), tp, IGN, vr, 2)
    bf16 = dtype == torch.bfloat16
    assert_close(loss.cpu(), rl, bf16, "loss")
    assert_close(dlog.cpu(), rdl, bf16, "dlogits")
    assert_close(dh.cpu(), rdh, bf16, "dHidden")
    assert_close(dw.cpu(), rdw, bf16, "dWhead")
    assert np.array_equal(own.cpu().numpy(), rown)
    assert abs(red.item() - rred) <= (2e-2 if bf16 else 1e-4) * abs(rred)
