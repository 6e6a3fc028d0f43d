"""GPU parity of tps_vocab_ce_fwd_bwd_ex (vocabulary padding, ignore_index,
sum / mean reduction with a local or job-wide denominator, the head's
gradient) against the oracle's extended cross-entropy.

"多卡张量：拆开计算，再合回同一结果", section 04 / VOCABULARY SHARDS (padding
and ignore_index in a real implementation) and "Sharded GEMM与Backprop",
section 易错点与追问 (a loss denominator that stays consistent across ranks
whose batches hold different numbers of supervised tokens)."""
import numpy as np
import pytest
import torch

from backward_tcgen05_tma_gemms_gb300 import api, inputs
from parity import assert_close

pytestmark = pytest.mark.gpu
IGN = -100
REDS = {"none": 0, "sum": 1, "mean": 2}


def case(seed, T, d, V, vr, dtype, n_ignore, w_std=0.3, ign=IGN):
    h, W, _ = inputs.ce_case(seed, T, d, V, dtype, w_std=w_std)
    rng = np.random.default_rng(seed + 1)
    y = rng.integers(0, vr, size=T)
    y[rng.choice(T, n_ignore, replace=False)] = ign
    return h, W, torch.from_numpy(y)


def run(h, W, y, tp, vr, reduction, denom, layout="in_out", ign=IGN):
    out = api.vocab_ce_fwd_bwd_ex(h.cuda(), W.cuda(), y.cuda(), tp, layout, ignore_index=ign, vocab_size=vr,
                                  reduction=reduction, denominator=denom, want_dwhead=True)
    assert api.last_device_error() == 0
    return [None if t is None else t.cpu() for t in out]


def check(orc, h, W, y, tp, vr, reduction, denom, bf16, what, layout="in_out", ign=IGN):
    loss, red, dlog, dh, dw, own = run(h, W, y, tp, vr, reduction, denom, layout, ign)
    w64 = inputs.as_f64(W) if layout == "in_out" else inputs.as_f64(W).T
    rl, rred, rdl, rdh, rdw, rown = orc.ce_ex(inputs.as_f64(h), w64, y.numpy(), tp, ign, vr, REDS[reduction], denom)
    assert_close(loss, rl, bf16, f"{what} loss")
    assert_close(dlog, rdl, bf16, f"{what} dlogits")
    assert_close(dh, rdh, bf16, f"{what} dHidden")
    assert_close(dw if layout == "in_out" else dw.t(), rdw, bf16, f"{what} dWhead")
    assert np.array_equal(own.numpy(), rown), f"{what} owner"
    if reduction != "none":
        assert abs(red.item() - rred) <= (2e-2 if bf16 else 1e-4) * max(1.0, abs(rred)), (red.item(), rred)
    ignored = torch.from_numpy(y.numpy() == ign)
    assert not dlog[ignored].any() and not loss[ignored].any(), what
    if 0 < vr < dlog.shape[1]:
        assert not dlog[:, vr:].any(), what


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
def test_fp32_two_pass(orc, reduction):
    h, W, y = case(1, 37, 48, 1000, 990, torch.float32, 5)
    check(orc, h, W, y, 3, 990, reduction, 0.0, False, f"fp32 {reduction}")


def test_fp32_job_denominator(orc):
    h, W, y = case(2, 21, 32, 700, 700, torch.float32, 4)
    check(orc, h, W, y, 5, 0, "mean", 123.0, False, "fp32 mean/123")


def test_fp32_all_ignored_mean(orc):
    """No supervised token: every loss and gradient is 0, the mean is 0."""
    h, W, y = case(3, 9, 16, 300, 300, torch.float32, 9)
    check(orc, h, W, y, 4, 0, "mean", 0.0, False, "all ignored")


def test_fp32_ignore_index_is_a_class(orc):
    """ignore_index = 0 names a real column: its one-hot must not appear."""
    h, W, y = case(4, 30, 16, 200, 200, torch.float32, 6, ign=0)
    check(orc, h, W, y, 3, 0, "sum", 0.0, False, "ignore 0", ign=0)


@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_bf16_statistics_from_the_logits_epilogue(orc, reduction, gemm_kernel):
    """Shards of at least one 128-column statistics tile: the fused path,
    with the padding boundary inside a statistics tile."""
    h, W, y = case(5, 300, 256, 32000, 31990, torch.bfloat16, 17, w_std=0.05)
    with api.profile() as p:
        check(orc, h, W, y, 8, 31990, reduction, 0.0, True, f"bf16 fused {reduction}")
    assert "ce_stream" in {k.split(":")[0] for k in p.summary}, p.summary


def test_bf16_shard_all_padding(orc, gemm_kernel):
    """The last shard (28672..32767) lies wholly in the padding; out_in head."""
    h, W, y = case(6, 130, 128, 32768, 28000, torch.bfloat16, 3, w_std=0.05)
    W = W.t().contiguous()
    check(orc, h, W, y, 8, 28000, "mean", 0.0, True, "bf16 padded shard", layout="out_in")


def test_bf16_two_pass(orc):
    """Shards narrower than a statistics tile take the two-pass kernels."""
    h, W, y = case(7, 64, 64, 1000, 996, torch.bfloat16, 9, w_std=0.2)
    with api.profile() as p:
        check(orc, h, W, y, 9, 996, "mean", 0.0, True, "bf16 two-pass mean")
    kinds = {k.split(":")[0] for k in p.summary}
    assert "ce_stats" in kinds and "ce_grad" in kinds, p.summary


def test_data_parallel_denominator(orc):
    """Two data-parallel batches with different numbers of supervised tokens,
    each divided by the job-wide count: the per-batch means and head
    gradients add up to those of the whole job."""
    h, W, y = case(8, 200, 128, 4096, 4096, torch.bfloat16, 40, w_std=0.05)
    y[:100][torch.arange(100) % 3 == 0] = IGN       # uneven masks
    total = int((y != IGN).sum())
    parts = [run(h[a:b], W, y[a:b], 4, 0, "mean", float(total)) for a, b in ((0, 100), (100, 200))]
    rl, rred, rdl, rdh, rdw, rown = orc.ce_ex(inputs.as_f64(h), inputs.as_f64(W), y.numpy(), 4, IGN, 0, 2, 0.0)
    red = sum(p[1].item() for p in parts)
    assert abs(red - rred) <= 2e-2 * max(1.0, abs(rred)), (red, rred)
    assert_close(parts[0][4] + parts[1][4], rdw, True, "dWhead summed over batches")
    assert_close(torch.cat([parts[0][3], parts[1][3]]), rdh, True, "dHidden")


def test_defaults_match_the_plain_entry_point():
    """No option set: the same kernels, bit-identical results."""
    h, W, y = inputs.ce_case(9, 100, 128, 8192, torch.bfloat16)
    h, W, y = h.cuda(), W.cuda(), y.cuda()
    a = api.vocab_ce_fwd_bwd(h, W, y, 8)
    loss, red, dlog, dh, dw, own = api.vocab_ce_fwd_bwd_ex(h, W, y, 8)
    assert red is None and dw is None
    for u, v in zip(a, (loss, dlog, dh, own)):
        assert torch.equal(u, v)


def test_no_tokens():
    h = torch.zeros(0, 32, device="cuda", dtype=torch.bfloat16)
    W = torch.randn(32, 512, device="cuda").to(torch.bfloat16)
    y = torch.zeros(0, dtype=torch.int64, device="cuda")
    loss, red, dlog, dh, dw, own = api.vocab_ce_fwd_bwd_ex(h, W, y, 4, reduction="sum", want_dwhead=True)
    assert api.last_device_error() == 0
    assert red.item() == 0.0 and not dw.any() and dw.shape == W.shape


def test_label_in_padding_is_an_error():
    h, W, _ = inputs.ce_case(10, 4, 16, 64, torch.float32)
    y = torch.tensor([0, 63, 2, IGN])       # 63 lies in the padding when vocab_size = 60
    loss, red, dlog, dh, dw, own = api.vocab_ce_fwd_bwd_ex(h.cuda(), W.cuda(), y.cuda(), 2, ignore_index=IGN,
                                                           vocab_size=60)
    assert api.last_device_error() == api.ERR_LABEL
    l = loss.cpu()
    assert torch.isnan(l[1]) and l[3] == 0 and torch.isfinite(l[[0, 2]]).all()
    assert own.cpu().tolist()[1] == -1


def test_bad_options():
    h, W, y = inputs.ce_case(11, 4, 16, 64, torch.float32)
    h, W, y = h.cuda(), W.cuda(), y.cuda()
    with pytest.raises(ValueError):
        api.vocab_ce_fwd_bwd_ex(h, W, y, 2, vocab_size=65)
    with pytest.raises(api.TpsError):
        api.vocab_ce_fwd_bwd_ex(h, W, y, 2, reduction="mean", denominator=-1.0)


def test_int32_labels_match_int64(gemm_kernel):
    """ignore_index, padding and the mean with int32 labels: bit-identical
    to the same call with int64 labels (fused statistics path)."""
    h, W, y = case(91, 300, 128, 4096, 4000, torch.bfloat16, 40)
    a = run(h, W, y, 4, 4000, "mean", 0.0)
    b = run(h, W, y.to(torch.int32), 4, 4000, "mean", 0.0)
    for x, z in zip(a, b):
        assert torch.equal(x, z)


def test_llama_shape_sampled(orc):
    """Llama-3-8B vocabulary head (T=8192, d=4096, V=128256 whose last 256
    columns are padding, tp=8), every eighth label ignored, the mean over
    the batch's supervised tokens and the head's gradient, at full size in
    the benchmark's launch configuration.  64 supervised tokens spread over
    the batch get labels at both ends of every shard's real columns (each
    rank owns eight; the first ones in tiles shared with the previous
    shard), and with four ignored tokens they are recomputed by the oracle
    with the batch's supervised count as the divisor: loss, dlogits row,
    dHidden row and owner.  The padding columns of dlogits are zero, four
    columns of dWhead match h^T dlogits in float64, and the reduced loss is
    the mean of the per-token losses."""
    from test_gpu_ce import boundary_labels, spread_tokens
    cfg = inputs.LLAMA_CE
    T, V, tp = cfg["T"], cfg["V"], cfg["tp"]
    vr = V - 256
    h, W, y = inputs.ce_case(0, T, cfg["d"], V, torch.bfloat16)
    y = y % vr
    y[::8] = IGN
    sup = spread_tokens(T, 64, 6, avoid_mod=8)
    y[torch.from_numpy(sup)] = torch.from_numpy(boundary_labels(V, tp, vr))
    toks = np.sort(np.concatenate([sup, [0, 8, 4096, T - 8]]))
    loss, red, dlog, dh, dw, own = api.vocab_ce_fwd_bwd_ex(h.cuda(), W.cuda(), y.cuda(), tp, ignore_index=IGN,
                                                           vocab_size=vr, reduction="mean", want_dwhead=True)
    assert api.last_device_error() == 0
    D = int((y != IGN).sum())
    rl, _, rdl, rdh, _, rown = orc.ce_ex(inputs.as_f64(h[toks]), inputs.as_f64(W), y[toks].numpy(), tp, IGN, vr, 2,
                                         float(D), want_dwhead=False)
    assert_close(loss[toks].cpu(), rl, True, "loss")
    assert_close(dlog[toks].cpu(), rdl, True, "dlogits")
    assert_close(dh[toks].cpu(), rdh, True, "dHidden")
    assert np.array_equal(own[toks].cpu().numpy(), rown)
    assert np.bincount(rown[rown >= 0], minlength=tp).min() >= 4 and (rown == -1).sum() == 4
    assert not dlog[:, vr:].any()
    cols = [0, 12345, 64000, vr - 1]
    ref = inputs.as_f64(h).T @ dlog[:, cols].cpu().double().numpy()
    assert_close(dw[:, cols].cpu(), ref, True, "dWhead columns")
    l = loss.cpu().double()
    assert abs(red.item() - l.sum().item() / D) <= 1e-4 * abs(red.item())
