"""GPU parity of the vocabulary CE's dHidden GEMM on 256 x 512 CTA-pair
tiles (the default), with dlogits taken from the CE core or formed inside
the GEMM, and on the 256 x 256 tiles it replaced.

"多卡张量：拆开计算，再合回同一结果", section 04 / VOCABULARY SHARDS:
dlogits = softmax - onehot and dHidden = sum over the vocabulary shards of
dlogits_r Whead_r^T.  With TPS_CE_GRAD_IN_GEMM the GEMM's A operand is the
logits GEMM's shifted bf16 logits, turned into the gradient in shared
memory as each tile arrives, and the passes over dHidden's first 512
columns write dlogits; the same formulas in the same order as the CE core,
so every output but dHidden must be bit-identical to the default path."""
import numpy as np
import pytest
import torch

from backward_tcgen05_tma_gemms_gb300 import api, inputs
from parity import assert_close
from test_gpu_ce import boundary_labels, run, spread_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["tiles", "grad"])
def wide(request, monkeypatch):
    """Wide tiles with dlogits from the CE core ("tiles"), or formed inside
    the dHidden GEMM ("grad")."""
    monkeypatch.setenv("TPS_CE_WIDE", "1")
    monkeypatch.setenv("TPS_CE_GRAD_IN_GEMM", "1" if request.param == "grad" else "0")
    return request.param


def launched(p, kind):
    return kind in {k.split(":")[0] for k in p.summary}


@pytest.mark.parametrize("ksplit", ["1", "3"])
@pytest.mark.parametrize("T,d,V,tp", [(600, 640, 5000, 4), (37, 512, 4096, 7), (300, 128, 16032, 8)])
def test_wide_matches_oracle(orc, wide, ksplit, T, d, V, tp, monkeypatch):
    """Ragged in every direction: 600 tokens leave a partial pair of row
    tiles, d = 640 a 128-column second tile, V = 5000 a last K tile of 8
    columns; with three K runs the runs are unequal and their partial tiles
    are added in order.  V = 16032 at tp = 8 puts the shard boundaries
    inside statistics tiles."""
    monkeypatch.setenv("TPS_CE_KSPLIT", ksplit)
    h, W, labels = inputs.ce_case(T + d + V, T, d, V, torch.bfloat16, w_std=0.2)
    with api.profile() as p:
        (loss, dlog, dh, own), rc = run(h, W, labels, tp)
    assert rc == 0
    assert launched(p, "ce_combine") == (wide == "grad"), p.summary
    rl, rdl, rdh, rown = orc.ce_tokens(inputs.as_f64(h), inputs.as_f64(W), labels.numpy(), tp)
    assert_close(loss, rl, True, f"{wide} loss")
    assert_close(dlog, rdl, True, f"{wide} dlogits")
    assert_close(dh, rdh, True, f"{wide} dHidden")
    assert np.array_equal(own.numpy(), rown)


@pytest.mark.parametrize("T,V,tp", [(300, 4096, 7), (513, 16032, 8)])
def test_grad_in_gemm_bits(T, V, tp, monkeypatch):
    """loss, dlogits and owner are bit-identical between the CE core and the
    in-GEMM gradient, and dHidden is bit-identical between the wide tiles
    fed by the CE core's dlogits and the wide tiles that form them (the same
    A values, K order and runs)."""
    h, W, labels = inputs.ce_case(T + V, T, 576, V, torch.bfloat16, w_std=0.2)
    base, rc0 = run(h, W, labels, tp)
    monkeypatch.setenv("TPS_CE_WIDE", "1")
    monkeypatch.setenv("TPS_CE_KSPLIT", "2")
    monkeypatch.setenv("TPS_CE_GRAD_IN_GEMM", "0")
    tiles, rc1 = run(h, W, labels, tp)
    monkeypatch.setenv("TPS_CE_GRAD_IN_GEMM", "1")
    grad, rc2 = run(h, W, labels, tp)
    assert rc0 == rc1 == rc2 == 0
    for i, name in ((0, "loss"), (1, "dlogits"), (3, "owner")):
        assert torch.equal(base[i], grad[i]), name
        assert torch.equal(tiles[i], grad[i]), name
    assert torch.equal(tiles[2], grad[2]), "dHidden"


@pytest.mark.parametrize("ksplit", ["1", "2"])
@pytest.mark.parametrize("T,d,V,tp", [(600, 640, 5000, 4), (300, 128, 16032, 8)])
def test_pair_tiles_match_oracle(orc, ksplit, T, d, V, tp, monkeypatch):
    """TPS_CE_WIDE=0: the dHidden GEMM on 256 x 256 CTA-pair tiles, the
    form the wide tiles replaced as the default."""
    monkeypatch.setenv("TPS_CE_WIDE", "0")
    monkeypatch.setenv("TPS_CE_KSPLIT", ksplit)
    h, W, labels = inputs.ce_case(T + d, T, d, V, torch.bfloat16, w_std=0.2)
    (loss, dlog, dh, own), rc = run(h, W, labels, tp)
    assert rc == 0
    rl, rdl, rdh, rown = orc.ce_tokens(inputs.as_f64(h), inputs.as_f64(W), labels.numpy(), tp)
    assert_close(loss, rl, True, "loss")
    assert_close(dlog, rdl, True, "dlogits")
    assert_close(dh, rdh, True, "dHidden")
    assert np.array_equal(own.numpy(), rown)


def test_grad_in_gemm_out_in_head(orc, monkeypatch):
    """The head in (V, d) layout: B of the dHidden GEMM is MN-major."""
    monkeypatch.setenv("TPS_CE_WIDE", "1")
    monkeypatch.setenv("TPS_CE_GRAD_IN_GEMM", "1")
    T, d, V, tp = 300, 640, 4096, 4
    h, W, labels = inputs.ce_case(3, T, d, V, torch.bfloat16, w_std=0.2)
    with api.profile() as p:
        (loss, dlog, dh, own), rc = run(h, W.t().contiguous(), labels, tp, "out_in")
    assert rc == 0 and launched(p, "ce_combine")
    rl, rdl, rdh, rown = orc.ce_tokens(inputs.as_f64(h), inputs.as_f64(W), labels.numpy(), tp)
    assert_close(loss, rl, True, "loss")
    assert_close(dlog, rdl, True, "dlogits")
    assert_close(dh, rdh, True, "dHidden")
    assert np.array_equal(own.numpy(), rown)


def test_grad_in_gemm_llama_sampled(orc, monkeypatch):
    """The Llama-3 vocabulary at full size (T=8192, d=4096, V=128256, tp=8)
    through the in-GEMM gradient, sampled like the default path: 64 tokens
    with labels at both ends of every shard, full dlogits and dHidden rows
    against the oracle."""
    monkeypatch.setenv("TPS_CE_WIDE", "1")
    monkeypatch.setenv("TPS_CE_GRAD_IN_GEMM", "1")
    cfg = inputs.LLAMA_CE
    T, V, tp = cfg["T"], cfg["V"], cfg["tp"]
    h, W, labels = inputs.ce_case(0, T, cfg["d"], V, torch.bfloat16)
    toks = spread_tokens(T, 64, 7)
    labels[torch.from_numpy(toks)] = torch.from_numpy(boundary_labels(V, tp))
    with api.profile() as p:
        (loss, dlog, dh, own), rc = run(h, W, labels, tp)
    assert rc == 0 and launched(p, "ce_combine")
    rl, rdl, rdh, rown = orc.ce_tokens(inputs.as_f64(h), inputs.as_f64(W), labels.numpy(), tp, toks)
    assert_close(loss[toks], rl, True, "loss")
    assert_close(dlog[toks], rdl, True, "dlogits")
    assert_close(dh[toks], rdh, True, "dHidden")
    assert np.array_equal(own[toks].numpy(), rown)
    assert torch.isfinite(loss).all()


@pytest.mark.parametrize("wide", ["1", "0"])
@pytest.mark.parametrize("ksplit", ["1", "2", "3"])
@pytest.mark.parametrize("T,d,V,tp", [(600, 640, 5000, 4), (2048, 1024, 16032, 8)])
def test_dynamic_schedule_bits(orc, wide, ksplit, T, d, V, tp, monkeypatch):
    """TPS_CE_DYNAMIC=1 (the default): the pairs take their (tile, K run)
    units in order from a counter instead of round-robin, on 256 x 512 and
    on 256 x 256 tiles.  Each unit computes the same sums in the same order,
    so every output is bit-identical to the static schedule, K split
    included; and it matches the oracle."""
    monkeypatch.setenv("TPS_CE_WIDE", wide)
    monkeypatch.setenv("TPS_CE_KSPLIT", ksplit)
    h, W, labels = inputs.ce_case(T + d + V, T, d, V, torch.bfloat16, w_std=0.2)
    monkeypatch.setenv("TPS_CE_DYNAMIC", "0")
    ref, rc0 = run(h, W, labels, tp)
    monkeypatch.setenv("TPS_CE_DYNAMIC", "1")
    got, rc1 = run(h, W, labels, tp)
    assert rc0 == rc1 == 0
    for x, y, name in zip(ref, got, ("loss", "dlogits", "dHidden", "owner")):
        assert torch.equal(x, y), name
    if T <= 600:
        rl, rdl, rdh, rown = orc.ce_tokens(inputs.as_f64(h), inputs.as_f64(W), labels.numpy(), tp)
        assert_close(got[2], rdh, True, "dHidden")


def test_llama_out_in_head_sampled(orc):
    """The Llama-3 vocabulary at full size with the head in (V, d) layout
    (torch's lm_head weight): the logits GEMM reads the head K-major and the
    wide dHidden GEMM reads it MN-major.  64 tokens with labels at both ends
    of every shard, full dlogits and dHidden rows against the oracle."""
    cfg = inputs.LLAMA_CE
    T, V, tp = cfg["T"], cfg["V"], cfg["tp"]
    h, W, labels = inputs.ce_case(0, T, cfg["d"], V, torch.bfloat16)
    toks = spread_tokens(T, 64, 11)
    labels[torch.from_numpy(toks)] = torch.from_numpy(boundary_labels(V, tp))
    (loss, dlog, dh, own), rc = run(h, W.t().contiguous(), labels, tp, "out_in")
    assert rc == 0
    rl, rdl, rdh, rown = orc.ce_tokens(inputs.as_f64(h), inputs.as_f64(W), labels.numpy(), tp, toks)
    assert_close(loss[toks], rl, True, "loss")
    assert_close(dlog[toks], rdl, True, "dlogits")
    assert_close(dh[toks], rdh, True, "dHidden")
    assert np.array_equal(own[toks].numpy(), rown)


@pytest.mark.parametrize("ksplit", [None, "3"])
def test_ragged_multiwave_sampled(orc, ksplit, monkeypatch):
    """T = 3000 (a partial pair of row tiles), d = 1536 (three 512-column
    tiles), V = 32000 at tp = 8 (500 K steps): 36 wide tiles, which the
    default K split turns into 72 (tile, run) units (one wave) and three
    runs into 108 (1.4 waves), taken in order; 48 sampled tokens against
    the oracle, including the last rows."""
    if ksplit:
        monkeypatch.setenv("TPS_CE_KSPLIT", ksplit)
    T, d, V, tp = 3000, 1536, 32000, 8
    h, W, labels = inputs.ce_case(17, T, d, V, torch.bfloat16, w_std=0.05)
    toks = spread_tokens(T, 48, 13)
    (loss, dlog, dh, own), rc = run(h, W, labels, tp)
    assert rc == 0
    rl, rdl, rdh, rown = orc.ce_tokens(inputs.as_f64(h), inputs.as_f64(W), labels.numpy(), tp, toks)
    assert_close(loss[toks], rl, True, "loss")
    assert_close(dlog[toks], rdl, True, "dlogits")
    assert_close(dh[toks], rdh, True, "dHidden")
    assert np.array_equal(own[toks].numpy(), rown)
