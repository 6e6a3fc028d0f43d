"""GPU parity of tps_vocab_ce_fwd_bwd against the float64 oracle.

"多卡张量：拆开计算，再合回同一结果", section 04 / VOCABULARY SHARDS: per-shard
max and sum-exp combined into one log-sum-exp, loss, dlogits = softmax -
onehot, dHidden summed over the vocabulary shards; the owner rank of each
label is compared bit-exactly."""
import json
import math
import os

import numpy as np
import pytest
import torch

from backward_tcgen05_tma_gemms_gb300 import api, inputs
from parity import assert_close

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run(h, W, labels, tp, layout="in_out"):
    out = api.vocab_ce_fwd_bwd(h.cuda(), W.cuda(), labels.cuda(), tp, layout)
    rc = api.last_device_error()
    return [t.cpu() for t in out], rc


def check(orc, h, W, labels, tp, bf16, layout="in_out", what=""):
    (loss, dlog, dh, own), rc = run(h, W, labels, tp, layout)
    assert rc == 0
    w = inputs.as_f64(W) if layout == "in_out" else inputs.as_f64(W).T
    rl, rdl, rdh, rown = orc.ce_tokens(inputs.as_f64(h), w, labels.numpy(), tp)
    assert_close(loss, rl, bf16, f"{what} loss")
    assert_close(dlog, rdl, bf16, f"{what} dlogits")
    assert_close(dh, rdh, bf16, f"{what} dHidden")
    assert np.array_equal(own.numpy(), rown), f"{what} owner"


def test_worked_logits(orc):
    z = json.load(open(os.path.join(GOLDEN, "ce_worked_logits.json")))["logits"]
    h = torch.tensor([z] * 6, dtype=torch.float32)
    W = torch.eye(6)
    labels = torch.arange(6)
    for tp in (1, 2, 3, 7):
        (loss, dlog, dh, own), rc = run(h, W, labels, tp)
        assert rc == 0
        den = sum(math.exp(v) for v in z)
        for y in range(6):
            assert abs(loss[y].item() - (math.log(den) - z[y])) < 1e-5
            p = np.array([math.exp(v) / den for v in z])
            assert np.abs(dlog[y].numpy() - (p - np.eye(6)[y])).max() < 1e-6
        off = api.plan_shards(6, tp)
        assert [int(v) for v in own] == [next(r for r in range(tp) if off[r] <= y < off[r + 1]) for y in range(6)]


@pytest.mark.parametrize("tp", [1, 3, 7, 8])
def test_fp32_cluster_path(orc, tp):
    h, W, labels = inputs.ce_case(tp, 37, 48, 1000, torch.float32, w_std=0.5)
    check(orc, h, W, labels, tp, False, what=f"tp{tp}")


@pytest.mark.parametrize("tp,V,T", [(3, 1001, 23), (2, 40000, 9), (8, 1000, 300), (5, 16380 * 5, 11)])
def test_fp32_cluster_variants(orc, tp, V, T):
    """Logits rows not 16-byte aligned (register kernel), shards above the
    register capacity (shared-memory kernel), many tokens per persistent
    cluster (ring wrap-around), shards at the persistent kernel's limit."""
    h, W, labels = inputs.ce_case(tp * 31 + V, T, 12, V, torch.float32, w_std=0.5)
    check(orc, h, W, labels, tp, False, what=f"tp{tp} V{V} T{T}")


@pytest.mark.parametrize("tp,V", [(9, 1000), (16, 5003), (1, 100000)])
def test_fp32_two_pass_path(orc, tp, V):
    """More ranks than a cluster holds, or a shard larger than shared memory."""
    h, W, labels = inputs.ce_case(tp + V, 5, 16, V, torch.float32, w_std=0.5)
    check(orc, h, W, labels, tp, False, what=f"tp{tp} V{V}")


def test_fp32_empty_shards(orc):
    h, W, labels = inputs.ce_case(3, 6, 8, 5, torch.float32, w_std=1.0)
    check(orc, h, W, labels, 8, False, what="tp8 V5")       # three empty shards


@pytest.mark.parametrize("tp", [8, 7])
@pytest.mark.parametrize("layout", ["in_out", "out_in"])
def test_bf16_tensor_core(orc, tp, layout, gemm_kernel):
    h, W, labels = inputs.ce_case(40 + tp, 200, 256, 32000, torch.bfloat16)
    if layout == "out_in":
        W = W.t().contiguous()
    with api.profile() as p:
        check(orc, h, W, labels, tp, True, layout, what=f"bf16 tp{tp} {layout}")
    kinds = {k.split(":")[0] for k in p.summary}
    assert kinds == {"gemm_tc", "ce_stream"}, p.summary   # statistics from the logits epilogue


@pytest.mark.parametrize("tp,V,T", [(8, 4096, 130), (3, 2048 + 768, 64), (2, 520, 33), (8, 1000, 50), (1, 32768, 17)])
def test_bf16_shard_layouts(orc, tp, V, T, gemm_kernel):
    """Shard boundaries on and off the 256-column tile edges, shards of
    exactly one tile, a ragged last tile, and shards narrower than a tile
    (which take the cluster kernel instead of the epilogue statistics)."""
    h, W, labels = inputs.ce_case(tp * 7 + V, T, 64, V, torch.bfloat16, w_std=0.1)
    with api.profile() as p:
        check(orc, h, W, labels, tp, True, what=f"bf16 tp{tp} V{V}")
    kinds = {k.split(":")[0] for k in p.summary}
    expect = "ce_stream" if V // tp >= 256 else "ce_cluster"
    assert expect in kinds, p.summary


@pytest.mark.parametrize("T", [64, 300])
def test_bf16_large_logits(orc, T, gemm_kernel):
    """Logits up to ~240 in magnitude (weights of std 3 on d = 256).  The
    fused path keeps the logits in bf16 relative to the max of their
    128-column tile, which holds the softmax weights near each max to fp32
    level (a float64 simulation of that storage: relative Frobenius error
    of dlogits 3e-6 to 3e-5).  bf16 logits without the shift are rounded by
    up to 2^-8 |z| (about 0.9 here) inside the exponent, and the same
    simulation puts their dlogits 1.5-3.4 % off, beyond the tolerance."""
    h, W, labels = inputs.ce_case(1234 + T, T, 256, 4096, torch.bfloat16, w_std=3.0)
    with api.profile() as p:
        check(orc, h, W, labels, 4, True, what=f"bf16 large logits T{T}")
    assert "ce_stream" in {k.split(":")[0] for k in p.summary}, p.summary


def test_label_out_of_range_sets_error():
    h, W, labels = inputs.ce_case(1, 4, 16, 64, torch.float32)
    labels[2] = 64
    (loss, dlog, dh, own), rc = run(h, W, labels, 4)
    assert rc == api.ERR_LABEL
    assert torch.isnan(loss[2]) and own[2] == -1
    assert torch.isfinite(loss[[0, 1, 3]]).all()
    assert api.last_device_error() == 0     # the word was cleared


def boundary_labels(V, tp, vreal=None):
    """Eight labels per rank: four at the first columns of its shard and
    four at its last (real) columns.  At V = 128256, tp = 8 the shards start
    at multiples of 16032 = 125 x 128 + 32, so each shard's first 96
    columns share a 128-column statistics tile with the previous shard: the
    labels there read their logit from a tile whose statistics are split
    between two shards."""
    off = api.plan_shards(V, tp)
    vr = V if vreal is None else vreal
    labs = []
    for r in range(tp):
        lo, hi = off[r], min(off[r + 1], vr)
        labs += [lo, lo + 1, lo + 31, lo + 95, hi - 96, hi - 33, hi - 2, hi - 1]
    return np.array(labs, dtype=np.int64)


def spread_tokens(T, n, seed, avoid_mod=None):
    """n distinct tokens spread over [0, T) including the first and last
    (optionally none that are multiples of avoid_mod)."""
    rng = np.random.default_rng(seed)
    pool = np.arange(1, T - 1)
    if avoid_mod:
        pool = pool[pool % avoid_mod != 0]
    toks = np.concatenate([[0 if not avoid_mod else 1, T - 1], rng.choice(pool, n - 2, replace=False)])
    return np.sort(toks)


def test_llama_vocab_sampled(orc):
    """h 8192 x 4096, head 4096 x 128256, tp=8 (16032 per shard), bf16, at
    full size in the benchmark's launch configuration.  64 tokens spread
    over the batch get labels at both ends of every shard (each rank owns
    eight), and the oracle recomputes their loss, full dlogits row and
    dHidden row; every owner rank of the batch is checked against a host
    scan."""
    cfg = inputs.LLAMA_CE
    T, V, tp = cfg["T"], cfg["V"], cfg["tp"]
    h, W, labels = inputs.ce_case(0, T, cfg["d"], V, torch.bfloat16)
    toks = spread_tokens(T, 64, 5)
    labels[torch.from_numpy(toks)] = torch.from_numpy(boundary_labels(V, tp))
    (loss, dlog, dh, own), rc = run(h, W, labels, tp)
    assert rc == 0
    rl, rdl, rdh, rown = orc.ce_tokens(inputs.as_f64(h), inputs.as_f64(W), labels.numpy(), tp, toks)
    assert_close(loss[toks], rl, True, "loss")
    assert_close(dlog[toks], rdl, True, "dlogits")
    assert_close(dh[toks], rdh, True, "dHidden")
    assert np.array_equal(own[toks].numpy(), rown)
    assert np.bincount(rown, minlength=tp).min() >= 4
    off = np.array(api.plan_shards(V, tp))
    assert np.array_equal(own.numpy(), np.searchsorted(off, labels.numpy(), side="right") - 1)
    assert torch.isfinite(loss).all()
    # mean loss near log V + var(z)/2 with var(z) = d * 0.02^2
    assert abs(loss.mean().item() - (math.log(V) + cfg["d"] * 0.02 ** 2 / 2)) < 0.1


def test_bf16_int32_labels_match_int64(gemm_kernel):
    """The logits epilogue reads each row's label to keep its fp32 logit;
    int32 labels give bit-identical results to the same labels as int64."""
    h, W, labels = inputs.ce_case(77, 300, 128, 4096, torch.bfloat16, w_std=0.2)
    a, rc_a = run(h, W, labels, 4)
    b, rc_b = run(h, W, labels.to(torch.int32), 4)
    assert rc_a == 0 and rc_b == 0
    for x, y, name in zip(a, b, ("loss", "dlogits", "dHidden", "owner")):
        assert torch.equal(x, y), name


@pytest.mark.parametrize("T", [37, 300])
def test_bf16_unaligned_vocab_rows(orc, T, gemm_kernel):
    """V = 4100: rows of bf16 logits and dlogits are 8200 B, not a multiple
    of 16, so the logits epilogue stores without TMA and the gradient
    stream takes its scalar path; the head in (V, d) layout keeps the GEMM
    operands TMA-compatible.  Shards of 2050 columns straddle tiles."""
    h, W, labels = inputs.ce_case(4100 + T, T, 128, 4100, torch.bfloat16, w_std=0.2)
    W = W.t().contiguous()
    with api.profile() as p:
        check(orc, h, W, labels, 2, True, "out_in", what=f"bf16 V4100 T{T}")
    assert "ce_stream" in {k.split(":")[0] for k in p.summary}, p.summary


@pytest.mark.parametrize("T,V,tp", [(300, 4096, 7), (513, 16032, 8)])
def test_fused_core_matches_two_kernels(T, V, tp, monkeypatch):
    """The fused CE core (per-shard combine and gradient stream in one
    kernel, logits bulk-copied into shared memory) and the two-kernel form
    (combine kernel, then streaming kernel) evaluate the same formulas in
    the same order: identical bits, shard boundaries inside tiles included
    (16032 / 8 = 2004 = 15 x 128 + 84)."""
    h, W, labels = inputs.ce_case(T + V, T, 64, V, torch.bfloat16, w_std=0.2)
    n0 = api.launch_count()
    a, rc_a = run(h, W, labels, tp)
    fused_launches = api.launch_count() - n0
    monkeypatch.setenv("TPS_CE_TWO_KERNELS", "1")
    n0 = api.launch_count()
    b, rc_b = run(h, W, labels, tp)
    assert api.launch_count() - n0 == fused_launches + 1   # logits GEMM, CE core, dHidden GEMM
    assert rc_a == 0 and rc_b == 0
    for x, y, name in zip(a, b, ("loss", "dlogits", "dHidden", "owner")):
        assert torch.equal(x, y), name


@pytest.mark.parametrize("ksplit", ["1", "3", "4"])
def test_dhidden_k_split(orc, ksplit, monkeypatch):
    """dHidden = dlogits Whead^T with its K (the vocabulary) cut into runs
    of K tiles, each run's partial tile added into dHidden in run order by
    TMA reductions once the previous run of the same tile is in memory
    (the default is two runs).  V = 5000 gives 79 K tiles, so three and
    four runs are unequal, and 600 tokens leave a ragged last pair tile.
    Every run count matches the oracle, and two calls give identical bits:
    the order of the partial sums is fixed."""
    monkeypatch.setenv("TPS_CE_KSPLIT", ksplit)
    h, W, labels = inputs.ce_case(11, 600, 256, 5000, torch.bfloat16, w_std=0.2)
    check(orc, h, W, labels, 4, True, what=f"{ksplit} runs")
    a, rc_a = run(h, W, labels, 4)
    b, rc_b = run(h, W, labels, 4)
    assert rc_a == 0 and rc_b == 0
    assert torch.equal(a[2], b[2])
