"""GPU parity of the attention projections (tps_attn_qkv_fwd,
tps_attn_qkv_bwd, tps_attn_out_fwd_bwd) against the float64 oracle.

"第 6 课：张量并行 TP", core concept 2.B (QKV column-parallel by heads, W_O
row-parallel, one sum) and core concept 3 item 4 (heads divisible by TP;
GQA with KV heads split or replicated)."""
import numpy as np
import pytest
import torch

from backward_tcgen05_tma_gemms_gb300 import api, inputs
from parity import assert_close

pytestmark = pytest.mark.gpu


def io(W, layout):
    w = inputs.as_f64(W)
    return w if layout == "in_out" else w.T


def check(orc, c, H, Hkv, tp, layout, bf16, what):
    g = {k: v.cuda() for k, v in c.items()}
    Q, K, V = api.attn_qkv_fwd(g["X"], g["Wq"], g["Wk"], g["Wv"], H, Hkv, tp, layout, out_dtype=torch.float32)
    dX, dWq, dWk, dWv = api.attn_qkv_bwd(g["X"], g["Wq"], g["Wk"], g["Wv"], g["dQ"], g["dK"], g["dV"], H, Hkv, tp,
                                         layout)
    Y, dC, dWo = api.attn_out_fwd_bwd(g["C"], g["Wo"], g["GY"], H, tp, layout, dC_dtype=torch.float32)
    assert api.last_device_error() == 0
    f = {k: inputs.as_f64(v) for k, v in c.items()}
    ref = orc.attn_qkv(f["X"], io(c["Wq"], layout), io(c["Wk"], layout), io(c["Wv"], layout), f["dQ"], f["dK"],
                       f["dV"])
    rY, rdC, rdWo = orc.attn_out(f["C"], io(c["Wo"], layout), f["GY"])
    tr = (lambda a: a) if layout == "in_out" else (lambda a: a.T)
    got = [Q, K, V, dX, dWq, dWk, dWv, Y, dC, dWo]
    want = list(ref[:4]) + [tr(ref[4]), tr(ref[5]), tr(ref[6]), rY, rdC, tr(rdWo)]
    for name, a, b in zip(["Q", "K", "V", "dX", "dWq", "dWk", "dWv", "Y", "dC", "dWo"], got, want):
        assert_close(a.cpu(), b, bf16, f"{what} {name}")


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
def test_fp32_kv_split_and_replicated(orc, tp):
    """H=8, H_kv=2: KV heads split at tp=1, 2 and replicated at tp=4, 8."""
    c = inputs.attn_case(tp, 37, 48, 8, 2, 16, torch.float32, w_std=0.2)
    check(orc, c, 8, 2, tp, "in_out", False, f"tp{tp}")


@pytest.mark.parametrize("layout", ["in_out", "out_in"])
def test_bf16_fused_qkv(orc, layout):
    """Head boundaries on 128-column blocks: Q, K and V in one launch, and
    with (in, out) gradients dWq, dWk, dWv in one launch too."""
    c = inputs.attn_case(3, 300, 256, 8, 2, 64, torch.bfloat16, w_std=0.05, layout=layout)
    with api.profile() as p:
        check(orc, c, 8, 2, 4, layout, True, f"bf16 {layout}")
    assert p.summary["gemm_tc:attn_qkv"]["launches"] == 1, p.summary
    if layout == "in_out":
        assert p.summary["gemm_tc:attn_dWqkv"]["launches"] == 1, p.summary
    else:
        assert all(f"gemm_tc:attn_dW{x}" in p.summary for x in "qkv"), p.summary
    assert {k.split(":")[0] for k in p.summary} == {"gemm_tc"}, p.summary


def test_bf16_unaligned_heads(orc):
    """dh=40: the K block starts at column 160, inside a 128-column block,
    so the three projections run as separate GEMMs."""
    c = inputs.attn_case(4, 129, 128, 4, 2, 40, torch.bfloat16, w_std=0.05)
    with api.profile() as p:
        check(orc, c, 4, 2, 2, "in_out", True, "dh40")
    assert "gemm_tc:attn_qkv" in p.summary and p.summary["gemm_tc:attn_qkv"]["launches"] == 3, p.summary
    assert p.summary["gemm_tc:attn_dWqkv"]["launches"] == 3, p.summary


def test_head_rules_enforced():
    c = {k: v.cuda() for k, v in inputs.attn_case(5, 8, 32, 6, 2, 8, torch.float32).items()}
    with pytest.raises(ValueError, match="partition"):
        api.attn_qkv_fwd(c["X"], c["Wq"], c["Wk"], c["Wv"], 6, 2, 4, "in_out")      # 6 heads over tp=4
    with pytest.raises(ValueError, match="partition"):
        api.attn_out_fwd_bwd(c["C"], c["Wo"], c["GY"], 6, 4)


def test_llama_shape_sampled(orc):
    """Llama-3-8B attention projections (T=8192, d=4096, 32 query and 8 KV
    heads of 128, tp=8, bf16) at full size: 6 token rows of Q, K, V, dX
    and Y, and 6 columns of each weight gradient, recomputed by the oracle
    from the corresponding rows and columns of the inputs."""
    cfg = inputs.LLAMA_ATTN
    H, Hkv, tp = cfg["H"], cfg["Hkv"], cfg["tp"]
    c = inputs.attn_case(0, cfg["T"], cfg["d"], H, Hkv, cfg["dh"], torch.bfloat16)
    g = {k: v.cuda() for k, v in c.items()}
    Q, K, V = api.attn_qkv_fwd(g["X"], g["Wq"], g["Wk"], g["Wv"], H, Hkv, tp, out_dtype=torch.float32)
    dX, dWq, dWk, dWv = api.attn_qkv_bwd(g["X"], g["Wq"], g["Wk"], g["Wv"], g["dQ"], g["dK"], g["dV"], H, Hkv, tp)
    Y, dC, dWo = api.attn_out_fwd_bwd(g["C"], g["Wo"], g["GY"], H, tp, dC_dtype=torch.float32)
    assert api.last_device_error() == 0
    f = {k: inputs.as_f64(v) for k, v in c.items()}
    rows = np.array([0, 1, 2047, 4096, 6000, 8191])
    rq, rk, rv, rdx, _, _, _ = orc.attn_qkv(f["X"][rows], f["Wq"], f["Wk"], f["Wv"], f["dQ"][rows], f["dK"][rows],
                                            f["dV"][rows])
    ry, rdc, _ = orc.attn_out(f["C"][rows], f["Wo"], f["GY"][rows])
    for name, a, b in [("Q", Q, rq), ("K", K, rk), ("V", V, rv), ("dX", dX, rdx), ("Y", Y, ry), ("dC", dC, rdc)]:
        assert_close(a[rows].cpu(), b, True, f"{name} rows")
    qc = np.array([0, 511, 512, 2048, 4000, 4095])        # spread over ranks' head ranges
    kc = np.array([0, 127, 128, 512, 900, 1023])
    _, _, _, _, rdwq, rdwk, rdwv = orc.attn_qkv(f["X"], f["Wq"][:, qc], f["Wk"][:, kc], f["Wv"][:, kc],
                                                f["dQ"][:, qc], f["dK"][:, kc], f["dV"][:, kc])
    assert_close(dWq[:, qc].cpu(), rdwq, True, "dWq cols")
    assert_close(dWk[:, kc].cpu(), rdwk, True, "dWk cols")
    assert_close(dWv[:, kc].cpu(), rdwv, True, "dWv cols")
    _, _, rdwo = orc.attn_out(f["C"][:, qc], f["Wo"][qc], f["GY"])
    assert_close(dWo[qc].cpu(), rdwo, True, "dWo rows")


@pytest.mark.parametrize("T", [0, 3])
def test_bf16_few_tokens(orc, T):
    c = inputs.attn_case(40 + T, max(T, 1), 128, 4, 2, 64, torch.bfloat16, w_std=0.1)
    for k in ("X", "dQ", "dK", "dV", "C", "GY"):
        c[k] = c[k][:T].contiguous()
    check(orc, c, 4, 2, 2, "in_out", True, f"T={T}")
