"""Pins for the oracle's attention projections and head-aligned plan (CPU
only).

"第 6 课：张量并行 TP", core concept 2.B (QKV projections column-parallel by
heads, W_O row-parallel, one sum) and core concept 3 item 4 (H divisible by
TP; GQA: Llama-3 8B, 32 query and 8 KV heads, at TP = 8 and TP = 16)."""
import json
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_lesson_head_counts(orc):
    g = json.load(open(os.path.join(GOLDEN, "tp_head_plan.json")))
    H, Hkv = g["n_heads"], g["n_kv_heads"]
    for c in g["cases"]:
        q_off, kv_first, kv_count, rep = orc.plan_heads(H, Hkv, c["tp"])
        assert set(np.diff(q_off)) == {c["q_heads_per_rank"]}
        assert kv_count == c["kv_heads_per_rank"]
        assert (rep == 1) == c["kv_divisible"]
        assert rep * c["tp"] * kv_count // rep == c["tp"] * kv_count   # every rank holds kv_count heads
        assert sorted(set(kv_first.tolist())) == list(range(0, Hkv, kv_count))


@pytest.mark.parametrize("H,Hkv", [(32, 8), (32, 32), (12, 4), (16, 1), (8, 2)])
def test_plan_invariants(orc, H, Hkv):
    """Brute force over TP: accepted exactly when H mod TP = 0 and the KV
    heads split or replicate evenly; then every query head has one owner,
    the ranks own equal contiguous head ranges, and each rank's query heads
    use only KV heads it holds (query head q uses KV head q // (H / Hkv))."""
    g = H // Hkv
    for tp in range(1, 2 * H + 2):
        ok = H % tp == 0 and (Hkv % tp == 0 or tp % Hkv == 0)
        if not ok:
            with pytest.raises(ValueError):
                orc.plan_heads(H, Hkv, tp)
            continue
        q_off, kv_first, kv_count, rep = orc.plan_heads(H, Hkv, tp)
        assert q_off[0] == 0 and q_off[-1] == H and len(set(np.diff(q_off))) == 1
        for r in range(tp):
            for q in range(q_off[r], q_off[r + 1]):
                assert kv_first[r] <= q // g < kv_first[r] + kv_count
        # each KV head is held by exactly `rep` ranks
        held = np.zeros(Hkv, dtype=int)
        for r in range(tp):
            held[kv_first[r]:kv_first[r] + kv_count] += 1
        assert (held == rep).all()


def test_uneven_heads_rejected(orc):
    with pytest.raises(ValueError):
        orc.plan_heads(32, 8, 3)       # 32 mod 3 != 0
    with pytest.raises(ValueError):
        orc.plan_heads(32, 8, 64)      # more ranks than heads
    with pytest.raises(ValueError):
        orc.plan_heads(30, 4, 2)       # a query group split across KV heads


def rand(seed, shapes):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal(s) for s in shapes]


def test_qkv_against_autograd(orc):
    T, d, nq, nkv = 7, 12, 16, 8
    X, Wq, Wk, Wv, dQ, dK, dV = rand(1, [(T, d), (d, nq), (d, nkv), (d, nkv), (T, nq), (T, nkv), (T, nkv)])
    tX, tWq, tWk, tWv = (torch.tensor(a, requires_grad=True) for a in (X, Wq, Wk, Wv))
    Q, K, V = tX @ tWq, tX @ tWk, tX @ tWv
    ((Q * torch.tensor(dQ)).sum() + (K * torch.tensor(dK)).sum() + (V * torch.tensor(dV)).sum()).backward()
    got = orc.attn_qkv(X, Wq, Wk, Wv, dQ, dK, dV)
    ref = [Q.detach().numpy(), K.detach().numpy(), V.detach().numpy(), tX.grad.numpy(), tWq.grad.numpy(),
           tWk.grad.numpy(), tWv.grad.numpy()]
    for name, a, b in zip(["Q", "K", "V", "dX", "dWq", "dWk", "dWv"], got, ref):
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(b).max()), name


def test_out_against_autograd(orc):
    T, d, nq = 9, 10, 12
    C, Wo, G = rand(2, [(T, nq), (nq, d), (T, d)])
    tC, tWo = torch.tensor(C, requires_grad=True), torch.tensor(Wo, requires_grad=True)
    Y = tC @ tWo
    (Y * torch.tensor(G)).sum().backward()
    Yo, dC, dWo = orc.attn_out(C, Wo, G)
    for a, b in [(Yo, Y.detach().numpy()), (dC, tC.grad.numpy()), (dWo, tWo.grad.numpy())]:
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(b).max())


def test_finite_differences(orc):
    """L = <dQ, Q> + <dK, K> + <dV, V> is linear in each weight and in X."""
    T, d, nq, nkv = 4, 5, 6, 4
    X, Wq, Wk, Wv, dQ, dK, dV = rand(3, [(T, d), (d, nq), (d, nkv), (d, nkv), (T, nq), (T, nkv), (T, nkv)])
    _, _, _, dX, dWq, dWk, dWv = orc.attn_qkv(X, Wq, Wk, Wv, dQ, dK, dV)

    def L(x, wq, wk, wv):
        q, k, v = orc.attn_qkv(x, wq, wk, wv, dQ, dK, dV)[:3]
        return float((q * dQ).sum() + (k * dK).sum() + (v * dV).sum())
    base = [X, Wq, Wk, Wv]
    h = 1e-6
    for i, grad in enumerate([dX, dWq, dWk, dWv]):
        for idx in [(0, 0), (base[i].shape[0] - 1, base[i].shape[1] - 1), (1, 2)]:
            E = np.zeros_like(base[i]); E[idx] = 1.0
            p, m = list(base), list(base)
            p[i], m[i] = base[i] + h * E, base[i] - h * E
            fd = (L(*p) - L(*m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (i, idx)


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
def test_head_sharded_equals_unsharded(orc, tp):
    """Each rank projects its own heads' columns (Q heads by the plan, KV
    heads possibly replicated) and multiplies its context columns by its
    rows of W_O; the rank outputs are summed once."""
    H, Hkv, dh, T, d = 8, 2, 4, 5, 12
    nq, nkv = H * dh, Hkv * dh
    X, Wq, Wk, Wv, C, Wo, G = rand(4, [(T, d), (d, nq), (d, nkv), (d, nkv), (T, nq), (nq, d), (T, d)])
    zq, zk = np.zeros((T, nq)), np.zeros((T, nkv))
    Q, K, V = orc.attn_qkv(X, Wq, Wk, Wv, zq, zk, zk)[:3]
    Y = orc.attn_out(C, Wo, G)[0]
    q_off, kv_first, kv_count, rep = orc.plan_heads(H, Hkv, tp)
    Ysum = 0
    for r in range(tp):
        qc = slice(q_off[r] * dh, q_off[r + 1] * dh)
        kc = slice(kv_first[r] * dh, (kv_first[r] + kv_count) * dh)
        np.testing.assert_allclose(X @ Wq[:, qc], Q[:, qc], rtol=0, atol=1e-12)
        np.testing.assert_allclose(X @ Wk[:, kc], K[:, kc], rtol=0, atol=1e-12)
        np.testing.assert_allclose(X @ Wv[:, kc], V[:, kc], rtol=0, atol=1e-12)
        Ysum = Ysum + C[:, qc] @ Wo[qc, :]
    assert np.abs(Ysum - Y).max() <= 1e-12 * np.abs(Y).max()
