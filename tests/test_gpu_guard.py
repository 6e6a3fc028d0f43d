"""Guard bands around every output and workspace (the sanitizer's stand-in).

Each output and workspace of an entry point is a view inside a larger
buffer filled with a canary byte: 4 KB before and after it, and for 2-D
outputs also a few elements past the end of every row (a row pitch wider
than the row).  The calls run at ragged shapes -- tiles cut by M, N and K,
T = 37 tokens, V = 4100 columns, shards of 7 ranks -- and afterwards every
canary byte must be unchanged, so a store past the end of a tile, a row or
a workspace region shows up here.  The results must also be bit-identical
to the same call on plain torch tensors of the same strides (an output's
pitch can decide which kernel later reads it, as dlogits feeds dHidden)."""
import pytest
import torch

from backward_tcgen05_tma_gemms_gb300 import api, inputs

pytestmark = pytest.mark.gpu

PAD = 4096      # canary bytes before and after each buffer
CANARY = 0xA5


class Guarded:
    """A tensor of `shape` and `dtype` inside a canary-filled buffer.  A 2-D
    tensor gets a row pitch `gap` elements wider than its width, rounded up
    to a 16-byte multiple so that the tensor-core kernels still store it
    with TMA."""

    def __init__(self, name, shape, dtype, gap=3):
        self.name, self.shape, self.dtype = name, tuple(shape), dtype
        self.esz = torch.empty((), dtype=dtype).element_size()
        if len(shape) == 2 and gap:
            rows, cols = shape
            per16 = 16 // self.esz
            self.pitch = (cols + gap + per16 - 1) // per16 * per16
            n = rows * self.pitch
        else:
            self.pitch = None
            n = 1
            for v in shape:
                n *= v
        self.n = n
        self.raw = torch.full((PAD + n * self.esz + PAD,), CANARY, dtype=torch.uint8, device="cuda")
        flat = self.raw[PAD:PAD + n * self.esz].view(dtype)
        if self.pitch is not None:
            self.t = flat.view(shape[0], self.pitch)[:, :shape[1]]
        else:
            self.t = flat.view(self.shape)

    def check(self):
        raw = self.raw.cpu()
        keep = torch.ones(raw.numel(), dtype=torch.bool)
        if self.pitch is not None:
            rows, cols = self.shape
            r = torch.arange(rows).unsqueeze(1) * (self.pitch * self.esz)
            c = torch.arange(cols * self.esz).unsqueeze(0)
            keep[(PAD + r + c).flatten()] = False
        else:
            keep[PAD:PAD + self.n * self.esz] = False
        bad = torch.nonzero(raw[keep] != CANARY).flatten()
        assert bad.numel() == 0, f"{self.name}: {bad.numel()} canary bytes overwritten"


def guard(*specs):
    return [Guarded(*s) for s in specs]


def plain(guards):
    """Unguarded tensors with the guarded ones' shapes and strides."""
    return [torch.empty_strided(g.t.size(), g.t.stride(), dtype=g.dtype, device="cuda") for g in guards]


def check_all(guards, refs):
    torch.cuda.synchronize()
    assert api.last_device_error() == 0
    for g in guards:
        g.check()
    for g, r in zip(guards, refs):
        if r is not None:
            assert torch.equal(g.t, r), f"{g.name}: differs from the unguarded call"


def workspace(name, nbytes):
    return Guarded(name, (max(nbytes, 1),), torch.uint8, gap=0)


MATMUL = [((300, 200, 520), torch.bfloat16), ((257, 1000, 136), torch.bfloat16), ((1, 64, 8), torch.bfloat16),
          ((4808, 384, 712), torch.bfloat16), ((37, 45, 53), torch.float32)]


@pytest.mark.parametrize("shape,dtype", MATMUL)
@pytest.mark.parametrize("axis,parts", [("inner", 7), ("rows", 3), ("columns", 7)])
def test_matmul_guard(shape, dtype, axis, parts, gemm_kernel):
    M, K, N = shape
    A, B, G = (t.cuda() for t in inputs.matmul_case(M + K + N, M, K, N, dtype))
    gs = guard(("Y", (M, N), torch.float32), ("dA", (M, K), torch.float32), ("dB", (K, N), torch.float32))
    refs = api.matmul_fwd_bwd(A, B, G, parts, axis, out=plain(gs))
    api.matmul_fwd_bwd(A, B, G, parts, axis, out=[g.t for g in gs])
    check_all(gs, refs)


@pytest.mark.parametrize("T,d,F", [(37, 136, 712), (300, 200, 520)])
def test_mlp_guard(T, d, F, gemm_kernel):
    X, W1, W2, GY = (t.cuda() for t in inputs.mlp_case(T + F, T, d, F, torch.bfloat16, w_std=0.05))
    gs = guard(("Y", (T, d), torch.float32), ("dX", (T, d), torch.float32), ("dW1", (d, F), torch.float32),
               ("dW2", (F, d), torch.float32))
    refs = api.mlp_fwd_bwd(X, W1, W2, GY, 7, "gelu_tanh", "in_out", out=plain(gs))
    ws = workspace("mlp workspace", api.mlp_workspace_bytes(T, d, F, 7, torch.bfloat16))
    api.mlp_fwd_bwd(X, W1, W2, GY, 7, "gelu_tanh", "in_out", workspace=ws.t, out=[g.t for g in gs])
    check_all(gs + [ws], list(refs) + [None])


def test_mlp_noalloc_outputs_guard():
    T, d, F = 300, 200, 520
    X, W1, W2, GY = (t.cuda() for t in inputs.mlp_case(3, T, d, F, torch.bfloat16, w_std=0.05))
    gs = guard(("Y", (T, d), torch.float32), ("dX", (T, d), torch.float32), ("dW1", (d, F), torch.float32),
               ("dW2", (F, d), torch.float32))
    refs = api.mlp_fwd_bwd(X, W1, W2, GY, 7, "silu", "in_out", out=plain(gs))
    api.mlp_fwd_bwd_noalloc(X, W1, W2, GY, 7, "silu", "in_out", out=[g.t for g in gs])
    check_all(gs, refs)


@pytest.mark.parametrize("T,d,F", [(37, 136, 712), (300, 200, 520)])
def test_glu_guard(T, d, F):
    X, Wg, Wu, W2, GY = (t.cuda() for t in inputs.glu_case(T + d, T, d, F, torch.bfloat16, w_std=0.05))
    gs = guard(("Y", (T, d), torch.float32), ("dX", (T, d), torch.float32), ("dWg", (d, F), torch.float32),
               ("dWu", (d, F), torch.float32), ("dW2", (F, d), torch.float32))
    refs = api.glu_mlp_fwd_bwd(X, Wg, Wu, W2, GY, 7, "silu", out=plain(gs))
    ws = workspace("glu workspace", api.glu_mlp_workspace_bytes(T, d, F, 7, torch.bfloat16))
    api.glu_mlp_fwd_bwd(X, Wg, Wu, W2, GY, 7, "silu", workspace=ws.t, out=[g.t for g in gs])
    check_all(gs + [ws], list(refs) + [None])


@pytest.mark.parametrize("T", [37, 300])
def test_attention_guard(T):
    d, H, Hkv, dh, tp = 136, 4, 2, 64, 2
    c = {k: v.cuda() for k, v in inputs.attn_case(T, T, d, H, Hkv, dh, torch.bfloat16, w_std=0.05).items()}
    nq, nkv = H * dh, Hkv * dh
    g_qkv = guard(("Q", (T, nq), torch.bfloat16), ("K", (T, nkv), torch.bfloat16), ("V", (T, nkv), torch.bfloat16))
    g_bwd = guard(("dX", (T, d), torch.float32), ("dWq", (d, nq), torch.float32), ("dWk", (d, nkv), torch.float32),
                  ("dWv", (d, nkv), torch.float32))
    g_out = guard(("Y", (T, d), torch.float32), ("dC", (T, nq), torch.bfloat16), ("dWo", (nq, d), torch.float32))
    ref_qkv = api.attn_qkv_fwd(c["X"], c["Wq"], c["Wk"], c["Wv"], H, Hkv, tp, out=plain(g_qkv))
    ref_bwd = api.attn_qkv_bwd(c["X"], c["Wq"], c["Wk"], c["Wv"], c["dQ"], c["dK"], c["dV"], H, Hkv, tp,
                               out=plain(g_bwd))
    ref_out = api.attn_out_fwd_bwd(c["C"], c["Wo"], c["GY"], H, tp, out=plain(g_out))
    api.attn_qkv_fwd(c["X"], c["Wq"], c["Wk"], c["Wv"], H, Hkv, tp, out=[g.t for g in g_qkv])
    api.attn_qkv_bwd(c["X"], c["Wq"], c["Wk"], c["Wv"], c["dQ"], c["dK"], c["dV"], H, Hkv, tp,
                     out=[g.t for g in g_bwd])
    api.attn_out_fwd_bwd(c["C"], c["Wo"], c["GY"], H, tp, out=[g.t for g in g_out])
    check_all(g_qkv + g_bwd + g_out, list(ref_qkv) + list(ref_bwd) + list(ref_out))


CE_CASES = [  # (T, d, V, tp, layout, dtype): the paths of the cross-entropy
    (37, 128, 4100, 7, "in_out", torch.bfloat16),    # head rows not 16-byte multiples: fp32 logits, cluster kernel
    (37, 128, 4100, 7, "out_in", torch.bfloat16),    # tensor cores, logits rows not 16-byte aligned: two kernels
    (300, 128, 4096, 7, "in_out", torch.bfloat16),   # tensor cores, fused CE core, shards straddling tiles
    (37, 48, 1000, 7, "in_out", torch.float32),      # fp32 operands
]


@pytest.mark.parametrize("T,d,V,tp,layout,dtype", CE_CASES)
def test_ce_guard(T, d, V, tp, layout, dtype):
    h, W, labels = inputs.ce_case(T + V, T, d, V, dtype, w_std=0.2)
    if layout == "out_in":
        W = W.t().contiguous()
    h, W, labels = h.cuda(), W.cuda(), labels.cuda()
    gs = guard(("loss", (T,), torch.float32), ("dlogits", (T, V), dtype), ("dHidden", (T, d), torch.float32),
               ("owner", (T,), torch.int32))
    refs = api.vocab_ce_fwd_bwd(h, W, labels, tp, layout, out=plain(gs))
    # the workspace the call's path needs (the bf16-logit size where that applies)
    need = api.ce_workspace_bytes(T, V, tp)
    small = api.ce_workspace_bytes(T, V, tp, dtype)
    ws = workspace("ce workspace", small)
    try:
        api.vocab_ce_fwd_bwd(h, W, labels, tp, layout, workspace=ws.t, out=[g.t for g in gs])
    except api.TpsError as e:
        assert e.code == api.ERR_WORKSPACE and need > small
        ws = workspace("ce workspace", need)
        api.vocab_ce_fwd_bwd(h, W, labels, tp, layout, workspace=ws.t, out=[g.t for g in gs])
    check_all(gs + [ws], list(refs) + [None])


@pytest.mark.parametrize("T,d,V,tp,layout", [(37, 128, 4100, 7, "out_in"), (300, 128, 4096, 7, "in_out")])
def test_ce_ex_guard(T, d, V, tp, layout):
    h, W, y = inputs.ce_case(T + 1, T, d, V, torch.bfloat16, w_std=0.2)
    vr = V - 100
    y = y % vr
    y[::5] = -100
    if layout == "out_in":
        W = W.t().contiguous()
    h, W, y = h.cuda(), W.cuda(), y.cuda()
    kw = dict(ignore_index=-100, vocab_size=vr, reduction="mean", want_dwhead=True)
    gs = guard(("loss", (T,), torch.float32), ("loss_reduced", (1,), torch.float32),
               ("dlogits", (T, V), torch.bfloat16), ("dHidden", (T, d), torch.float32),
               ("dWhead", tuple(W.shape), torch.float32), ("owner", (T,), torch.int32))
    refs = api.vocab_ce_fwd_bwd_ex(h, W, y, tp, layout, out=plain(gs), **kw)
    ws = workspace("ce_ex workspace", api.ce_workspace_bytes(T, V, tp))
    api.vocab_ce_fwd_bwd_ex(h, W, y, tp, layout, workspace=ws.t, out=[g.t for g in gs], **kw)
    check_all(gs + [ws], list(refs) + [None])


@pytest.mark.parametrize("form", ["pair", "wide", "grad"])
@pytest.mark.parametrize("T,d,V,tp,layout", [(300, 128, 4096, 7, "in_out"), (600, 640, 5000, 4, "out_in")])
def test_ce_wide_guard(T, d, V, tp, layout, form, monkeypatch):
    """The dHidden GEMM with a K split in three runs: on 256 x 256 tiles
    ("pair"), on 256 x 512 tiles ("wide", the default), and on 256 x 512
    tiles forming dlogits and storing them ("grad"); ragged rows, a
    128-column second output tile, a last K tile of 8 columns."""
    monkeypatch.setenv("TPS_CE_WIDE", "0" if form == "pair" else "1")
    monkeypatch.setenv("TPS_CE_GRAD_IN_GEMM", "1" if form == "grad" else "0")
    monkeypatch.setenv("TPS_CE_KSPLIT", "3")
    h, W, labels = inputs.ce_case(T + V + d, T, d, V, torch.bfloat16, w_std=0.2)
    if layout == "out_in":
        W = W.t().contiguous()
    h, W, labels = h.cuda(), W.cuda(), labels.cuda()
    gs = guard(("loss", (T,), torch.float32), ("dlogits", (T, V), torch.bfloat16), ("dHidden", (T, d), torch.float32),
               ("owner", (T,), torch.int32))
    refs = api.vocab_ce_fwd_bwd(h, W, labels, tp, layout, out=plain(gs))
    ws = workspace("ce workspace", api.ce_workspace_bytes(T, V, tp, torch.bfloat16))
    api.vocab_ce_fwd_bwd(h, W, labels, tp, layout, workspace=ws.t, out=[g.t for g in gs])
    check_all(gs + [ws], list(refs) + [None])
