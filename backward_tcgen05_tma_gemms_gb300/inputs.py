"""Seeded synthetic inputs shared by the CUDA path and the oracle.

This module holds no arithmetic of the method: it only draws seeded random
numbers, rounds them to the storage dtype and describes the workloads.  Both
the tests (for the oracle) and the benchmark (for the CUDA path) take their
inputs from here so that the two sides see bit-identical operands.

Workloads (all synthetic; the pages use no dataset):
  * sharded matmul, M=3 K=5 N=4, parts=2, axes rows/columns/inner --
    "Sharded GEMM与Backprop：行、列、内维三种切分", section 手动走一遍;
  * the randomised sweep of that section: M, K, N uniform in [1, 16] and
    parts uniform in [1, 20], three axes per case;
  * the TP-MLP of "第 6 课：张量并行 TP" (reference answer): x (2, 8, 64),
    w1 (256, 64), w2 (64, 256) in torch (out, in) layout, tp=4, exact GELU;
  * a Llama-3-8B-shaped TP-MLP: d=4096, F=14336, T=8192 tokens, tp=8,
    tanh-GELU, bf16 operands (weights N(0, 0.02), activations N(0, 1));
  * a vocabulary-sharded cross-entropy: hidden 8192 x 4096, head
    4096 x 128256 (N(0, 0.02)), labels uniform in [0, 128256), tp=8.
"""
from __future__ import annotations

import numpy as np
import torch

# ---------------------------------------------------------------------------
# elementary draws


def normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """float32 N(0, std^2) samples from a numpy Generator."""
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """Round a float32 array to bfloat16 (round-to-nearest-even), on the CPU."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def as_f64(t) -> np.ndarray:
    """Exact widening of a CPU tensor / array to float64 numpy."""
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


# ---------------------------------------------------------------------------
# sharded matmul


def matmul_case(seed: int, M: int, K: int, N: int, dtype=torch.float32):
    """A (M x K), B (K x N), G (M x N) i.i.d. N(0, 1) from default_rng(seed)."""
    rng = np.random.default_rng(seed)
    A, B, G = normal(rng, (M, K)), normal(rng, (K, N)), normal(rng, (M, N))
    if dtype == torch.bfloat16:
        return to_bf16(A), to_bf16(B), to_bf16(G)
    return torch.from_numpy(A), torch.from_numpy(B), torch.from_numpy(G)


def worked_matmul_case():
    """M=3, K=5, N=4, parts=2 from seed 0 (fp32)."""
    A, B, G = matmul_case(0, 3, 5, 4)
    return A, B, G, 2


def sweep_case(seed: int):
    """One case of the randomised sweep: returns (A, B, G, parts), fp32."""
    rng = np.random.default_rng(seed)
    M, K, N = (int(v) for v in rng.integers(1, 17, size=3))
    parts = int(rng.integers(1, 21))
    A, B, G = normal(rng, (M, K)), normal(rng, (K, N)), normal(rng, (M, N))
    return torch.from_numpy(A), torch.from_numpy(B), torch.from_numpy(G), parts


AXES = ("rows", "columns", "inner")

# ---------------------------------------------------------------------------
# TP MLP


def lesson_mlp_case():
    """The reference answer's exercise inputs: torch.manual_seed(0), then x,
    w1, w2 in that order, then the upstream gradient gy of Y's shape."""
    g = torch.Generator().manual_seed(0)
    x = torch.randn(2, 8, 64, generator=g)
    w1 = torch.randn(256, 64, generator=g)
    w2 = torch.randn(64, 256, generator=g)
    gy = torch.randn(2, 8, 64, generator=g)
    return x, w1, w2, gy, 4


def mlp_case(seed: int, T: int, d: int, F: int, dtype=torch.bfloat16, w_std: float = 0.02,
             layout: str = "in_out"):
    """X (T x d), W1, W2, G_Y (T x d).  Weights are (in, out) -- W1 d x F and
    W2 F x d -- for layout "in_out", or torch (out, in) -- W1 F x d and W2
    d x F -- for layout "out_in".  Weights N(0, w_std^2), X and G_Y N(0, 1)."""
    rng = np.random.default_rng(seed)
    X = normal(rng, (T, d))
    W1 = normal(rng, (d, F), w_std)
    W2 = normal(rng, (F, d), w_std)
    GY = normal(rng, (T, d))
    if layout == "out_in":
        W1, W2 = np.ascontiguousarray(W1.T), np.ascontiguousarray(W2.T)
    conv = to_bf16 if dtype == torch.bfloat16 else torch.from_numpy
    return conv(X), conv(W1), conv(W2), conv(GY)


LLAMA_MLP = dict(T=8192, d=4096, F=14336, tp=8)


def glu_case(seed: int, T: int, d: int, F: int, dtype=torch.bfloat16, w_std: float = 0.02,
             layout: str = "in_out"):
    """X (T x d), Wg, Wu, W2, G_Y (T x d) for the gated MLP, drawn in that
    order.  Wg and Wu are d x F and W2 F x d for layout "in_out", or their
    transposes for "out_in".  Weights N(0, w_std^2), X and G_Y N(0, 1)."""
    rng = np.random.default_rng(seed)
    X = normal(rng, (T, d))
    Wg = normal(rng, (d, F), w_std)
    Wu = normal(rng, (d, F), w_std)
    W2 = normal(rng, (F, d), w_std)
    GY = normal(rng, (T, d))
    if layout == "out_in":
        Wg, Wu, W2 = (np.ascontiguousarray(w.T) for w in (Wg, Wu, W2))
    conv = to_bf16 if dtype == torch.bfloat16 else torch.from_numpy
    return conv(X), conv(Wg), conv(Wu), conv(W2), conv(GY)

# ---------------------------------------------------------------------------
# attention projections


def attn_case(seed: int, T: int, d: int, H: int, Hkv: int, dh: int, dtype=torch.bfloat16, w_std: float = 0.02,
              layout: str = "in_out"):
    """X (T x d); Wq (d x H dh), Wk, Wv (d x Hkv dh), Wo (H dh x d) for
    layout "in_out" or their transposes for "out_in"; the attention core's
    gradients dQ (T x H dh), dK, dV (T x Hkv dh), its context C (T x H dh),
    and G_Y (T x d), drawn in that order.  Weights N(0, w_std^2), the rest
    N(0, 1)."""
    rng = np.random.default_rng(seed)
    nq, nkv = H * dh, Hkv * dh
    X = normal(rng, (T, d))
    Wq = normal(rng, (d, nq), w_std)
    Wk = normal(rng, (d, nkv), w_std)
    Wv = normal(rng, (d, nkv), w_std)
    Wo = normal(rng, (nq, d), w_std)
    dQ = normal(rng, (T, nq))
    dK = normal(rng, (T, nkv))
    dV = normal(rng, (T, nkv))
    C = normal(rng, (T, nq))
    GY = normal(rng, (T, d))
    if layout == "out_in":
        Wq, Wk, Wv, Wo = (np.ascontiguousarray(w.T) for w in (Wq, Wk, Wv, Wo))
    conv = to_bf16 if dtype == torch.bfloat16 else torch.from_numpy
    return dict(X=conv(X), Wq=conv(Wq), Wk=conv(Wk), Wv=conv(Wv), Wo=conv(Wo), dQ=conv(dQ), dK=conv(dK),
                dV=conv(dV), C=conv(C), GY=conv(GY))


LLAMA_ATTN = dict(T=8192, d=4096, H=32, Hkv=8, dh=128, tp=8)

# ---------------------------------------------------------------------------
# vocabulary cross-entropy


def ce_case(seed: int, T: int, d: int, V: int, dtype=torch.bfloat16, w_std: float = 0.02):
    """hidden (T x d) N(0, 1), head (d x V) N(0, w_std^2) in (in, out) layout,
    labels uniform in [0, V) as int64."""
    rng = np.random.default_rng(seed)
    h = normal(rng, (T, d))
    W = normal(rng, (d, V), w_std)
    labels = rng.integers(0, V, size=T, dtype=np.int64)
    conv = to_bf16 if dtype == torch.bfloat16 else torch.from_numpy
    return conv(h), conv(W), torch.from_numpy(labels)


LLAMA_CE = dict(T=8192, d=4096, V=128256, tp=8)
