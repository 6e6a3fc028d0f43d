"""Parity tolerances for comparing the CUDA path with the float64 oracle.

fp32 operands (true fp32 FMA on the GPU):   max |got - ref| <= 1e-4 * max |ref|
bf16 operands (fp32 accumulation):         max |got - ref| <= 2e-2 * max |ref|
                                           and ||got - ref||_F <= 5e-3 * ||ref||_F
Integer / index results (shard offsets, owner ranks) must match exactly."""
import numpy as np

FP32_MAXABS = 1e-4
BF16_MAXABS = 2e-2
BF16_FROB = 5e-3


def _np(x):
    import torch
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def errors(got, ref):
    g, r = _np(got), _np(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    if r.size == 0:
        return 0.0, 0.0, 0.0
    scale = float(np.abs(r).max())
    maxabs = float(np.abs(g - r).max())
    fro = float(np.linalg.norm(g - r)) / max(float(np.linalg.norm(r)), 1e-300)
    return maxabs, scale, fro


def assert_fp32(got, ref, what=""):
    maxabs, scale, _ = errors(got, ref)
    assert np.all(np.isfinite(_np(got))), f"{what}: non-finite values"
    assert maxabs <= FP32_MAXABS * max(scale, 1e-30), f"{what}: max-abs {maxabs:.3e} > 1e-4 x {scale:.3e}"


def assert_bf16(got, ref, what=""):
    maxabs, scale, fro = errors(got, ref)
    assert np.all(np.isfinite(_np(got))), f"{what}: non-finite values"
    assert maxabs <= BF16_MAXABS * max(scale, 1e-30), f"{what}: max-abs {maxabs:.3e} > 2e-2 x {scale:.3e}"
    assert fro <= BF16_FROB, f"{what}: relative Frobenius {fro:.3e} > 5e-3"


def assert_close(got, ref, bf16: bool, what=""):
    (assert_bf16 if bf16 else assert_fp32)(got, ref, what)
