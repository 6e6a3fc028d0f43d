"""The precision argument for keeping the CE logits as bf16 relative to the
max of their 128-column tile, checked in float64 on the CPU.

With c the tile's max, storing bf16(z - c) rounds each logit by at most
2^-8 (c - z) (round to nearest, 8 significant bits), so a softmax weight
p = e^{z - m} / s moves by at most about p (c - z) 2^-8 <= 2^-8 / e in
absolute terms, whatever the scale of the logits.  Storing bf16(z) itself
rounds by up to 2^-8 |z|, which at large logits breaks the dlogits
tolerance; the shifted form stays far inside it."""
import math

import numpy as np
import pytest
import torch

from parity import BF16_FROB, BF16_MAXABS

TILE = 128


def bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def dlogits(z, y):
    p = np.exp(z - z.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    p[np.arange(len(y)), y] -= 1.0
    return p


def shifted(z):
    t = z.reshape(z.shape[0], -1, TILE)
    c = t.max(2, keepdims=True)
    return (bf16(t - c) + c).reshape(z.shape)


@pytest.mark.parametrize("std", [0.1, 1.28, 10.0, 100.0])
def test_shifted_bf16_logits_bound(std):
    rng = np.random.default_rng(int(std * 100))
    T, V = 16, 64 * TILE
    z = rng.normal(0.0, std, size=(T, V))
    y = rng.integers(0, V, size=T)
    ref = dlogits(z, y)
    err = dlogits(shifted(z), y) - ref
    # per weight: at most 2^-8 / e, plus the second-order terms of the exponential
    assert np.abs(err).max() <= 2.0 ** -8 / math.e * 1.05
    scale = np.abs(ref).max()
    assert np.abs(err).max() <= BF16_MAXABS * scale / 10
    assert np.linalg.norm(err) / np.linalg.norm(ref) <= BF16_FROB / 10


def test_unshifted_bf16_logits_fail_at_large_scale():
    rng = np.random.default_rng(7)
    T, V = 16, 64 * TILE
    z = rng.normal(0.0, 60.0, size=(T, V))
    y = rng.integers(0, V, size=T)
    ref = dlogits(z, y)
    err = dlogits(bf16(z), y) - ref
    assert np.linalg.norm(err) / np.linalg.norm(ref) > BF16_FROB
