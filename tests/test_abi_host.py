"""Host-side checks of the C ABI (CPU only, no GPU call).

The library must load without a GPU, export every entry point declared in
include/tps.h, plan shards exactly like the oracle, and reject bad
arguments before anything is launched."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from backward_tcgen05_tma_gemms_gb300 import build, api
    build.build()
    return api.library()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "tps.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tps_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_entry_points():
    syms = declared_symbols()
    for s in ["tps_plan_shards", "tps_matmul_fwd_bwd", "tps_mlp_fwd_bwd", "tps_vocab_ce_fwd_bwd",
              "tps_mlp_workspace_bytes", "tps_ce_workspace_bytes", "tps_last_device_error", "tps_strerror"]:
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, f"not exported: {missing}"


def test_plan_shards_matches_oracle(lib, orc):
    for dim in range(0, 70):
        for parts in range(1, 90):
            off = (ctypes.c_int64 * (parts + 1))()
            assert lib.tps_plan_shards(dim, parts, off) == 0
            assert list(off) == list(orc.plan_shards(dim, parts))
    off = (ctypes.c_int64 * 1)()
    assert lib.tps_plan_shards(5, 0, off) == 2       # TPS_ERR_PARTITION
    assert lib.tps_plan_shards(-1, 2, off) == 1      # TPS_ERR_SHAPE


def _fake(shape, dtype=0, strides=None):
    from backward_tcgen05_tma_gemms_gb300.api import TpsTensor
    t = TpsTensor()
    t.data = 0x1000  # never dereferenced: every call below fails validation first
    t.dtype = dtype
    t.ndim = len(shape)
    if strides is None:
        strides, acc = [], 1
        for s in reversed(shape):
            strides.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, strides)):
        t.shape[i] = s
        t.stride[i] = st
    return t


def _mm(lib, A, B, G, parts, axis, Y=None, dA=None, dB=None):
    r = lambda t: ctypes.byref(t) if t is not None else None
    return lib.tps_matmul_fwd_bwd(r(A), r(B), r(G), parts, axis, r(Y), r(dA), r(dB), None)


def test_matmul_validation_codes(lib):
    A, B, G = _fake([3, 5]), _fake([5, 4]), _fake([3, 4])
    assert _mm(lib, A, _fake([6, 4]), G, 2, 2) == 1                 # K mismatch -> shape
    assert _mm(lib, A, B, _fake([4, 3]), 2, 2) == 1                 # G shape
    assert _mm(lib, _fake([3, 5, 1]), B, G, 2, 2) == 1              # not 2-D
    assert _mm(lib, A, B, G, 0, 2) == 2                             # parts < 1 -> partition
    assert _mm(lib, A, B, G, 2, 7) == 2                             # unknown axis
    assert _mm(lib, A, _fake([5, 4], dtype=1), G, 2, 2) == 3        # mixed dtypes
    assert _mm(lib, A, B, G, 2, 2, Y=_fake([3, 5])) == 1            # wrong output shape
    assert _mm(lib, A, B, G, 2, 2, Y=_fake([3, 4], dtype=1)) == 3   # bf16 output
    assert _mm(lib, _fake([3, 5], strides=[10, 2]), B, G, 2, 2) == 4  # no unit stride
    assert lib.tps_matmul_fwd_bwd(None, ctypes.byref(B), ctypes.byref(G), 2, 2, None, None, None, None) == 9


def test_mlp_and_ce_validation_codes(lib):
    r = ctypes.byref
    X, W1, W2, GY = _fake([16, 64]), _fake([64, 256]), _fake([256, 64]), _fake([16, 64])
    Y, dX, dW1, dW2 = _fake([16, 64]), _fake([16, 64]), _fake([64, 256]), _fake([256, 64])
    ws = ctypes.c_void_p(0x100000)
    call = lambda tp, act, lay, w2=W2, size=1 << 30: lib.tps_mlp_fwd_bwd(
        r(X), r(W1), r(w2), r(GY), tp, act, lay, r(Y), r(dX), r(dW1), r(dW2), ws, size, None)
    assert call(0, 0, 0) == 2
    assert call(4, 9, 0) == 9
    assert call(4, 0, 5) == 9
    assert call(4, 0, 0, w2=_fake([64, 256])) == 1
    assert call(4, 0, 0, size=16) == 6                              # workspace too small
    h, W, lab = _fake([8, 32]), _fake([32, 100]), _fake([8], dtype=3)
    loss, dl, dh = _fake([8]), _fake([8, 100]), _fake([8, 32])
    ce = lambda tp, lab=lab, dl=dl: lib.tps_vocab_ce_fwd_bwd(r(h), r(W), r(lab), tp, 0, r(loss), r(dl), r(dh), None,
                                                             ws, 1 << 30, None)
    assert ce(0) == 2
    assert ce(3, lab=_fake([8], dtype=0)) == 3                      # float labels
    assert ce(3, lab=_fake([7], dtype=3)) == 1
    assert ce(3, dl=_fake([8, 100], dtype=1)) == 3                  # dlogits dtype must match h


def test_workspace_queries(lib):
    assert lib.tps_mlp_workspace_bytes(8192, 4096, 14336, 8, 1) >= 8192 * 14336 * 8
    assert lib.tps_ce_workspace_bytes(8192, 128256, 8) >= 8192 * 128256 * 4


def test_python_wrapper_rejects_like_the_page():
    from backward_tcgen05_tma_gemms_gb300 import api
    A = torch.zeros(3, 5)
    with pytest.raises(ValueError, match="partition"):
        api.matmul_fwd_bwd(A, torch.zeros(5, 4), torch.zeros(3, 4), True, "inner")   # bool is not int
    with pytest.raises(ValueError, match="partition"):
        api.matmul_fwd_bwd(A, torch.zeros(5, 4), torch.zeros(3, 4), 2.0, "inner")
    with pytest.raises(ValueError, match="partition"):
        api.matmul_fwd_bwd(A, torch.zeros(5, 4), torch.zeros(3, 4), 2, "diagonal")
    with pytest.raises(ValueError, match="shape"):
        api.matmul_fwd_bwd(A, torch.zeros(4, 4), torch.zeros(3, 4), 2, "inner")


def test_no_cpu_path():
    """CPU tensors are refused (the library has no CPU fallback)."""
    from backward_tcgen05_tma_gemms_gb300 import api
    with pytest.raises(ValueError, match="GPU"):
        api.matmul_fwd_bwd(torch.zeros(3, 5), torch.zeros(5, 4), torch.zeros(3, 4), 2, "inner")


def test_plan_heads_matches_oracle(orc):
    """The library's head plan (host code, no device work) against the
    oracle's, bit for bit, over a grid of head counts and tp."""
    from backward_tcgen05_tma_gemms_gb300 import api
    for H in (1, 4, 6, 8, 12, 32, 64):
        for Hkv in (1, 2, 4, 8, 32):
            for tp in range(1, 70):
                try:
                    want = orc.plan_heads(H, Hkv, tp)
                except ValueError:
                    with pytest.raises(ValueError, match="partition"):
                        api.plan_heads(H, Hkv, tp)
                    continue
                q_off, kv_first, cnt, rep = api.plan_heads(H, Hkv, tp)
                assert q_off == want[0].tolist() and kv_first == want[1].tolist(), (H, Hkv, tp)
                assert (cnt, rep) == (want[2], want[3]), (H, Hkv, tp)
