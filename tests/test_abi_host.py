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
              "tps_mlp_workspace_bytes", "tps_ce_workspace_bytes", "tps_ce_workspace_bytes_ex", "tps_last_device_error",
              "tps_strerror"]:
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
    # pre-activation, activation and dZ, T x F each in the operand dtype
    assert lib.tps_mlp_workspace_bytes(8192, 4096, 14336, 8, 1) == 3 * 8192 * 14336 * 2
    assert lib.tps_mlp_workspace_bytes(64, 32, 100, 8, 0) == 3 * ((64 * 100 * 4 + 255) // 256 * 256)
    assert lib.tps_ce_workspace_bytes(8192, 128256, 8) >= 8192 * 128256 * 4


def test_ce_workspace_query_by_dtype(lib):
    """bf16 operands with shards of >= 128 columns keep the logits as bf16:
    the query drops half of the T x V fp32 region; every other case asks
    for the full size."""
    T, V, tp = 8192, 128256, 8
    full = lib.tps_ce_workspace_bytes(T, V, tp)
    bf16 = lib.tps_ce_workspace_bytes_ex(T, V, tp, 1)
    assert full - bf16 == T * V * 2
    assert 0.45 < bf16 / full < 0.55
    assert lib.tps_ce_workspace_bytes_ex(T, V, tp, 0) == full            # fp32 operands
    assert lib.tps_ce_workspace_bytes_ex(64, 1000, 8, 1) == lib.tps_ce_workspace_bytes(64, 1000, 8)  # 125-col shards
    assert lib.tps_ce_workspace_bytes_ex(64, 1024, 8, 1) < lib.tps_ce_workspace_bytes(64, 1024, 8)   # 128-col shards
    assert lib.tps_ce_workspace_bytes_ex(-1, V, tp, 1) == 0 and lib.tps_ce_workspace_bytes_ex(T, V, 0, 1) == 0


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


def test_widened_rows_validation_codes(lib):
    """The gated MLP, attention projections and extended CE reject bad
    arguments with the documented codes before anything is launched."""
    from backward_tcgen05_tma_gemms_gb300.api import TpsCeOptions, NO_IGNORE
    r = ctypes.byref
    ws = ctypes.c_void_p(0x100000)
    # gated MLP: X 16x64, Wg/Wu 64x96, W2 96x64
    X, Wg, Wu, W2, GY = _fake([16, 64]), _fake([64, 96]), _fake([64, 96]), _fake([96, 64]), _fake([16, 64])
    outs = [_fake([16, 64]), _fake([16, 64]), _fake([64, 96]), _fake([64, 96]), _fake([96, 64])]
    glu = lambda tp=4, act=3, wu=Wu, size=1 << 30, x=X: lib.tps_glu_mlp_fwd_bwd(
        r(x), r(Wg), r(wu), r(W2), r(GY), tp, act, 0, *[r(o) for o in outs], ws, size, None)
    assert glu(tp=0) == 2
    assert glu(act=9) == 9
    assert glu(wu=_fake([64, 95])) == 1
    assert glu(x=_fake([16, 64], dtype=1)) == 3
    assert glu(size=64) == 6
    # attention: 6 query heads of 16, 2 KV heads
    Xa, Wq, Wk, Wv = _fake([8, 32]), _fake([32, 96]), _fake([32, 32]), _fake([32, 32])
    Q, K, V = _fake([8, 96]), _fake([8, 32]), _fake([8, 32])
    qkv = lambda H=6, Hkv=2, tp=2, wk=Wk, q=Q, k=K: lib.tps_attn_qkv_fwd(
        r(Xa), r(Wq), r(wk), r(Wv), H, Hkv, tp, 0, r(q), r(k), r(V), None)
    assert qkv(tp=4) == 2                       # 6 heads do not split over 4 ranks
    assert qkv(H=4, Hkv=3) == 2                 # 4 query heads do not group over 3 KV heads
    assert qkv(H=5, Hkv=1, tp=1) == 1           # 96 columns are not 5 whole heads
    assert qkv(wk=_fake([32, 48])) == 1         # Wk not H_kv heads wide
    assert qkv(q=_fake([8, 95])) == 1
    assert qkv(k=_fake([8, 32], dtype=1)) == 3  # Q, K, V dtypes differ
    C, Wo, G = _fake([8, 96]), _fake([96, 32]), _fake([8, 32])
    out = lambda H=6, tp=2, dc=_fake([8, 96]): lib.tps_attn_out_fwd_bwd(
        r(C), r(Wo), r(G), H, tp, 0, r(_fake([8, 32])), r(dc), r(_fake([96, 32])), None)
    assert out(tp=4) == 2
    assert out(dc=_fake([8, 96], dtype=3)) == 3
    # extended CE: vocabulary 100, 4 tokens
    h, W, lab = _fake([4, 16]), _fake([16, 100]), _fake([4], dtype=3)
    loss, dl, dh = _fake([4]), _fake([4, 100]), _fake([4, 16])

    def ce(ignore=NO_IGNORE, vocab=0, red=0, den=0.0, reserved=0, lred=None, dw=None):
        o = TpsCeOptions(ignore, vocab, red, reserved, den)
        return lib.tps_vocab_ce_fwd_bwd_ex(r(h), r(W), r(lab), 2, 0, r(o), r(loss),
                                           r(lred) if lred is not None else None, r(dl), r(dh),
                                           r(dw) if dw is not None else None, None, ws, 1 << 30, None)
    assert ce(vocab=101) == 1
    assert ce(vocab=-1) == 1
    assert ce(red=3) == 9
    assert ce(red=2, den=-1.0) == 9
    assert ce(red=2, den=float("nan")) == 9
    assert ce(reserved=1) == 9
    assert ce(red=1, lred=_fake([2])) == 1      # loss_reduced holds one float
    assert ce(dw=_fake([16, 99])) == 1          # dWhead must match Whead
    assert ce(dw=_fake([16, 100], dtype=1)) == 3


def test_header_is_plain_c(tmp_path):
    """include/tps.h is a C ABI: it compiles as strict C99 and as C++."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    src = tmp_path / "use_tps.c"
    src.write_text('#include "tps.h"\n'
                   'int main(void) {\n'
                   '  tps_ce_options o = {TPS_NO_IGNORE, 0, TPS_REDUCE_MEAN, 0, 0.0};\n'
                   '  tps_tensor t;\n'
                   '  (void)o; (void)t;\n'
                   '  return TPS_OK;\n'
                   '}\n')
    inc = os.path.join(ROOT, "include")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, "-c", str(src), "-o",
                    str(tmp_path / "c.o")], check=True)
    if shutil.which("g++"):
        subprocess.run(["g++", "-std=c++11", "-Wall", "-Werror", "-I", inc, "-x", "c++", "-c", str(src), "-o",
                        str(tmp_path / "cpp.o")], check=True)


def test_debug_build_reports_its_flag(lib):
    """The debug build (TPS_DEBUG=1, bounds-checked stores) compiles, loads
    without a GPU and says what it is; the release build says it is not."""
    from backward_tcgen05_tma_gemms_gb300 import api, build
    path = build.build(debug=True)
    dbg = ctypes.CDLL(path)
    assert dbg.tps_build_flags() & api.BUILD_DEBUG
    assert not lib.tps_build_flags() & api.BUILD_DEBUG
    dbg.tps_strerror.restype = ctypes.c_char_p
    assert b"debug" in dbg.tps_strerror(api.ERR_BOUNDS)
