"""tps_mlp_fwd_bwd_noalloc: the MLP entry point for callers that cannot
allocate device memory (a hosting framework owns the allocator, or the call
sits on a path that must not call cudaMalloc).  It uses the library's static
device scratch instead of a workspace.

The GPU test calls it through the C ABI twice in a row, on different inputs,
and checks each result against the regular entry point (tps_mlp_fwd_bwd with
a torch-allocated workspace) within the bf16 parity tolerance.  This file is
collected last so that a run stopping at the first failure has already run
every other test."""
import ctypes

import pytest
import torch

from backward_tcgen05_tma_gemms_gb300 import api, build, inputs
from parity import assert_close


def _raw_noalloc(X, W1, W2, GY, tp, act, layout, outs):
    """Direct C-ABI call of tps_mlp_fwd_bwd_noalloc (no Python wrapper)."""
    lib = api.library()
    views = [api._tt(t) for t in (X, W1, W2, GY, *outs)]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.tps_mlp_fwd_bwd_noalloc(*[v[0] for v in views[:4]], tp, api.ACTS[act], api.LAYOUTS[layout],
                                       *[v[0] for v in views[4:]], stream)


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    T, d, F, tp = 512, 256, 1024, 8
    assert api.mlp_workspace_bytes(T, d, F, tp, torch.bfloat16) <= api.MLP_NOALLOC_SCRATCH_BYTES
    for seed in (1, 2):   # two calls in a row; the second sees the first's scratch contents
        X, W1, W2, GY = (t.cuda() for t in inputs.mlp_case(seed, T, d, F, torch.bfloat16, w_std=0.05))
        ref = api.mlp_fwd_bwd(X, W1, W2, GY, tp, "gelu_tanh", "in_out")
        torch.cuda.synchronize()
        outs = [torch.full(t.shape, float("nan"), device="cuda") for t in ref]
        rc = _raw_noalloc(X, W1, W2, GY, tp, "gelu_tanh", "in_out", outs)
        assert rc == 0, api.library().tps_last_error_detail()
        assert api.last_device_error() == 0
        for name, g, r in zip(("Y", "dX", "dW1", "dW2"), outs, ref):
            assert_close(g.cpu(), r.cpu(), True, f"call {seed} {name}")


def test_noalloc_rejects_oversize_before_any_launch():
    """The size check is on the host, before any CUDA call, so this runs
    without a GPU: the tensors' data pointers are never dereferenced."""
    build.build()
    lib = api.library()

    def fake(shape, dtype):
        t = api.TpsTensor()
        t.data, t.dtype, t.ndim = 0x1000, dtype, len(shape)
        acc = 1
        for i in reversed(range(len(shape))):
            t.shape[i], t.stride[i] = shape[i], acc
            acc *= shape[i]
        return t

    T, d, F = 8192, 4096, 14336       # needs 940 MB of scratch
    ts = [fake(s, api.BF16) for s in [(T, d), (d, F), (F, d), (T, d)]] + \
         [fake(s, api.F32) for s in [(T, d), (T, d), (d, F), (F, d)]]
    rc = lib.tps_mlp_fwd_bwd_noalloc(*[ctypes.byref(t) for t in ts[:4]], 8, 1, 0,
                                     *[ctypes.byref(t) for t in ts[4:]], None)
    assert rc == api.ERR_WORKSPACE
    assert b"static scratch holds" in lib.tps_last_error_detail()
