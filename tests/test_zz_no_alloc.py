"""tps_mlp_fwd_bwd_noalloc: the MLP entry point for callers that cannot
allocate device memory (a hosting framework owns the allocator, or the call
sits on a path that must not call cudaMalloc).  It uses the library's static
device scratch instead of a workspace.

The GPU test calls it through the C ABI twice in a row, the second time on a
smaller problem (its scratch regions then start at other offsets, over the
first call's leftover bytes), and checks that each result is bit-identical
to the regular entry point's (tps_mlp_fwd_bwd with a torch-allocated
workspace: the same kernels in the same order), and that the second call
leaves the device's free memory unchanged.  This file is collected last so
that a run stopping at the first failure has already run every other test."""
import ctypes

import pytest
import torch

from backward_tcgen05_tma_gemms_gb300 import api, build, inputs


def _raw_noalloc(X, W1, W2, GY, tp, act, layout, outs):
    """Direct C-ABI call of tps_mlp_fwd_bwd_noalloc (no Python wrapper)."""
    lib = api.library()
    views = [api._tt(t) for t in (X, W1, W2, GY, *outs)]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.tps_mlp_fwd_bwd_noalloc(*[v[0] for v in views[:4]], tp, api.ACTS[act], api.LAYOUTS[layout],
                                       *[v[0] for v in views[4:]], stream)


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    tp = 8
    # two calls in a row; the second is smaller, so its pre-activation,
    # activation and dZ regions overlay the first call's at other offsets
    for seed, (T, d, F) in ((1, (512, 256, 1024)), (2, (256, 256, 768))):
        assert api.mlp_workspace_bytes(T, d, F, tp, torch.bfloat16) <= api.MLP_NOALLOC_SCRATCH_BYTES
        X, W1, W2, GY = (t.cuda() for t in inputs.mlp_case(seed, T, d, F, torch.bfloat16, w_std=0.05))
        ref = api.mlp_fwd_bwd(X, W1, W2, GY, tp, "gelu_tanh", "in_out")
        outs = [torch.full(t.shape, float("nan"), device="cuda") for t in ref]
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        rc = _raw_noalloc(X, W1, W2, GY, tp, "gelu_tanh", "in_out", outs)
        assert rc == 0, api.library().tps_last_error_detail()
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert api.last_device_error() == 0
        if seed == 2:   # the first call may load the module and place the array; later calls take nothing
            assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
        for name, g, r in zip(("Y", "dX", "dW1", "dW2"), outs, ref):
            assert torch.equal(g, r), f"call {seed} {name}: differs from the workspace entry point"


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
