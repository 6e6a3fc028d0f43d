"""ctypes binding of libtps.so (include/tps.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  Tensors must be CUDA tensors on the current device;
outputs and workspace are allocated with torch on that device and the work
is enqueued on torch's current stream.  There is no CPU path: without the
built library or a GPU these functions raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# TPS_LIBRARY selects another build of the library (the debug build,
# libtps_debug.so, whose kernels bounds-check every store).
LIB_PATH = os.environ.get("TPS_LIBRARY") or os.path.join(_PKG, "libtps.so")

F32, BF16, I32, I64 = 0, 1, 2, 3
(OK, ERR_SHAPE, ERR_PARTITION, ERR_DTYPE, ERR_LAYOUT, ERR_LABEL, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_ARG,
 ERR_BOUNDS) = range(11)
BUILD_DEBUG = 1  # bit of tps_build_flags()
AXES = {"rows": 0, "columns": 1, "inner": 2}
ACTS = {"gelu": 0, "gelu_erf": 0, "gelu_tanh": 1, "tanh": 2, "silu": 3}
LAYOUTS = {"in_out": 0, "out_in": 1}

_DTYPES = {torch.float32: F32, torch.bfloat16: BF16, torch.int32: I32, torch.int64: I64}


class TpsTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class TpsCeOptions(ctypes.Structure):
    """tps_ce_options of include/tps.h."""
    _fields_ = [("ignore_index", ctypes.c_int64), ("vocab_size", ctypes.c_int64), ("reduction", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("denominator", ctypes.c_double)]


NO_IGNORE = -(2 ** 63)
REDUCTIONS = {"none": 0, "sum": 1, "mean": 2}


class TpsError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} (code {code})")
        self.code = code


_lib = None


def library():
    """Load libtps.so once.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libtps.so is not built ({LIB_PATH}); run "
                           "`python -m backward_tcgen05_tma_gemms_gb300.build` first")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(TpsTensor)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.tps_plan_shards.argtypes = [i64, i32, ctypes.POINTER(i64)]
    lib.tps_matmul_fwd_bwd.argtypes = [P, P, P, i32, i32, P, P, P, vp]
    lib.tps_mlp_fwd_bwd.argtypes = [P, P, P, P, i32, i32, i32, P, P, P, P, vp, sz, vp]
    lib.tps_mlp_fwd_bwd_noalloc.argtypes = [P, P, P, P, i32, i32, i32, P, P, P, P, vp]
    lib.tps_glu_mlp_fwd_bwd.argtypes = [P, P, P, P, P, i32, i32, i32, P, P, P, P, P, vp, sz, vp]
    lib.tps_glu_mlp_workspace_bytes.argtypes = [i64, i64, i64, i32, i32]
    lib.tps_glu_mlp_workspace_bytes.restype = sz
    lib.tps_plan_heads.argtypes = [i32, i32, i32, ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i32),
                                   ctypes.POINTER(i32)]
    lib.tps_attn_qkv_fwd.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P, P, vp]
    lib.tps_attn_qkv_bwd.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, P, P, P, P, vp]
    lib.tps_attn_out_fwd_bwd.argtypes = [P, P, P, i32, i32, i32, P, P, P, vp]
    lib.tps_mlp_workspace_bytes.argtypes = [i64, i64, i64, i32, i32]
    lib.tps_mlp_workspace_bytes.restype = sz
    lib.tps_vocab_ce_fwd_bwd.argtypes = [P, P, P, i32, i32, P, P, P, P, vp, sz, vp]
    lib.tps_vocab_ce_fwd_bwd_ex.argtypes = [P, P, P, i32, i32, ctypes.POINTER(TpsCeOptions), P, P, P, P, P, P, vp,
                                            sz, vp]
    lib.tps_ce_workspace_bytes.argtypes = [i64, i64, i32]
    lib.tps_ce_workspace_bytes.restype = sz
    lib.tps_ce_workspace_bytes_ex.argtypes = [i64, i64, i32, i32]
    lib.tps_ce_workspace_bytes_ex.restype = sz
    lib.tps_last_device_error.argtypes = [vp]
    lib.tps_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    lib.tps_strerror.argtypes = [ctypes.c_int]
    lib.tps_strerror.restype = ctypes.c_char_p
    lib.tps_last_error_detail.restype = ctypes.c_char_p
    lib.tps_profile_reset.argtypes = [ctypes.c_int]
    lib.tps_profile_summary.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(i64),
                                        ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_double)]
    lib.tps_launch_count.restype = i64
    _lib = lib
    return lib


# --------------------------------------------------------------------- helpers

def _tt(t: Optional[torch.Tensor]):
    """tps_tensor view of a CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("tensors must live on the GPU (no CPU path)")
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() > 4 or t.dim() < 1:
        raise ValueError("shape")
    s = TpsTensor()
    s.data = t.data_ptr()
    s.dtype = _DTYPES[t.dtype]
    s.ndim = t.dim()
    for i in range(t.dim()):
        s.shape[i] = t.shape[i]
        s.stride[i] = t.stride(i)
    return ctypes.byref(s), s  # keep the struct alive with the reference


def _ref(x):
    return None if x is None else x[0]


def _check(rc: int):
    if rc == OK:
        return
    lib = library()
    detail = lib.tps_last_error_detail().decode()
    if rc == ERR_SHAPE:
        raise ValueError("shape")
    if rc == ERR_PARTITION:
        raise ValueError("partition")
    raise TpsError(rc, f"{lib.tps_strerror(rc).decode()}: {detail}")


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _parts(v, name="parts") -> int:
    if type(v) is not int or v < 1:
        raise ValueError("partition")
    return v


# --------------------------------------------------------------------- API

def plan_shards(dim: int, parts: int) -> list:
    """array_split offsets (parts + 1 entries) computed by the library."""
    _parts(parts)
    off = (ctypes.c_int64 * (parts + 1))()
    _check(library().tps_plan_shards(int(dim), parts, off))
    return list(off)


def matmul_fwd_bwd(A: torch.Tensor, B: torch.Tensor, G: torch.Tensor, parts: int, axis: str,
                   out: Optional[Sequence[torch.Tensor]] = None):
    """(Y, dA, dB) of L = <G, AB> split over `parts` ranks along `axis`.
    Results are fp32; `out` may supply (Y, dA, dB) to write into."""
    _parts(parts)
    if axis not in AXES:
        raise ValueError("partition")
    if A.dim() != 2 or B.dim() != 2 or G.dim() != 2 or A.shape[1] != B.shape[0] or tuple(G.shape) != (A.shape[0], B.shape[1]):
        raise ValueError("shape")
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        kw = dict(device=A.device, dtype=torch.float32)
        out = (torch.empty(M, N, **kw), torch.empty(M, K, **kw), torch.empty(K, N, **kw))
    Y, dA, dB = out
    a, b, g, y, da, db = (_tt(t) for t in (A, B, G, Y, dA, dB))
    _check(library().tps_matmul_fwd_bwd(_ref(a), _ref(b), _ref(g), parts, AXES[axis], _ref(y), _ref(da), _ref(db),
                                        _stream(A.device)))
    return Y, dA, dB


def mlp_workspace_bytes(T: int, d: int, F: int, tp: int, dtype: torch.dtype) -> int:
    return int(library().tps_mlp_workspace_bytes(T, d, F, tp, _DTYPES[dtype]))


def mlp_fwd_bwd(X: torch.Tensor, W1: torch.Tensor, W2: torch.Tensor, GY: torch.Tensor, tp: int,
                act: str = "gelu_tanh", weight_layout: str = "in_out", workspace: Optional[torch.Tensor] = None,
                out: Optional[Sequence[torch.Tensor]] = None):
    """Column-then-row TP MLP forward + backward.  Returns (Y, dX, dW1, dW2)
    in fp32 (Y, dX shaped like X; dW1, dW2 like W1, W2)."""
    _parts(tp, "tp")
    if act not in ACTS or weight_layout not in LAYOUTS:
        raise ValueError("argument")
    d = X.shape[-1]
    T = X.numel() // d if d else 0
    F = W1.shape[1] if weight_layout == "in_out" else W1.shape[0]
    if out is None:
        kw = dict(device=X.device, dtype=torch.float32)
        out = (torch.empty(X.shape, **kw), torch.empty(X.shape, **kw), torch.empty(W1.shape, **kw),
               torch.empty(W2.shape, **kw))
    Y, dX, dW1, dW2 = out
    need = mlp_workspace_bytes(T, d, F, tp, X.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=X.device)
    args = [_tt(t) for t in (X, W1, W2, GY, Y, dX, dW1, dW2)]
    _check(library().tps_mlp_fwd_bwd(*[_ref(a) for a in args[:4]], tp, ACTS[act], LAYOUTS[weight_layout],
                                     *[_ref(a) for a in args[4:]], ctypes.c_void_p(workspace.data_ptr()),
                                     workspace.numel() * workspace.element_size(), _stream(X.device)))
    return Y, dX, dW1, dW2


# Size of the static scratch of tps_mlp_fwd_bwd_noalloc (TPS_MLP_NOALLOC_SCRATCH_BYTES).
MLP_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def mlp_fwd_bwd_noalloc(X: torch.Tensor, W1: torch.Tensor, W2: torch.Tensor, GY: torch.Tensor, tp: int,
                        act: str = "gelu_tanh", weight_layout: str = "in_out",
                        out: Optional[Sequence[torch.Tensor]] = None):
    """mlp_fwd_bwd without a workspace, for callers that cannot allocate
    device memory (an allocator owned by a hosting framework, or a path that
    must not call cudaMalloc): the library's static 32 MiB device scratch is
    used instead.  Larger problems are rejected; calls that overlap on the
    GPU race on the shared scratch.  Outputs still come from `out` (or are
    allocated here by torch when `out` is None)."""
    _parts(tp, "tp")
    if act not in ACTS or weight_layout not in LAYOUTS:
        raise ValueError("argument")
    if out is None:
        kw = dict(device=X.device, dtype=torch.float32)
        out = (torch.empty(X.shape, **kw), torch.empty(X.shape, **kw), torch.empty(W1.shape, **kw),
               torch.empty(W2.shape, **kw))
    args = [_tt(t) for t in (X, W1, W2, GY, *out)]
    _check(library().tps_mlp_fwd_bwd_noalloc(*[_ref(a) for a in args[:4]], tp, ACTS[act], LAYOUTS[weight_layout],
                                             *[_ref(a) for a in args[4:]], _stream(X.device)))
    return tuple(out)


def ce_workspace_bytes(T: int, V: int, tp: int, dtype: Optional[torch.dtype] = None) -> int:
    """Workspace bytes of the CE entry points: enough for every path when
    `dtype` is None, else for operands of `dtype` on the tensor-core path
    (bf16 logits)."""
    if dtype is None:
        return int(library().tps_ce_workspace_bytes(T, V, tp))
    return int(library().tps_ce_workspace_bytes_ex(T, V, tp, _DTYPES[dtype]))


def _ce_call(fn, T, V, tp, dtype, workspace, device):
    """Run fn(workspace) with the given workspace, or with one sized for
    the tensor-core path; operands that take the fp32 path instead are
    refused before any launch (TPS_ERR_WORKSPACE) and run again with the
    full size."""
    if workspace is not None:
        _check(fn(workspace))
        return
    small = ce_workspace_bytes(T, V, tp, dtype)
    ws = torch.empty(max(small, 1), dtype=torch.uint8, device=device)
    rc = fn(ws)
    full = ce_workspace_bytes(T, V, tp)
    if rc == ERR_WORKSPACE and full > small:
        del ws
        rc = fn(torch.empty(max(full, 1), dtype=torch.uint8, device=device))
    _check(rc)


def glu_mlp_workspace_bytes(T: int, d: int, F: int, tp: int, dtype: torch.dtype) -> int:
    return int(library().tps_glu_mlp_workspace_bytes(T, d, F, tp, _DTYPES[dtype]))


def glu_mlp_fwd_bwd(X: torch.Tensor, Wg: torch.Tensor, Wu: torch.Tensor, W2: torch.Tensor, GY: torch.Tensor,
                    tp: int, act: str = "silu", weight_layout: str = "in_out",
                    workspace: Optional[torch.Tensor] = None, out: Optional[Sequence[torch.Tensor]] = None):
    """Gated tensor-parallel MLP (SwiGLU for act="silu") forward + backward.
    Returns fp32 (Y, dX, dWg, dWu, dW2)."""
    _parts(tp, "tp")
    if act not in ACTS or weight_layout not in LAYOUTS:
        raise ValueError("argument")
    d = X.shape[-1]
    T = X.numel() // d if d else 0
    F = Wg.shape[1] if weight_layout == "in_out" else Wg.shape[0]
    dev = X.device
    if out is None:
        out = (torch.empty(X.shape, device=dev, dtype=torch.float32),
               torch.empty(X.shape, device=dev, dtype=torch.float32),
               torch.empty(Wg.shape, device=dev, dtype=torch.float32),
               torch.empty(Wu.shape, device=dev, dtype=torch.float32),
               torch.empty(W2.shape, device=dev, dtype=torch.float32))
    if workspace is None:
        need = glu_mlp_workspace_bytes(T, d, F, tp, X.dtype)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    args = [_tt(t) for t in (X, Wg, Wu, W2, GY, *out)]
    _check(library().tps_glu_mlp_fwd_bwd(*[_ref(a) for a in args[:5]], tp, ACTS[act], LAYOUTS[weight_layout],
                                         *[_ref(a) for a in args[5:]], ctypes.c_void_p(workspace.data_ptr()),
                                         workspace.numel() * workspace.element_size(), _stream(dev)))
    return tuple(out)


def plan_heads(n_heads: int, n_kv_heads: int, tp: int):
    """Head-aligned plan: (q_off [tp+1], kv_first [tp], kv_count, kv_replicas)."""
    _parts(tp, "tp")
    q_off = (ctypes.c_int64 * (tp + 1))()
    kv_first = (ctypes.c_int64 * tp)()
    cnt, rep = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(library().tps_plan_heads(n_heads, n_kv_heads, tp, q_off, kv_first, ctypes.byref(cnt), ctypes.byref(rep)))
    return list(q_off), list(kv_first), int(cnt.value), int(rep.value)


def attn_qkv_fwd(X, Wq, Wk, Wv, n_heads: int, n_kv_heads: int, tp: int, weight_layout: str = "in_out",
                 out_dtype: Optional[torch.dtype] = None, out: Optional[Sequence[torch.Tensor]] = None):
    """(Q, K, V) of the head-split column-parallel projections."""
    _parts(tp, "tp")
    if weight_layout not in LAYOUTS:
        raise ValueError("argument")
    d = X.shape[-1]
    T = X.numel() // d if d else 0
    nq = Wq.shape[1] if weight_layout == "in_out" else Wq.shape[0]
    nkv = Wk.shape[1] if weight_layout == "in_out" else Wk.shape[0]
    dt = out_dtype or X.dtype
    if out is None:
        out = tuple(torch.empty(T, n, device=X.device, dtype=dt) for n in (nq, nkv, nkv))
    args = [_tt(t) for t in (X, Wq, Wk, Wv, *out)]
    _check(library().tps_attn_qkv_fwd(*[_ref(a) for a in args[:4]], n_heads, n_kv_heads, tp, LAYOUTS[weight_layout],
                                      *[_ref(a) for a in args[4:]], _stream(X.device)))
    return tuple(out)


def attn_qkv_bwd(X, Wq, Wk, Wv, dQ, dK, dV, n_heads: int, n_kv_heads: int, tp: int, weight_layout: str = "in_out",
                 out: Optional[Sequence[torch.Tensor]] = None):
    """fp32 (dX, dWq, dWk, dWv)."""
    _parts(tp, "tp")
    if weight_layout not in LAYOUTS:
        raise ValueError("argument")
    dev = X.device
    if out is None:
        out = (torch.empty(X.shape, device=dev, dtype=torch.float32),
               *(torch.empty(w.shape, device=dev, dtype=torch.float32) for w in (Wq, Wk, Wv)))
    args = [_tt(t) for t in (X, Wq, Wk, Wv, dQ, dK, dV, *out)]
    _check(library().tps_attn_qkv_bwd(*[_ref(a) for a in args[:7]], n_heads, n_kv_heads, tp, LAYOUTS[weight_layout],
                                      *[_ref(a) for a in args[7:]], _stream(dev)))
    return tuple(out)


def attn_out_fwd_bwd(C, Wo, GY, n_heads: int, tp: int, weight_layout: str = "in_out",
                     dC_dtype: Optional[torch.dtype] = None, out: Optional[Sequence[torch.Tensor]] = None):
    """(Y fp32, dC, dWo fp32) of the row-parallel output projection."""
    _parts(tp, "tp")
    if weight_layout not in LAYOUTS:
        raise ValueError("argument")
    dev = C.device
    if out is None:
        out = (torch.empty(GY.shape, device=dev, dtype=torch.float32),
               torch.empty(C.shape, device=dev, dtype=dC_dtype or C.dtype),
               torch.empty(Wo.shape, device=dev, dtype=torch.float32))
    args = [_tt(t) for t in (C, Wo, GY, *out)]
    _check(library().tps_attn_out_fwd_bwd(*[_ref(a) for a in args[:3]], n_heads, tp, LAYOUTS[weight_layout],
                                          *[_ref(a) for a in args[3:]], _stream(dev)))
    return tuple(out)


def vocab_ce_fwd_bwd(h: torch.Tensor, Whead: torch.Tensor, labels: torch.Tensor, tp: int,
                     weight_layout: str = "in_out", workspace: Optional[torch.Tensor] = None,
                     out: Optional[Sequence[torch.Tensor]] = None):
    """Vocabulary-sharded cross-entropy forward + backward.  Returns
    (loss fp32 [T], dlogits [T, V] in h's dtype, dHidden fp32 like h,
    owner int32 [T])."""
    _parts(tp, "tp")
    if weight_layout not in LAYOUTS:
        raise ValueError("argument")
    d = h.shape[-1]
    T = h.numel() // d if d else 0
    V = Whead.shape[1] if weight_layout == "in_out" else Whead.shape[0]
    if out is None:
        out = (torch.empty(T, device=h.device, dtype=torch.float32),
               torch.empty(T, V, device=h.device, dtype=h.dtype),
               torch.empty(h.shape, device=h.device, dtype=torch.float32),
               torch.empty(T, device=h.device, dtype=torch.int32))
    loss, dlog, dh, owner = out
    args = [_tt(t) for t in (h, Whead, labels, loss, dlog, dh, owner)]
    _ce_call(lambda ws: library().tps_vocab_ce_fwd_bwd(
        _ref(args[0]), _ref(args[1]), _ref(args[2]), tp, LAYOUTS[weight_layout], *[_ref(a) for a in args[3:]],
        ctypes.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(), _stream(h.device)),
        T, V, tp, h.dtype, workspace, h.device)
    return loss, dlog, dh, owner


def vocab_ce_fwd_bwd_ex(h: torch.Tensor, Whead: torch.Tensor, labels: torch.Tensor, tp: int,
                        weight_layout: str = "in_out", ignore_index: Optional[int] = None, vocab_size: int = 0,
                        reduction: str = "none", denominator: float = 0.0, want_dwhead: bool = False,
                        workspace: Optional[torch.Tensor] = None, out: Optional[Sequence] = None):
    """Cross-entropy with vocabulary padding (the first `vocab_size` columns
    of the head are real, 0 = all), `ignore_index`, a "sum" or "mean"
    reduction (the mean divides by `denominator` when > 0, e.g. the
    job-wide count of supervised tokens, else by this call's count), and
    optionally the head's gradient.  Returns (loss [T], loss_reduced (0-d)
    or None, dlogits, dHidden, dWhead or None, owner); `out` may supply
    those six to write into (loss_reduced and dWhead may be None)."""
    _parts(tp, "tp")
    if weight_layout not in LAYOUTS or reduction not in REDUCTIONS:
        raise ValueError("argument")
    d = h.shape[-1]
    T = h.numel() // d if d else 0
    V = Whead.shape[1] if weight_layout == "in_out" else Whead.shape[0]
    dev = h.device
    if out is not None:
        loss, red, dlog, dh, dw, owner = out
    else:
        loss = torch.empty(T, device=dev, dtype=torch.float32)
        red = torch.zeros((), device=dev, dtype=torch.float32) if reduction != "none" else None
        dlog = torch.empty(T, V, device=dev, dtype=h.dtype)
        dh = torch.empty(h.shape, device=dev, dtype=torch.float32)
        dw = torch.empty(Whead.shape, device=dev, dtype=torch.float32) if want_dwhead else None
        owner = torch.empty(T, device=dev, dtype=torch.int32)
    opts = TpsCeOptions(NO_IGNORE if ignore_index is None else int(ignore_index), int(vocab_size),
                        REDUCTIONS[reduction], 0, float(denominator))
    red_t = _tt(red.reshape(1)) if red is not None else None
    head = [_tt(t) for t in (h, Whead, labels, loss)]
    tail = [_tt(t) for t in (dlog, dh, dw, owner)]
    _ce_call(lambda ws: library().tps_vocab_ce_fwd_bwd_ex(
        _ref(head[0]), _ref(head[1]), _ref(head[2]), tp, LAYOUTS[weight_layout], ctypes.byref(opts), _ref(head[3]),
        _ref(red_t), *[_ref(a) for a in tail], ctypes.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(),
        _stream(dev)), T, V, tp, h.dtype, workspace, dev)
    return loss, red, dlog, dh, dw, owner


def selftest_wait_timeout(limit_ns: int = 50_000_000) -> None:
    """Enqueue the bounded-wait self test (a wait nothing satisfies, given up
    after `limit_ns`); read the outcome with last_device_error()."""
    _check(library().tps_selftest_wait_timeout(int(limit_ns), _stream(None)))


def last_device_error(device=None) -> int:
    """Synchronize the current stream and read + clear the device error word."""
    return int(library().tps_last_device_error(_stream(device)))


class profile:
    """Context manager recording per-launch CUDA events inside the library.

        with profile() as p:
            ...
        p.summary  ->  {"gemm_tc:mlp_dX": dict(launches, ms, flops, bytes), ...}
    """

    def __enter__(self):
        library().tps_profile_reset(1)
        self.summary = {}
        return self

    def __exit__(self, *exc):
        lib = library()
        lib.tps_profile_stop()
        cap = 64
        names = (ctypes.c_char_p * cap)()
        launches = (ctypes.c_int64 * cap)()
        ms, fl, by = (ctypes.c_double * cap)(), (ctypes.c_double * cap)(), (ctypes.c_double * cap)()
        n = lib.tps_profile_summary(cap, names, launches, ms, fl, by)
        if n < 0:
            raise TpsError(-n, "profile summary failed")
        self.summary = {names[i].decode(): dict(launches=int(launches[i]), ms=float(ms[i]), flops=float(fl[i]),
                                                bytes=float(by[i])) for i in range(min(n, cap))}
        self.launches = int(lib.tps_launch_count())
        return False


def launch_count() -> int:
    return int(library().tps_launch_count())


def reset_launch_count():
    library().tps_profile_reset(0)
