"""Float64 CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports it and
it never imports the CUDA library; the only code both sides share is the
seeded input generator module, which holds none of the method's arithmetic.

The arithmetic lives in ``oracle.c`` (plain triple loops in double precision,
one function per definition, each citing the page and section it follows).
This module compiles it with gcc on first use and marshals numpy arrays.

Parity status per function (what pins it is in ``tests/test_oracle_*.py``):
  plan_shards, owner          pinned (worked example + brute force vs numpy)
  matmul                      pinned (numpy matmul, finite differences,
                              torch float64 autograd, sharded == unsharded)
  act, act_grad               pinned (torch gelu/tanh, closed forms, FD)
  mlp_rows, mlp_cols          pinned (finite differences, torch autograd)
  glu_rows, glu_cols          pinned (torch autograd, finite differences,
                              reduction to mlp_* when U = 1, the lesson's
                              per-rank sum)
  plan_heads                  pinned (the lesson's Llama-3-8B head counts
                              for TP = 8 and 16, brute-force invariants)
  attn_qkv, attn_out          pinned (torch autograd, finite differences,
                              the lesson's per-rank column / row split)
  ce_tokens, ce_sharded_one   pinned (closed-form softmax on the worked
                              example's logits, torch cross_entropy, FD)
  ce_ex                       pinned (torch cross_entropy with ignore_index
                              and sum/mean reduction + autograd of h and W,
                              truncated-vocabulary equivalence, ce_tokens)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None

ACT_GELU_ERF, ACT_GELU_TANH, ACT_TANH, ACT_SILU = 0, 1, 2, 3

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc (-O2, OpenMP).

    No fast-math and no FMA contraction, so every product and sum is the
    IEEE double operation the source states."""
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-std=c11", src, "-o", out, "-lm", *extra_flags]
    subprocess.run(cmd, check=True)
    return out


def _declare(lib):
    lib.orc_num_threads.restype = ctypes.c_int
    lib.orc_plan_shards.argtypes = [ctypes.c_int64, ctypes.c_int32, _i64p]
    lib.orc_plan_shards.restype = ctypes.c_int
    lib.orc_owner.argtypes = [ctypes.c_int64, _i64p, ctypes.c_int32]
    lib.orc_owner.restype = ctypes.c_int32
    lib.orc_matmul.argtypes = [ctypes.c_int64] * 3 + [_dp] * 6
    lib.orc_matmul.restype = None
    lib.orc_act.argtypes = [ctypes.c_int, ctypes.c_double]
    lib.orc_act.restype = ctypes.c_double
    lib.orc_act_grad.argtypes = [ctypes.c_int, ctypes.c_double]
    lib.orc_act_grad.restype = ctypes.c_double
    lib.orc_mlp_rows.argtypes = [ctypes.c_int64] * 3 + [_dp] * 4 + [ctypes.c_int, ctypes.c_int64, _i64p, _dp, _dp]
    lib.orc_mlp_rows.restype = None
    lib.orc_mlp_cols.argtypes = [ctypes.c_int64] * 3 + [_dp] * 4 + [ctypes.c_int, ctypes.c_int64, _i64p, _dp, _dp]
    lib.orc_mlp_cols.restype = None
    lib.orc_glu_rows.argtypes = [ctypes.c_int64] * 3 + [_dp] * 5 + [ctypes.c_int, ctypes.c_int64, _i64p, _dp, _dp]
    lib.orc_glu_rows.restype = None
    lib.orc_glu_cols.argtypes = ([ctypes.c_int64] * 3 + [_dp] * 5 + [ctypes.c_int, ctypes.c_int64, _i64p, _dp, _dp,
                                 _dp])
    lib.orc_glu_cols.restype = None
    lib.orc_plan_heads.argtypes = [ctypes.c_int32] * 3 + [_i64p, _i64p, _i32p, _i32p]
    lib.orc_plan_heads.restype = ctypes.c_int
    lib.orc_attn_qkv.argtypes = [ctypes.c_int64] * 4 + [_dp] * 14
    lib.orc_attn_qkv.restype = None
    lib.orc_attn_out.argtypes = [ctypes.c_int64] * 3 + [_dp] * 6
    lib.orc_attn_out.restype = None
    lib.orc_ce_tokens.argtypes = ([ctypes.c_int64] * 3 + [_dp, _dp, _i64p, ctypes.c_int32, ctypes.c_int64, _i64p,
                                  _dp, _dp, _dp, _i32p])
    lib.orc_ce_tokens.restype = ctypes.c_int
    lib.orc_ce_sharded_one.argtypes = [ctypes.c_int64, _dp, ctypes.c_int64, ctypes.c_int32, _dp, _dp, _dp]
    lib.orc_ce_sharded_one.restype = ctypes.c_double
    lib.orc_ce_ex.argtypes = ([ctypes.c_int64] * 3 + [_dp, _dp, _i64p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                              ctypes.c_int, ctypes.c_double, _dp, _dp, _dp, _dp, _dp, _i32p])
    lib.orc_ce_ex.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library.  With ``path`` given,
    load that file instead (used by the mutation tests)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            stale = (not os.path.exists(_LIB_PATH)
                     or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
            if stale:
                compile_oracle()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


class Oracle:
    """numpy-facing wrapper over one loaded copy of the oracle library."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    # -- helpers ---------------------------------------------------------
    @staticmethod
    def _f64(a):
        return np.ascontiguousarray(np.asarray(a, dtype=np.float64))

    @staticmethod
    def _p(a, t=_dp):
        return a.ctypes.data_as(t) if a is not None else None

    def num_threads(self) -> int:
        return int(self.lib.orc_num_threads())

    # -- shard plan ------------------------------------------------------
    def plan_shards(self, dim: int, parts: int) -> np.ndarray:
        off = np.zeros(max(parts, 0) + 1, dtype=np.int64)
        rc = self.lib.orc_plan_shards(dim, parts, self._p(off, _i64p))
        if rc != 0:
            raise ValueError("partition" if rc == 2 else "shape")
        return off

    def owner(self, y: int, off: np.ndarray) -> int:
        off = np.ascontiguousarray(off, dtype=np.int64)
        return int(self.lib.orc_owner(int(y), self._p(off, _i64p), len(off) - 1))

    # -- GEMM ------------------------------------------------------------
    def matmul(self, A, B, G):
        """(Y, dA, dB) of L = <G, AB>, unsharded, float64."""
        A, B, G = self._f64(A), self._f64(B), self._f64(G)
        M, K = A.shape
        K2, N = B.shape
        if K2 != K or G.shape != (M, N):
            raise ValueError("shape")
        Y = np.empty((M, N))
        dA = np.empty((M, K))
        dB = np.empty((K, N))
        self.lib.orc_matmul(M, K, N, self._p(A), self._p(B), self._p(G),
                            self._p(Y), self._p(dA), self._p(dB))
        return Y, dA, dB

    # -- activations -----------------------------------------------------
    def act(self, kind: int, x) -> np.ndarray:
        x = np.asarray(x, dtype=np.float64)
        return np.vectorize(lambda v: self.lib.orc_act(kind, float(v)), otypes=[np.float64])(x)

    def act_grad(self, kind: int, x) -> np.ndarray:
        x = np.asarray(x, dtype=np.float64)
        return np.vectorize(lambda v: self.lib.orc_act_grad(kind, float(v)), otypes=[np.float64])(x)

    # -- MLP (weights in (in, out) layout: W1 d x F, W2 F x d) -------------
    def mlp_rows(self, X, W1, W2, GY, act: int, rows=None):
        X, W1, W2, GY = map(self._f64, (X, W1, W2, GY))
        T, d = X.shape
        F = W1.shape[1]
        rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        Y = np.empty((len(rows), d))
        dX = np.empty((len(rows), d))
        self.lib.orc_mlp_rows(T, d, F, self._p(X), self._p(W1), self._p(W2), self._p(GY), act,
                              len(rows), self._p(rows, _i64p), self._p(Y), self._p(dX))
        return Y, dX

    def mlp_cols(self, X, W1, W2, GY, act: int, cols=None):
        """Returns (dW1[:, cols] as d x ncols, dW2[cols, :] as ncols x d)."""
        X, W1, W2, GY = map(self._f64, (X, W1, W2, GY))
        T, d = X.shape
        F = W1.shape[1]
        cols = np.arange(F, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
        dW1 = np.empty((d, len(cols)))
        dW2 = np.empty((len(cols), d))
        self.lib.orc_mlp_cols(T, d, F, self._p(X), self._p(W1), self._p(W2), self._p(GY), act,
                              len(cols), self._p(cols, _i64p), self._p(dW1), self._p(dW2))
        return dW1, dW2

    def mlp(self, X, W1, W2, GY, act: int):
        """Full (Y, dX, dW1, dW2) with weights in (in, out) layout."""
        Y, dX = self.mlp_rows(X, W1, W2, GY, act)
        dW1, dW2 = self.mlp_cols(X, W1, W2, GY, act)
        return Y, dX, dW1, dW2

    # -- gated MLP (weights (in, out): Wg, Wu d x F, W2 F x d) -------------
    def glu_rows(self, X, Wg, Wu, W2, GY, act: int, rows=None):
        """(Y[rows], dX[rows]) of the gated MLP."""
        X, Wg, Wu, W2, GY = map(self._f64, (X, Wg, Wu, W2, GY))
        T, d = X.shape
        F = Wg.shape[1]
        rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        Y = np.empty((len(rows), d))
        dX = np.empty((len(rows), d))
        self.lib.orc_glu_rows(T, d, F, self._p(X), self._p(Wg), self._p(Wu), self._p(W2), self._p(GY), act,
                              len(rows), self._p(rows, _i64p), self._p(Y), self._p(dX))
        return Y, dX

    def glu_cols(self, X, Wg, Wu, W2, GY, act: int, cols=None):
        """(dWg[:, cols], dWu[:, cols] as d x ncols, dW2[cols, :] as ncols x d)."""
        X, Wg, Wu, W2, GY = map(self._f64, (X, Wg, Wu, W2, GY))
        T, d = X.shape
        F = Wg.shape[1]
        cols = np.arange(F, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
        dWg = np.empty((d, len(cols)))
        dWu = np.empty((d, len(cols)))
        dW2 = np.empty((len(cols), d))
        self.lib.orc_glu_cols(T, d, F, self._p(X), self._p(Wg), self._p(Wu), self._p(W2), self._p(GY), act,
                              len(cols), self._p(cols, _i64p), self._p(dWg), self._p(dWu), self._p(dW2))
        return dWg, dWu, dW2

    def glu(self, X, Wg, Wu, W2, GY, act: int):
        """Full (Y, dX, dWg, dWu, dW2), weights in (in, out) layout."""
        Y, dX = self.glu_rows(X, Wg, Wu, W2, GY, act)
        dWg, dWu, dW2 = self.glu_cols(X, Wg, Wu, W2, GY, act)
        return Y, dX, dWg, dWu, dW2

    # -- attention projections (weights (in, out)) -------------------------
    def plan_heads(self, n_heads: int, n_kv_heads: int, tp: int):
        """(q_off [tp+1], kv_first [tp], kv_count, kv_replicas)."""
        q_off = np.zeros(max(tp, 0) + 1, dtype=np.int64)
        kv_first = np.zeros(max(tp, 1), dtype=np.int64)
        cnt, rep = ctypes.c_int32(0), ctypes.c_int32(0)
        rc = self.lib.orc_plan_heads(n_heads, n_kv_heads, tp, self._p(q_off, _i64p), self._p(kv_first, _i64p),
                                     ctypes.byref(cnt), ctypes.byref(rep))
        if rc != 0:
            raise ValueError("partition")
        return q_off, kv_first[:tp], int(cnt.value), int(rep.value)

    def attn_qkv(self, X, Wq, Wk, Wv, dQ, dK, dV):
        """(Q, K, V, dX, dWq, dWk, dWv)."""
        X, Wq, Wk, Wv, dQ, dK, dV = map(self._f64, (X, Wq, Wk, Wv, dQ, dK, dV))
        T, d = X.shape
        nq, nkv = Wq.shape[1], Wk.shape[1]
        out = [np.empty((T, nq)), np.empty((T, nkv)), np.empty((T, nkv)), np.empty((T, d)),
               np.empty((d, nq)), np.empty((d, nkv)), np.empty((d, nkv))]
        self.lib.orc_attn_qkv(T, d, nq, nkv, *[self._p(a) for a in (X, Wq, Wk, Wv, dQ, dK, dV)],
                              *[self._p(a) for a in out])
        return tuple(out)

    def attn_out(self, C, Wo, GY):
        """(Y, dC, dWo)."""
        C, Wo, GY = map(self._f64, (C, Wo, GY))
        T, nq = C.shape
        d = Wo.shape[1]
        out = [np.empty((T, d)), np.empty((T, nq)), np.empty((nq, d))]
        self.lib.orc_attn_out(T, d, nq, self._p(C), self._p(Wo), self._p(GY), *[self._p(a) for a in out])
        return tuple(out)

    # -- cross-entropy ---------------------------------------------------
    def ce_tokens(self, h, W, labels, parts: int, toks=None):
        """(loss, dlogits, dhidden, owner) for the selected tokens."""
        h, W = self._f64(h), self._f64(W)
        labels = np.ascontiguousarray(labels, dtype=np.int64)
        T, d = h.shape
        V = W.shape[1]
        toks = np.arange(T, dtype=np.int64) if toks is None else np.ascontiguousarray(toks, dtype=np.int64)
        n = len(toks)
        loss = np.empty(n)
        dlog = np.empty((n, V))
        dh = np.empty((n, d))
        own = np.empty(n, dtype=np.int32)
        rc = self.lib.orc_ce_tokens(T, d, V, self._p(h), self._p(W), self._p(labels, _i64p), parts, n,
                                    self._p(toks, _i64p), self._p(loss), self._p(dlog), self._p(dh),
                                    self._p(own, _i32p))
        if rc == 5:
            raise ValueError("label")
        if rc != 0:
            raise ValueError("partition" if rc == 2 else "shape")
        return loss, dlog, dh, own

    def ce_ex(self, h, W, labels, parts: int, ignore_index: int = -(2 ** 63), vocab_real: int = 0,
              reduction: int = 0, denominator: float = 0.0, want_dwhead: bool = True):
        """Cross-entropy with vocabulary padding, ignore_index and a sum / mean
        reduction (reduction 0 none, 1 sum, 2 mean).  Returns (loss [T],
        loss_reduced or None, dlogits [T, V], dhidden [T, d], dwhead [d, V]
        or None, owner [T])."""
        h, W = self._f64(h), self._f64(W)
        labels = np.ascontiguousarray(labels, dtype=np.int64)
        T, d = h.shape
        V = W.shape[1]
        vr = V if vocab_real in (0, None) else vocab_real
        loss = np.empty(T)
        red = np.zeros(1)
        dlog = np.empty((T, V))
        dh = np.empty((T, d))
        dw = np.empty((d, V)) if want_dwhead else None
        own = np.empty(T, dtype=np.int32)
        rc = self.lib.orc_ce_ex(T, d, V, self._p(h), self._p(W), self._p(labels, _i64p), parts, int(ignore_index),
                                int(vr), int(reduction), float(denominator), self._p(loss), self._p(red),
                                self._p(dlog), self._p(dh), self._p(dw), self._p(own, _i32p))
        if rc == 5:
            raise ValueError("label")
        if rc != 0:
            raise ValueError("partition" if rc == 2 else "shape")
        return loss, (float(red[0]) if reduction else None), dlog, dh, dw, own

    def ce_sharded_one(self, z, y: int, parts: int):
        """The pages' per-shard form for one position: (L, m_r, s_r, t_r)."""
        z = self._f64(z)
        m_r, s_r, t_r = np.empty(parts), np.empty(parts), np.empty(parts)
        L = self.lib.orc_ce_sharded_one(len(z), self._p(z), int(y), parts,
                                        self._p(m_r), self._p(s_r), self._p(t_r))
        return float(L), m_r, s_r, t_r


_default = None


def get() -> Oracle:
    """The shared oracle.  ``ORACLE_LIB`` names another build of oracle.c to
    load instead (the mutation tests point it at deliberately broken copies)."""
    global _default
    if _default is None:
        alt = os.environ.get("ORACLE_LIB")
        _default = Oracle(load(alt) if alt else None)
    return _default
