// epilogue.cuh -- per-element epilogue arithmetic shared by the tensor-core
// and SIMT GEMM kernels: plain store, activation forward (pre-activation and
// activation), activation backward (multiply by phi' of the pre-activation),
// and the gated MLP's forms (gate times up, and its backward).
#pragma once
#include <cuda_bf16.h>

#include "internal.cuh"

namespace tps {

__device__ __forceinline__ void store_elem(void* base, int dtype, int64_t idx, float v) {
  if (dtype == TPS_F32)
    static_cast<float*>(base)[idx] = v;
  else
    static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
}

// Store `n` (<= 32) consecutive values of one output row starting at element
// index `idx`; uses 16-byte vector stores when the full run is aligned.
__device__ __forceinline__ void store_run32(void* base, int dtype, int64_t idx, int n, const float (&v)[32]) {
  if (dtype == TPS_F32) {
    float* p = static_cast<float*>(base) + idx;
    if (n == 32 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        reinterpret_cast<float4*>(p)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < n) p[i] = v[i];
    }
  } else {
    __nv_bfloat16* p = static_cast<__nv_bfloat16*>(base) + idx;
    if (n == 32 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 w;
        __nv_bfloat162 b0 = __floats2bfloat162_rn(v[8 * i + 0], v[8 * i + 1]);
        __nv_bfloat162 b1 = __floats2bfloat162_rn(v[8 * i + 2], v[8 * i + 3]);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * i + 4], v[8 * i + 5]);
        __nv_bfloat162 b3 = __floats2bfloat162_rn(v[8 * i + 6], v[8 * i + 7]);
        w.x = *reinterpret_cast<uint32_t*>(&b0);
        w.y = *reinterpret_cast<uint32_t*>(&b1);
        w.z = *reinterpret_cast<uint32_t*>(&b2);
        w.w = *reinterpret_cast<uint32_t*>(&b3);
        reinterpret_cast<uint4*>(p)[i] = w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < n) p[i] = __float2bfloat16_rn(v[i]);
    }
  }
}

__device__ __forceinline__ void load_run32(const float* p, int n, float (&a)[32]) {
  if (n == 32 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(p) + i);
      a[4 * i] = q.x;
      a[4 * i + 1] = q.y;
      a[4 * i + 2] = q.z;
      a[4 * i + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) a[i] = (i < n) ? __ldg(p + i) : 0.0f;
  }
}

// `n` (<= 32) bf16 values from p (zero beyond n) as floats.
__device__ __forceinline__ void load_run32_bf16(const uint16_t* p, int n, float (&a)[32]) {
  if (n == 32 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(p) + i);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        a[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
        a[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) a[i] = (i < n) ? __uint_as_float(static_cast<uint32_t>(__ldg(p + i)) << 16) : 0.0f;
  }
}

// The EPI_ACT_BWD pre-activation of row `row`, columns [col0, col0 + n).
__device__ __forceinline__ void load_pre32(const Epilogue& e, int64_t row, int64_t col0, int n, float (&a)[32]) {
  if (e.aux_bf16 != nullptr)
    load_run32_bf16(e.aux_bf16 + row * e.ld_aux + col0, n, a);
  else
    load_run32(e.aux + row * e.ld_aux + col0, n, a);
}

// Debug builds: does the run of n values of row `row` from column col0 lie
// inside the output?  If not, records TPS_DEVERR_BOUNDS and returns false
// (the caller skips the store).  Release builds compile this to `true`.
__device__ __forceinline__ bool dbg_store_ok(const Epilogue& e, int64_t row, int64_t col0, int64_t n) {
#if TPS_DEBUG
  if (row < 0 || row >= e.dbg_rows || col0 < 0 || col0 + n > e.dbg_cols) {
    if (e.dbg_err != nullptr) atomicOr(e.dbg_err, TPS_DEVERR_BOUNDS);
    return false;
  }
#else
  (void)e;
  (void)row;
  (void)col0;
  (void)n;
#endif
  return true;
}

// Apply the epilogue to 32 consecutive accumulator values of row `row`,
// columns [col0, col0 + n).
__device__ __forceinline__ void epilogue_run32(const Epilogue& e, int64_t row, int64_t col0, int n,
                                               float (&v)[32]) {
  if (!dbg_store_ok(e, row, col0, n)) return;
  if (e.mode == EPI_STORE || e.mode == EPI_CE_STATS) {
    store_run32(e.d, e.d_dtype, row * e.ldd + col0, n, v);
  } else if (e.mode == EPI_ACT_FWD) {
    if (e.d != nullptr) store_run32(e.d, e.d_dtype, row * e.ldd + col0, n, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = act_fwd(e.act, v[i]);
    store_run32(e.d2, e.d2_dtype, row * e.ldd2 + col0, n, v);
  } else if (e.mode == EPI_GLU_UP) {
    if (e.d != nullptr) store_run32(e.d, TPS_F32, row * e.ldd + col0, n, v);
    float a[32];
    load_run32(e.aux + row * e.ld_aux + col0, n, a);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] *= act_fwd(e.act, a[i]);
    store_run32(e.d2, e.d2_dtype, row * e.ldd2 + col0, n, v);
  } else {
    float a[32];
    load_pre32(e, row, col0, n, a);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] *= act_grad(e.act, a[i]);
    store_run32(e.d, e.d_dtype, row * e.ldd + col0, n, v);
  }
}

// EPI_GLU_BWD without TMA stores (kept apart from epilogue_run32 so that
// the kernels which never run it do not carry its registers).
__device__ __forceinline__ void epilogue_glu_bwd_run32(const Epilogue& e, int64_t row, int64_t col0, int n,
                                                       float (&v)[32]) {
  if (!dbg_store_ok(e, row, col0, n)) return;
  float hg[32], u[32];
  load_run32(e.aux + row * e.ld_aux + col0, n, hg);
  load_run32(e.aux2 + row * e.ld_aux2 + col0, n, u);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float f, g;
    act_fwd_grad(e.act, hg[i], f, g);
    const float da = v[i];
    v[i] = da * u[i] * g;
    u[i] = da * f;
  }
  store_run32(e.d, e.d_dtype, row * e.ldd + col0, n, v);
  store_run32(e.d2, e.d2_dtype, row * e.ldd2 + col0, n, u);
}

// EPI_GLU_FWD without TMA stores: `hg` and `u` are the gate and up
// accumulators of the same 32 columns.
__device__ __forceinline__ void epilogue_glu_run32(const Epilogue& e, int64_t row, int64_t col0, int n,
                                                   float (&hg)[32], float (&u)[32]) {
  if (!dbg_store_ok(e, row, col0, n)) return;
  store_run32(e.d, TPS_F32, row * e.ldd + col0, n, hg);
  store_run32(e.d3, TPS_F32, row * e.ldd3 + col0, n, u);
#pragma unroll
  for (int i = 0; i < 32; ++i) u[i] *= act_fwd(e.act, hg[i]);
  store_run32(e.d2, e.d2_dtype, row * e.ldd2 + col0, n, u);
}

// Scalar form used by the SIMT kernel.
__device__ __forceinline__ void epilogue_elem(const Epilogue& e, int64_t row, int64_t col, float v) {
  if (!dbg_store_ok(e, row, col, 1)) return;
  if (e.mode == EPI_STORE || e.mode == EPI_CE_STATS) {
    store_elem(e.d, e.d_dtype, row * e.ldd + col, v);
  } else if (e.mode == EPI_ACT_FWD) {
    if (e.d != nullptr) store_elem(e.d, e.d_dtype, row * e.ldd + col, v);
    store_elem(e.d2, e.d2_dtype, row * e.ldd2 + col, act_fwd(e.act, v));
  } else if (e.mode == EPI_GLU_UP) {
    if (e.d != nullptr) store_elem(e.d, TPS_F32, row * e.ldd + col, v);
    store_elem(e.d2, e.d2_dtype, row * e.ldd2 + col, v * act_fwd(e.act, e.aux[row * e.ld_aux + col]));
  } else if (e.mode == EPI_GLU_BWD) {
    float f, g;
    act_fwd_grad(e.act, e.aux[row * e.ld_aux + col], f, g);
    store_elem(e.d, e.d_dtype, row * e.ldd + col, v * e.aux2[row * e.ld_aux2 + col] * g);
    store_elem(e.d2, e.d2_dtype, row * e.ldd2 + col, v * f);
  } else {
    const int64_t i = row * e.ld_aux + col;
    const float pre = e.aux_bf16 != nullptr ? __uint_as_float(static_cast<uint32_t>(e.aux_bf16[i]) << 16) : e.aux[i];
    store_elem(e.d, e.d_dtype, row * e.ldd + col, v * act_grad(e.act, pre));
  }
}

}  // namespace tps
