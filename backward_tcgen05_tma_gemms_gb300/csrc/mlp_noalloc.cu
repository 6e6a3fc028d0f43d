// mlp_noalloc.cu -- tps_mlp_fwd_bwd_noalloc: the tensor-parallel MLP forward
// and backward for callers that cannot allocate device memory.
//
// tps_mlp_fwd_bwd needs a caller-provided workspace (pre-activation,
// activation and dZ, T x F each).  Some callers have no way to obtain one:
// code that runs under a framework or server that owns all device memory
// through its own allocator and forbids side allocations, or code on a
// latency-critical path that must not call cudaMalloc because of its implicit
// device synchronization.  This entry point takes its scratch from a
// file-scope static device array instead, so it allocates nothing.
//
// The array is TPS_MLP_NOALLOC_SCRATCH_BYTES long.  The driver places it on
// a device when the library's device code is loaded there: with lazy module
// loading (the CUDA default) that happens in the first call on the device,
// which can synchronize; from then on the device holds the array until the
// process exits.  Every call on a device shares it, and it keeps the
// previous call's contents; the MLP overwrites each scratch byte before
// reading it, so nothing needs clearing.  Calls whose execution overlaps on
// the GPU (other streams, other host threads) race on the array and must be
// serialised by the caller.
#include <cuda_runtime.h>

#include <cstdio>

#include "internal.cuh"
#include "tps.h"

namespace {

static __device__ __align__(256) unsigned char g_mlp_noalloc_scratch[TPS_MLP_NOALLOC_SCRATCH_BYTES];

// In host code the array's name is only a host-side stand-in; the device
// address comes from cudaGetSymbolAddress with the device current.  It is
// looked up on every call (a table lookup once the module is loaded), so an
// address never outlives the context it belongs to.
int scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_mlp_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) return TPS_ERR_CUDA;
  *out = p;
  return TPS_OK;
}

}  // namespace

extern "C" int tps_mlp_fwd_bwd_noalloc(const tps_tensor* X, const tps_tensor* W1, const tps_tensor* W2,
                                       const tps_tensor* GY, int32_t tp, int32_t act, int32_t weight_layout,
                                       const tps_tensor* Y, const tps_tensor* dX, const tps_tensor* dW1,
                                       const tps_tensor* dW2, void* cuda_stream) {
  // Size check first, on the host, before any CUDA call.
  if (X != nullptr && W1 != nullptr && X->ndim >= 2 && X->ndim <= 4 && W1->ndim == 2) {
    const int64_t d = X->shape[X->ndim - 1];
    int64_t T = 1;
    for (int i = 0; i < X->ndim - 1; ++i) T *= X->shape[i];
    const int64_t F = (weight_layout == TPS_W_OUT_IN) ? W1->shape[0] : W1->shape[1];
    const size_t need = tps_mlp_workspace_bytes(T, d, F, tp, X->dtype);
    if (need > static_cast<size_t>(TPS_MLP_NOALLOC_SCRATCH_BYTES)) {
      char msg[256];
      snprintf(msg, sizeof(msg),
               "tps_mlp_fwd_bwd_noalloc: T=%lld x F=%lld needs %zu bytes of scratch; the static scratch holds %zu",
               (long long)T, (long long)F, need, static_cast<size_t>(TPS_MLP_NOALLOC_SCRATCH_BYTES));
      tps::set_error_detail(msg);
      return TPS_ERR_WORKSPACE;
    }
  }
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != TPS_OK) {
    tps::set_error_detail("tps_mlp_fwd_bwd_noalloc: cudaGetSymbolAddress of the static scratch failed");
    return rc;
  }
  return tps_mlp_fwd_bwd(X, W1, W2, GY, tp, act, weight_layout, Y, dX, dW1, dW2, scratch,
                         static_cast<size_t>(TPS_MLP_NOALLOC_SCRATCH_BYTES), cuda_stream);
}
