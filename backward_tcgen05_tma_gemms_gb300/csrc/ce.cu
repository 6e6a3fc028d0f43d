// ce.cu -- vocabulary-sharded cross-entropy core: per-shard statistics,
// their combination into the global log-sum-exp, the loss and the logits
// gradient ("多卡张量：拆开计算，再合回同一结果", section 04 / VOCABULARY
// SHARDS).  The logits z come from the logits GEMM (T x V fp32).
//
// One-read path (ce_cluster_kernel): a thread-block cluster per token, one
// CTA per logical rank.  CTA r stages its shard of the token's logits in
// shared memory (one HBM read), computes m_r = max z and
// s_r = sum e^{z - m_r} over the shard, publishes (m_r, s_r) in its shared
// memory; after a cluster barrier every CTA reads all ranks' pairs through
// distributed shared memory -- the on-chip form of the pages' all-reduce of
// the per-shard max and sum -- combines them into m = max_r m_r and
// s = sum_r s_r e^{m_r - m}, and writes its shard of
// dlogits = e^{z - m}/s - 1[j = y] from shared memory.  The rank whose
// shard holds the label writes loss = log s + m - z_y and the owner index.
//
// Two-pass path (ce_stats_kernel + ce_grad_kernel) for plans the cluster
// cannot hold (more than 8 ranks or a shard larger than shared memory):
// the statistics go through a workspace and z is read twice.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "internal.cuh"
#include "ptx.cuh"

namespace tps {

constexpr int CE_THREADS = 512;
constexpr int CE_MAX_CLUSTER = 8;
// Largest shard (fp32 elements) the cluster path stages in shared memory.
constexpr int64_t CE_MAX_SHARD = 48 * 1024;

struct CeParams {
  int64_t T, V;
  int32_t parts;
  const float* z;
  int64_t ldz;
  const void* labels;
  int label_is_i64;
  float* loss;
  void* dlog;
  int64_t ldg;
  int32_t* owner;
  float* stats;
  float* zy;
  uint32_t* err;
};

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ int64_t load_label(const CeParams& p, int64_t t) {
  return p.label_is_i64 ? static_cast<const int64_t*>(p.labels)[t]
                        : static_cast<int64_t>(static_cast<const int32_t*>(p.labels)[t]);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block-wide reductions; `red` holds one float per warp.  All threads
// receive the result.
__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float r = (l < nw) ? red[l] : -INFINITY;
  return warp_max(r);
}
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float r = (l < nw) ? red[l] : 0.0f;
  return warp_sum(r);
}

template <typename TOut>
__device__ __forceinline__ void store_grad(TOut* p, float v) {
  if constexpr (sizeof(TOut) == 4)
    __stcs(reinterpret_cast<float*>(p), v);
  else
    *p = __float2bfloat16_rn(v);
}

// ------------------------------------------------------------ one-read path
template <typename TOut>
__global__ void __launch_bounds__(CE_THREADS) ce_cluster_kernel(const CeParams p) {
  extern __shared__ float4 zs4[];
  float* zs = reinterpret_cast<float*>(zs4);
  __shared__ float red[32];
  __shared__ float stat[2];  // (m_r, s_r) published to the cluster
  __shared__ float comb[2];  // combined (m, s)

  const uint32_t r = cluster_ctarank();  // logical rank == shard index
  const int64_t t = blockIdx.y;
  const int64_t beg = shard_offset(p.V, p.parts, r);
  const int64_t len = shard_offset(p.V, p.parts, r + 1) - beg;
  const float* zrow = p.z + t * p.ldz + beg;

  // Stage the shard in shared memory with 16-byte loads: `head` scalars
  // reach a 16-byte boundary; `shift` places that boundary on a float4
  // boundary of zs.
  const int64_t head = imin64(len, (4 - ((reinterpret_cast<uintptr_t>(zrow) >> 2) & 3)) & 3);
  const int64_t shift = (4 - head) & 3;
  const int64_t body4 = (len - head) / 4;
  float mx = -INFINITY;
  for (int64_t j = threadIdx.x; j < head; j += blockDim.x) {
    const float v = __ldcs(zrow + j);
    zs[shift + j] = v;
    mx = fmaxf(mx, v);
  }
  const float4* z4 = reinterpret_cast<const float4*>(zrow + head);
  float4* s4 = reinterpret_cast<float4*>(zs + shift + head);
  for (int64_t j = threadIdx.x; j < body4; j += blockDim.x) {
    const float4 v = __ldcs(z4 + j);
    s4[j] = v;
    mx = fmaxf(fmaxf(mx, v.x), fmaxf(v.y, fmaxf(v.z, v.w)));
  }
  for (int64_t j = head + 4 * body4 + threadIdx.x; j < len; j += blockDim.x) {
    const float v = __ldcs(zrow + j);
    zs[shift + j] = v;
    mx = fmaxf(mx, v);
  }
  const float m_r = block_max(mx, red);
  float se = 0.0f;
  if (len > 0) {
    for (int64_t j = threadIdx.x; j < len; j += blockDim.x) se += __expf(zs[shift + j] - m_r);
  }
  const float s_r = block_sum(se, red);

  if (threadIdx.x == 0) {
    stat[0] = m_r;  // -inf for an empty shard
    stat[1] = s_r;  // 0 for an empty shard
  }
  cluster_sync();  // publish (m_r, s_r) to the other ranks

  const int64_t y = load_label(p, t);
  const bool valid = (y >= 0 && y < p.V);
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    for (int q = 0; q < p.parts; ++q) m = fmaxf(m, ld_cluster_f32(cluster_map(smem_u32(&stat[0]), q)));
    float s = 0.0f;
    for (int q = 0; q < p.parts; ++q) {
      const float mq = ld_cluster_f32(cluster_map(smem_u32(&stat[0]), q));
      const float sq = ld_cluster_f32(cluster_map(smem_u32(&stat[1]), q));
      if (sq > 0.0f) s += sq * __expf(mq - m);
    }
    comb[0] = m;
    comb[1] = s;
    if (valid && y >= beg && y < beg + len) {
      p.loss[t] = logf(s) + m - zs[shift + (y - beg)];
      if (p.owner) p.owner[t] = static_cast<int32_t>(r);
    } else if (!valid && r == 0) {
      p.loss[t] = __int_as_float(0x7fc00000);  // NaN
      if (p.owner) p.owner[t] = -1;
      atomicOr(p.err, TPS_DEVERR_LABEL);
    }
  }
  __syncthreads();
  const float m = comb[0];
  const float inv_s = 1.0f / comb[1];
  TOut* grow = static_cast<TOut*>(p.dlog) + t * p.ldg + beg;
  const int64_t yl = (valid && y >= beg && y < beg + len) ? (y - beg) : -1;
  if constexpr (sizeof(TOut) == 2) {
    // Pairs of bf16 (4-byte stores) once the row is 4-byte aligned.
    const int64_t h2 = imin64(len, (reinterpret_cast<uintptr_t>(grow) >> 1) & 1);
    for (int64_t j = threadIdx.x; j < h2; j += blockDim.x)
      store_grad(grow + j, __expf(zs[shift + j] - m) * inv_s - (j == yl ? 1.0f : 0.0f));
    const int64_t npair = (len - h2) / 2;
    __nv_bfloat162* g2 = reinterpret_cast<__nv_bfloat162*>(grow + h2);
    for (int64_t j = threadIdx.x; j < npair; j += blockDim.x) {
      const int64_t e = h2 + 2 * j;
      const float g0 = __expf(zs[shift + e] - m) * inv_s - (e == yl ? 1.0f : 0.0f);
      const float g1 = __expf(zs[shift + e + 1] - m) * inv_s - (e + 1 == yl ? 1.0f : 0.0f);
      g2[j] = __floats2bfloat162_rn(g0, g1);
    }
    for (int64_t j = h2 + 2 * npair + threadIdx.x; j < len; j += blockDim.x)
      store_grad(grow + j, __expf(zs[shift + j] - m) * inv_s - (j == yl ? 1.0f : 0.0f));
  } else {
    for (int64_t j = threadIdx.x; j < len; j += blockDim.x)
      store_grad(grow + j, __expf(zs[shift + j] - m) * inv_s - (j == yl ? 1.0f : 0.0f));
  }
  cluster_sync();  // no CTA leaves while another may still read its `stat`
}

// Register-resident variant of the one-read path for shards of up to
// CE_THREADS * 4 * VPT4 elements (plus an unaligned head and tail of at most
// three each): every thread issues all of its 16-byte loads before using
// any, so a CTA keeps its whole shard (64 KB at V=128256, P=8) in flight,
// and the slice never touches shared memory.
template <typename TOut, int VPT4>
__global__ void __launch_bounds__(CE_THREADS) ce_cluster_reg_kernel(const CeParams p) {
  __shared__ float red[32];
  __shared__ float stat[2];
  __shared__ float comb[2];

  const uint32_t r = cluster_ctarank();
  const int64_t t = blockIdx.y;
  const int64_t beg = shard_offset(p.V, p.parts, r);
  const int64_t len = shard_offset(p.V, p.parts, r + 1) - beg;
  const float* zrow = p.z + t * p.ldz + beg;
  const int tid = threadIdx.x;

  const int64_t head = imin64(len, (4 - ((reinterpret_cast<uintptr_t>(zrow) >> 2) & 3)) & 3);
  const int64_t body4 = (len - head) / 4;
  const int64_t tail0 = head + 4 * body4;  // first tail element
  const float4* z4 = reinterpret_cast<const float4*>(zrow + head);

  float4 v[VPT4];
#pragma unroll
  for (int k = 0; k < VPT4; ++k) {
    const int64_t j = tid + static_cast<int64_t>(k) * CE_THREADS;
    v[k] = (j < body4) ? __ldcs(z4 + j) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
  // at most 3 head and 3 tail scalars, held by threads 0..5
  float e = -INFINITY;
  int64_t e_idx = -1;
  if (tid < head) {
    e_idx = tid;
  } else if (tid >= 3 && tid - 3 < len - tail0) {
    e_idx = tail0 + (tid - 3);
  }
  if (e_idx >= 0) e = __ldcs(zrow + e_idx);

  float mx = e;
#pragma unroll
  for (int k = 0; k < VPT4; ++k) mx = fmaxf(mx, fmaxf(fmaxf(v[k].x, v[k].y), fmaxf(v[k].z, v[k].w)));
  const float m_r = block_max(mx, red);
  float se = 0.0f;
  if (len > 0) {
    // exp(-inf - m_r) = 0 for the padding slots
#pragma unroll
    for (int k = 0; k < VPT4; ++k)
      se += __expf(v[k].x - m_r) + __expf(v[k].y - m_r) + __expf(v[k].z - m_r) + __expf(v[k].w - m_r);
    if (e_idx >= 0) se += __expf(e - m_r);
  }
  const float s_r = block_sum(se, red);
  if (tid == 0) {
    stat[0] = m_r;
    stat[1] = s_r;
  }
  cluster_sync();

  const int64_t y = load_label(p, t);
  const bool valid = (y >= 0 && y < p.V);
  const int64_t yl = (valid && y >= beg && y < beg + len) ? (y - beg) : -1;
  if (tid == 0) {
    float m = -INFINITY;
    for (int q = 0; q < p.parts; ++q) m = fmaxf(m, ld_cluster_f32(cluster_map(smem_u32(&stat[0]), q)));
    float s = 0.0f;
    for (int q = 0; q < p.parts; ++q) {
      const float mq = ld_cluster_f32(cluster_map(smem_u32(&stat[0]), q));
      const float sq = ld_cluster_f32(cluster_map(smem_u32(&stat[1]), q));
      if (sq > 0.0f) s += sq * __expf(mq - m);
    }
    comb[0] = m;
    comb[1] = s;
    if (!valid && r == 0) {
      p.loss[t] = __int_as_float(0x7fc00000);  // NaN
      if (p.owner) p.owner[t] = -1;
      atomicOr(p.err, TPS_DEVERR_LABEL);
    }
  }
  __syncthreads();
  const float m = comb[0];
  const float s = comb[1];
  const float inv_s = 1.0f / s;
  // the owner rank's thread holding z_y writes the loss
  if (yl >= 0) {
    float zy = 0.0f;
    bool mine = false;
    if (yl == e_idx) {
      zy = e;
      mine = true;
    } else if (yl >= head && yl < tail0) {
      const int64_t q4 = (yl - head) >> 2;
      if (q4 % CE_THREADS == tid) {
        const int64_t slot = q4 / CE_THREADS;
        float4 w = v[0];
#pragma unroll
        for (int k = 1; k < VPT4; ++k)
          if (k == slot) w = v[k];  // static register indexing
        const int c = static_cast<int>((yl - head) & 3);
        zy = c == 0 ? w.x : (c == 1 ? w.y : (c == 2 ? w.z : w.w));
        mine = true;
      }
    }
    if (mine) {
      p.loss[t] = logf(s) + m - zy;
      if (p.owner) p.owner[t] = static_cast<int32_t>(r);
    }
  }

  TOut* grow = static_cast<TOut*>(p.dlog) + t * p.ldg + beg;
  auto g = [&](float x, int64_t idx) { return __expf(x - m) * inv_s - (idx == yl ? 1.0f : 0.0f); };
  if (e_idx >= 0) store_grad(grow + e_idx, g(e, e_idx));
  const bool vec_ok = (reinterpret_cast<uintptr_t>(grow + head) & (4 * sizeof(TOut) - 1)) == 0;
#pragma unroll
  for (int k = 0; k < VPT4; ++k) {
    const int64_t j = tid + static_cast<int64_t>(k) * CE_THREADS;
    if (j < body4) {
      const int64_t i0 = head + 4 * j;
      const float g0 = g(v[k].x, i0), g1 = g(v[k].y, i0 + 1), g2 = g(v[k].z, i0 + 2), g3 = g(v[k].w, i0 + 3);
      if (vec_ok) {
        if constexpr (sizeof(TOut) == 2) {
          __nv_bfloat162 a = __floats2bfloat162_rn(g0, g1), b = __floats2bfloat162_rn(g2, g3);
          uint2 w;
          w.x = *reinterpret_cast<uint32_t*>(&a);
          w.y = *reinterpret_cast<uint32_t*>(&b);
          __stcs(reinterpret_cast<uint2*>(grow + i0), w);
        } else {
          __stcs(reinterpret_cast<float4*>(grow + i0), make_float4(g0, g1, g2, g3));
        }
      } else {
        store_grad(grow + i0, g0);
        store_grad(grow + i0 + 1, g1);
        store_grad(grow + i0 + 2, g2);
        store_grad(grow + i0 + 3, g3);
      }
    }
  }
  cluster_sync();  // no CTA leaves while another may still read its `stat`
}

// ------------------------------------------------------------ two-pass path
// Grid (parts, T): rank r's (m_r, s_r) for token t with an online max/sum
// (one read of the shard), the label's logit and owner.
__global__ void __launch_bounds__(256) ce_stats_kernel(const CeParams p) {
  __shared__ float red_m[32], red_s[32];
  const int32_t r = blockIdx.x;
  const int64_t t = blockIdx.y;
  const int64_t beg = shard_offset(p.V, p.parts, r);
  const int64_t end = shard_offset(p.V, p.parts, r + 1);
  const float* zrow = p.z + t * p.ldz;
  float m = -INFINITY, s = 0.0f;
  for (int64_t j = beg + threadIdx.x; j < end; j += blockDim.x) {
    const float v = zrow[j];
    if (v > m) {
      s = s * __expf(m - v) + 1.0f;
      m = v;
    } else {
      s += __expf(v - m);
    }
  }
  // combine (m, s) pairs: warp then block
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, o);
    const float so = __shfl_xor_sync(0xffffffffu, s, o);
    const float mn = fmaxf(m, mo);
    s = (s > 0.0f ? s * __expf(m - mn) : 0.0f) + (so > 0.0f ? so * __expf(mo - mn) : 0.0f);
    m = mn;
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    red_m[w] = m;
    red_s[w] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY, S = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) M = fmaxf(M, red_m[i]);
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i)
      if (red_s[i] > 0.0f) S += red_s[i] * __expf(red_m[i] - M);
    p.stats[(t * p.parts + r) * 2 + 0] = M;
    p.stats[(t * p.parts + r) * 2 + 1] = S;
    const int64_t y = load_label(p, t);
    const bool valid = (y >= 0 && y < p.V);
    if (valid && y >= beg && y < end) {
      p.zy[t] = zrow[y];
      if (p.owner) p.owner[t] = r;
    } else if (!valid && r == 0) {
      p.zy[t] = __int_as_float(0x7fc00000);
      if (p.owner) p.owner[t] = -1;
      atomicOr(p.err, TPS_DEVERR_LABEL);
    }
  }
}

constexpr int64_t CE_GRAD_CHUNK = 8192;

// Grid (ceil(V / chunk), T): combines the token's per-rank statistics and
// writes one chunk of the gradient row (second read of z); chunk 0 writes
// the loss.
template <typename TOut>
__global__ void __launch_bounds__(256) ce_grad_kernel(const CeParams p) {
  __shared__ float comb[2];
  const int64_t t = blockIdx.y;
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    for (int q = 0; q < p.parts; ++q) m = fmaxf(m, p.stats[(t * p.parts + q) * 2]);
    float s = 0.0f;
    for (int q = 0; q < p.parts; ++q) {
      const float sq = p.stats[(t * p.parts + q) * 2 + 1];
      if (sq > 0.0f) s += sq * __expf(p.stats[(t * p.parts + q) * 2] - m);
    }
    comb[0] = m;
    comb[1] = s;
    if (blockIdx.x == 0) p.loss[t] = logf(s) + m - p.zy[t];  // NaN propagates for a bad label
  }
  __syncthreads();
  const float m = comb[0], inv_s = 1.0f / comb[1];
  const int64_t y = load_label(p, t);
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * CE_GRAD_CHUNK;
  const int64_t c1 = imin64(p.V, c0 + CE_GRAD_CHUNK);
  const float* zrow = p.z + t * p.ldz;
  TOut* grow = static_cast<TOut*>(p.dlog) + t * p.ldg;
  for (int64_t j = c0 + threadIdx.x; j < c1; j += blockDim.x)
    store_grad(grow + j, __expf(zrow[j] - m) * inv_s - (j == y ? 1.0f : 0.0f));
}

// ------------------------------------------------------------ host
bool ce_cluster_supported(int64_t V, int32_t parts, int /*dlogits_dtype*/) {
  if (parts < 1 || parts > CE_MAX_CLUSTER) return false;
  const int64_t max_len = (V + parts - 1) / parts;
  return max_len <= CE_MAX_SHARD;
}

template <typename TOut, int VPT4>
static cudaError_t launch_cluster_reg(const CeParams& p, cudaLaunchConfig_t cfg) {
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, ce_cluster_reg_kernel<TOut, VPT4>, p);
}

template <typename TOut>
static int launch_cluster(const CeParams& p, cudaStream_t stream) {
  const int64_t max_len = (p.V + p.parts - 1) / p.parts;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.parts), static_cast<unsigned>(p.T), 1);
  cfg.blockDim = dim3(CE_THREADS, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.parts);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const double bytes = double(p.T) * double(p.V) * (4.0 + sizeof(TOut)) + double(p.T) * (8.0 + 4.0);
  ProfScope prof("ce_cluster", "ce_core", 0.0, bytes, stream);
  cudaError_t e;
  // body capacity of the register kernel: CE_THREADS * 4 * VPT4 elements
  if (max_len <= CE_THREADS * 4 * 2) {
    e = launch_cluster_reg<TOut, 2>(p, cfg);
  } else if (max_len <= CE_THREADS * 4 * 4) {
    e = launch_cluster_reg<TOut, 4>(p, cfg);
  } else if (max_len <= CE_THREADS * 4 * 8) {
    e = launch_cluster_reg<TOut, 8>(p, cfg);
  } else {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
      attr_err = cudaFuncSetAttribute(ce_cluster_kernel<TOut>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>((CE_MAX_SHARD + 4) * sizeof(float)));
    });
    if (attr_err != cudaSuccess) return TPS_ERR_CUDA;
    cfg.dynamicSmemBytes = static_cast<size_t>(max_len + 4) * sizeof(float);
    e = cudaLaunchKernelEx(&cfg, ce_cluster_kernel<TOut>, p);
  }
  note_launch();
  return e == cudaSuccess ? TPS_OK : TPS_ERR_CUDA;
}

template <typename TOut>
static int launch_two_pass(const CeParams& p, cudaStream_t stream) {
  {
    ProfScope prof("ce_stats", "ce_core", 0.0, double(p.T) * double(p.V) * 4.0, stream);
    ce_stats_kernel<<<dim3(static_cast<unsigned>(p.parts), static_cast<unsigned>(p.T)), 256, 0, stream>>>(p);
    note_launch();
  }
  if (cudaPeekAtLastError() != cudaSuccess) return TPS_ERR_CUDA;
  {
    const int64_t chunks = (p.V + CE_GRAD_CHUNK - 1) / CE_GRAD_CHUNK;
    ProfScope prof("ce_grad", "ce_core", 0.0, double(p.T) * double(p.V) * (4.0 + sizeof(TOut)), stream);
    ce_grad_kernel<TOut><<<dim3(static_cast<unsigned>(chunks), static_cast<unsigned>(p.T)), 256, 0, stream>>>(p);
    note_launch();
  }
  return cudaPeekAtLastError() == cudaSuccess ? TPS_OK : TPS_ERR_CUDA;
}

int launch_ce(const CeDesc& c, uint32_t* dev_err, cudaStream_t stream, bool* used_cluster) {
  CeParams p;
  p.T = c.T;
  p.V = c.V;
  p.parts = c.parts;
  p.z = c.logits;
  p.ldz = c.ldz;
  p.labels = c.labels;
  p.label_is_i64 = (c.label_dtype == TPS_I64);
  p.loss = c.loss;
  p.dlog = c.dlogits;
  p.ldg = c.ldg;
  p.owner = c.owner;
  p.stats = c.stats;
  p.zy = c.zy;
  p.err = dev_err;
  const bool cl = ce_cluster_supported(c.V, c.parts, c.dlogits_dtype);
  if (used_cluster) *used_cluster = cl;
  const size_t gsize = (c.dlogits_dtype == TPS_F32) ? 4 : 2;
  // Tokens go on grid.y (at most 65535 per launch): process slabs.
  for (int64_t t0 = 0; t0 < c.T; t0 += 65535) {
    CeParams q = p;
    q.T = imin64(65535, c.T - t0);
    q.z = p.z + t0 * p.ldz;
    q.labels = p.label_is_i64 ? static_cast<const void*>(static_cast<const int64_t*>(p.labels) + t0)
                              : static_cast<const void*>(static_cast<const int32_t*>(p.labels) + t0);
    q.loss = p.loss + t0;
    q.dlog = static_cast<char*>(p.dlog) + t0 * p.ldg * gsize;
    q.owner = p.owner ? p.owner + t0 : nullptr;
    q.stats = p.stats ? p.stats + t0 * p.parts * 2 : nullptr;
    q.zy = p.zy ? p.zy + t0 : nullptr;
    int rc;
    if (cl)
      rc = (c.dlogits_dtype == TPS_F32) ? launch_cluster<float>(q, stream) : launch_cluster<__nv_bfloat16>(q, stream);
    else
      rc = (c.dlogits_dtype == TPS_F32) ? launch_two_pass<float>(q, stream)
                                        : launch_two_pass<__nv_bfloat16>(q, stream);
    if (rc != TPS_OK) return rc;
  }
  return TPS_OK;
}

}  // namespace tps
