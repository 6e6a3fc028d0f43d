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
// cannot hold (more than 8 ranks or a shard larger than shared memory), and
// for the extended form (vocabulary padding, ignore_index, reductions): the
// statistics go through a workspace and z is read twice.
//
// Extended form: columns [vreal, V) are padding -- outside every max and
// sum, gradient 0; a label equal to ignore_index gives loss 0, gradient 0,
// owner -1 and is not counted; the gradient is scaled by 1 / D for a mean
// (ce_finalize_kernel forms D and the reduced loss).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
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
  // the logits GEMM's CE-statistics epilogue: bf16 logits relative to the
  // shift of their 128-column tile (leading dimension ldz), the shifts
  // (T x n_tiles) and, in zy, the fp32 logit at each label
  const __nv_bfloat16* z16;
  const float* zshift;
  int64_t shift_ld;  // row stride of zshift
  int64_t n_tiles;
  const void* labels;
  int label_is_i64;
  float* loss;
  void* dlog;
  int64_t ldg;
  int32_t* owner;
  float* stats;
  float* zy;
  uint32_t* err;
  int64_t ignore_index;  // TPS_NO_IGNORE: every label is supervised
  int64_t vreal;         // columns [vreal, V) are vocabulary padding
  const float* scale;    // gradient scale 1 / D (nullptr: 1)
  int32_t* count;        // supervised labels are counted here (nullable)
};

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ int64_t load_label(const CeParams& p, int64_t t) {
  return p.label_is_i64 ? static_cast<const int64_t*>(p.labels)[t]
                        : static_cast<int64_t>(static_cast<const int32_t*>(p.labels)[t]);
}

// 0: a supervised label in [0, vreal); 1: ignore_index; 2: invalid.
__device__ __forceinline__ int label_kind(const CeParams& p, int64_t y) {
  if (p.ignore_index != TPS_NO_IGNORE && y == p.ignore_index) return 1;
  return (y >= 0 && y < p.vreal) ? 0 : 2;
}
__device__ __forceinline__ float grad_scale(const CeParams& p) { return p.scale ? *p.scale : 1.0f; }

// Debug builds: does a store of n dlogits of token t from column col (n = 0:
// token t's loss, owner or statistics) lie inside the outputs?  If not,
// records TPS_DEVERR_BOUNDS and returns false (the caller skips the store).
// Release builds compile this to `true`.
__device__ __forceinline__ bool ce_dbg_ok(const CeParams& p, int64_t t, int64_t col, int64_t n) {
#if TPS_DEBUG
  if (t < 0 || t >= p.T || col < 0 || col + n > p.V) {
    atomicOr(p.err, TPS_DEVERR_BOUNDS);
    return false;
  }
#else
  (void)p;
  (void)t;
  (void)col;
  (void)n;
#endif
  return true;
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

// ------------------------------------------------------------ persistent path
// Persistent clusters fed by a ring of bulk copies.  Cluster c handles
// tokens c, c + C, c + 2C, ...; CTA r of the cluster owns shard r.  Thread
// 0 keeps CEP_NBUF bulk copies (cp.async.bulk, one token's shard each) in
// flight, so HBM reads continue while the CTA reduces, exchanges and writes
// the previous token.  The shard goes from shared memory to registers once;
// the exponentials e_j = exp(z_j - m_r) computed for s_r are reused for the
// gradient, which is e_j * exp(m_r - m) / s - 1[j = y].
constexpr int CEP_THREADS = 512;
constexpr int CEP_NBUF = 3;
constexpr int CEP_VPT4 = 8;                                  // float4 slots per thread
constexpr int CEP_BUF_FLOATS = CEP_THREADS * 4 * CEP_VPT4;  // 16384 floats = 64 KB
constexpr int CEP_CHUNK_BYTES = 16384;                       // bulk copy granule

struct CepGeom {  // one rank's slice, identical for every token
  int64_t beg, end;  // shard columns [beg, end)
  int64_t a0;        // beg rounded down to 4: first column copied to smem
  int64_t a1;        // end rounded down to 4: end of the bulk copy
  int64_t tail0;     // first column loaded from global by threads (< 4 of them)
};

__device__ __forceinline__ CepGeom cep_geom(int64_t V, int32_t parts, int64_t r) {
  CepGeom g;
  g.beg = shard_offset(V, parts, r);
  g.end = shard_offset(V, parts, r + 1);
  g.a0 = g.beg & ~int64_t(3);
  g.a1 = g.end & ~int64_t(3);
  if (g.a1 < g.a0) g.a1 = g.a0;
  g.tail0 = g.beg > g.a1 ? g.beg : g.a1;
  return g;
}

__device__ __forceinline__ void cep_issue(const CeParams& p, const CepGeom& g, int64_t t, float* buf,
                                          uint64_t* bar) {
  const uint32_t bytes = static_cast<uint32_t>((g.a1 - g.a0) * 4);
  mbar_expect_tx(bar, bytes);
  const char* src = reinterpret_cast<const char*>(p.z + t * p.ldz + g.a0);
  char* dst = reinterpret_cast<char*>(buf);
  for (uint32_t off = 0; off < bytes; off += CEP_CHUNK_BYTES) {
    const uint32_t n = bytes - off < CEP_CHUNK_BYTES ? bytes - off : CEP_CHUNK_BYTES;
    bulk_load(dst + off, src + off, n, bar);
  }
}

constexpr float kLog2e = 1.4426950408889634f;

// e^{x - m} as 2^{x log2(e) - m log2(e)}: one FMA and one ex2.
__device__ __forceinline__ float exp_shift(float x, float m_l2e) { return ex2_approx(fmaf(x, kLog2e, -m_l2e)); }

// (m, s) <- statistics of the union of (m, s) and (m2, s2), each a (max,
// sum of e^{z - max}) pair; (-inf, 0) is the empty set.
__device__ __forceinline__ void ms_combine_acc(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  s = (m == -INFINITY ? 0.0f : s * ex2_approx((m - M) * kLog2e)) +
      (m2 == -INFINITY ? 0.0f : s2 * ex2_approx((m2 - M) * kLog2e));
  m = M;
}

// Combine per-thread (max, sum of e^{z - max}) pairs over the block: first
// the maximum, then the sums rescaled to it.  One __syncthreads: every warp
// then reduces the per-warp partials itself.  `red` holds 64 floats and must
// not be reused before every thread has returned (callers alternate two).
// Returns the block's (m, s); an empty block gives (-inf, 0).
__device__ __forceinline__ float2 block_ms(float mt, float st, float* red) {
  float m = mt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float sl = (mt == -INFINITY) ? 0.0f : st * ex2_approx((mt - m) * kLog2e);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sl += __shfl_xor_sync(0xffffffffu, sl, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (l == 0) {
    red[w] = m;
    red[32 + w] = sl;
  }
  __syncthreads();
  const float m2 = (l < nw) ? red[l] : -INFINITY;
  float M = m2;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float s2 = (m2 == -INFINITY) ? 0.0f : red[32 + l] * ex2_approx((m2 - M) * kLog2e);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
  return make_float2(M, s2);
}

// One token's shard in registers: e_j = exp(z_j - mt) with the thread's own
// maximum mt (0 for padding), and the CTA's (m_r, s_r).
struct CepTok {
  float4 v[CEP_VPT4];
  float tail;
  float mt;
  float m_r, s_r;
};

struct CepCtx {  // per-CTA constants of the persistent CE kernel
  int64_t c, C, n_iter;
  CepGeom g;
  int h0, h1, ntail, q_first, q_last;
  bool has_body, vec_store;
  uint32_t r;
};

struct CepSmem {
  uint64_t full[CEP_NBUF];
  float red[2][64];                     // block_ms partials, alternating per token
  __align__(8) float stat_in[2][8][2];  // [token parity][rank] (m_q, s_q), written by rank q
  uint32_t abort_flag;
};

// Load token i (ring buffer i % NBUF) into registers, compute the
// statistics, and refill the buffer with token i + NBUF.
__device__ __forceinline__ void cep_load_stats(const CeParams& p, const CepCtx& x, int64_t i, CepTok& k, float* ring,
                                               CepSmem& sm) {
  const int tid = threadIdx.x;
  const int64_t t = x.c + i * x.C;
  const int b = static_cast<int>(i % CEP_NBUF);
  float tail_v = -INFINITY;
  if (tid < x.ntail) tail_v = __ldcs(p.z + t * p.ldz + x.g.tail0 + tid);
  const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  if (x.has_body) {
    mbar_wait(&sm.full[b], static_cast<uint32_t>((i / CEP_NBUF) & 1), &sm.abort_flag, p.err);
    const float4* buf4 = reinterpret_cast<const float4*>(ring + b * CEP_BUF_FLOATS);
#pragma unroll
    for (int j = 0; j < CEP_VPT4; ++j) {
      const int q = tid + j * CEP_THREADS;
      float4 w = (q <= x.q_last) ? buf4[q] : ninf;
      if (q == x.q_first) {  // the slot holding the shard's first element
        const int e0 = 4 * q;
        if (e0 + 0 < x.h0) w.x = -INFINITY;
        if (e0 + 1 < x.h0) w.y = -INFINITY;
        if (e0 + 2 < x.h0) w.z = -INFINITY;
        if (e0 + 3 < x.h0) w.w = -INFINITY;
      }
      k.v[j] = w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < CEP_VPT4; ++j) k.v[j] = ninf;
  }
  float mt = tail_v;
#pragma unroll
  for (int j = 0; j < CEP_VPT4; ++j) mt = fmaxf(fmaxf(mt, fmaxf(k.v[j].x, k.v[j].y)), fmaxf(k.v[j].z, k.v[j].w));
  float st = 0.0f;
  if (mt != -INFINITY) {
    const float ml = mt * kLog2e;
#pragma unroll
    for (int j = 0; j < CEP_VPT4; ++j) {
      k.v[j].x = exp_shift(k.v[j].x, ml);
      k.v[j].y = exp_shift(k.v[j].y, ml);
      k.v[j].z = exp_shift(k.v[j].z, ml);
      k.v[j].w = exp_shift(k.v[j].w, ml);
      st += (k.v[j].x + k.v[j].y) + (k.v[j].z + k.v[j].w);
    }
    k.tail = exp_shift(tail_v, ml);
    st += k.tail;
  } else {
#pragma unroll
    for (int j = 0; j < CEP_VPT4; ++j) k.v[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    k.tail = 0.0f;
  }
  k.mt = mt;
  // block_ms's barrier also certifies that buffer b has been read by all
  const float2 ms = block_ms(mt, st, sm.red[i & 1]);
  k.m_r = ms.x;
  k.s_r = ms.y;
  if (tid == 0 && x.has_body && i + CEP_NBUF < x.n_iter) {
    fence_async_smem();
    cep_issue(p, x.g, x.c + (i + CEP_NBUF) * x.C, ring + b * CEP_BUF_FLOATS, &sm.full[b]);
  }
}

// Push the CTA's (m_r, s_r) for token parity `par` into every rank's
// stat_in[par][r] (remote shared-memory stores), then arrive on the
// cluster barrier; the stores are ordered before the arrive by a fence.
__device__ __forceinline__ void cep_publish(const CeParams& p, const CepCtx& x, int par, const CepTok& k,
                                            CepSmem& sm) {
  if (threadIdx.x < p.parts) {
    st_cluster_f32x2(cluster_map(smem_u32(&sm.stat_in[par][x.r][0]), threadIdx.x), k.m_r, k.s_r);
    fence_cluster();
  }
  cluster_arrive_relaxed();
}

// One pipeline step: statistics of token i+1 (overlapping the barrier of
// token i), then the combine, loss and gradient of token i.
template <typename TOut>
__device__ __forceinline__ void cep_step(const CeParams& p, const CepCtx& x, int64_t i, CepTok& cur, CepTok& nxt,
                                         float* ring, CepSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t t = x.c + i * x.C;
  const int64_t y = load_label(p, t);
  const bool valid = (y >= 0 && y < p.V);
  const bool owner = valid && y >= x.g.beg && y < x.g.end;
  float zy = 0.0f;
  if (tid == 0 && owner) zy = p.z[t * p.ldz + y];
  const bool has_next = i + 1 < x.n_iter;
  if (has_next) cep_load_stats(p, x, i + 1, nxt, ring, sm);
  cluster_wait();  // every rank's statistics of token t are in stat_in
  const int par = static_cast<int>(i & 1);
  // every warp combines the ranks' (m_q, s_q) itself: no block barrier
  const float mq = (lane < p.parts) ? sm.stat_in[par][lane][0] : -INFINITY;
  const float sq = (lane < p.parts) ? sm.stat_in[par][lane][1] : 0.0f;
  float m = mq;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = (mq == -INFINITY) ? 0.0f : sq * ex2_approx((mq - m) * kLog2e);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (tid == 0) {
    if (owner) {
      p.loss[t] = logf(s) + m - zy;
      if (p.owner) p.owner[t] = static_cast<int32_t>(x.r);
    } else if (!valid && x.r == 0) {
      p.loss[t] = __int_as_float(0x7fc00000);  // NaN
      if (p.owner) p.owner[t] = -1;
      atomicOr(p.err, TPS_DEVERR_LABEL);
    }
  }
  // dlogits_j = e^{z_j - m}/s - 1[j = y] = e_j * e^{mt - m}/s - 1[j = y]
  const float f = (cur.mt != -INFINITY) ? ex2_approx((cur.mt - m) * kLog2e) / s : 0.0f;
  const int yl = owner ? static_cast<int>(y - x.g.a0) : -1;  // smem-local index of the label
  const int qy = (yl >= 0 && yl < x.h1) ? (yl >> 2) : -1;
  TOut* gbase = static_cast<TOut*>(p.dlog) + t * p.ldg + x.g.a0;  // element 0 = smem index 0
  if (tid < x.ntail) {
    const int il = x.h1 + tid;  // tail elements follow the body
    store_grad(gbase + il, cur.tail * f - (il == yl ? 1.0f : 0.0f));
  }
#pragma unroll
  for (int j = 0; j < CEP_VPT4; ++j) {
    const int q = tid + j * CEP_THREADS;
    if (q > x.q_last) continue;
    float g0 = cur.v[j].x * f, g1 = cur.v[j].y * f, g2 = cur.v[j].z * f, g3 = cur.v[j].w * f;
    if (q == qy) {
      const int cpt = yl & 3;
      g0 -= (cpt == 0) ? 1.0f : 0.0f;
      g1 -= (cpt == 1) ? 1.0f : 0.0f;
      g2 -= (cpt == 2) ? 1.0f : 0.0f;
      g3 -= (cpt == 3) ? 1.0f : 0.0f;
    }
    const int i0 = 4 * q;
    if (x.vec_store && q != x.q_first) {
      if constexpr (sizeof(TOut) == 2) {
        __nv_bfloat162 a = __floats2bfloat162_rn(g0, g1), bb = __floats2bfloat162_rn(g2, g3);
        uint2 w;
        w.x = *reinterpret_cast<uint32_t*>(&a);
        w.y = *reinterpret_cast<uint32_t*>(&bb);
        __stcs(reinterpret_cast<uint2*>(gbase + i0), w);
      } else {
        __stcs(reinterpret_cast<float4*>(gbase + i0), make_float4(g0, g1, g2, g3));
      }
    } else {
      if (i0 + 0 >= x.h0) store_grad(gbase + i0, g0);
      if (i0 + 1 >= x.h0) store_grad(gbase + i0 + 1, g1);
      if (i0 + 2 >= x.h0) store_grad(gbase + i0 + 2, g2);
      if (i0 + 3 >= x.h0) store_grad(gbase + i0 + 3, g3);
    }
  }
  // Every rank read stat_in[par ^ 1] (token i-1) before arriving at the
  // barrier just waited on, so the next token's values may land there now.
  if (has_next) cep_publish(p, x, par ^ 1, nxt, sm);
}

template <typename TOut>
__global__ void __launch_bounds__(CEP_THREADS, 1) ce_persistent_kernel(const CeParams p) {
  extern __shared__ float4 cep_smem4[];
  float* ring = reinterpret_cast<float*>(cep_smem4);
  __shared__ CepSmem sm;

  CepCtx x;
  x.r = cluster_ctarank();
  x.c = blockIdx.y;
  x.C = gridDim.y;
  x.g = cep_geom(p.V, p.parts, x.r);
  x.h0 = static_cast<int>(x.g.beg - x.g.a0);
  x.h1 = static_cast<int>(x.g.tail0 - x.g.a0);
  x.ntail = static_cast<int>(x.g.end - x.g.tail0);
  x.has_body = x.g.a1 > x.g.a0;
  x.q_first = x.has_body ? (x.h0 >> 2) : -1;
  x.q_last = x.has_body ? ((x.h1 - 1) >> 2) : -1;
  x.n_iter = (p.T - x.c + x.C - 1) / x.C;
  x.vec_store = ((p.ldg & 3) == 0) && ((reinterpret_cast<uintptr_t>(p.dlog) & (4 * sizeof(TOut) - 1)) == 0);
  const int tid = threadIdx.x;

  if (tid == 0) {
    for (int b = 0; b < CEP_NBUF; ++b) mbar_init(&sm.full[b], 1);
    sm.abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync();  // every CTA of the cluster is running before any DSMEM access
  if (tid == 0 && x.has_body)
    for (int64_t i = 0; i < CEP_NBUF && i < x.n_iter; ++i)
      cep_issue(p, x.g, x.c + i * x.C, ring + i * CEP_BUF_FLOATS, &sm.full[i]);

  CepTok A, B;  // two register sets, alternating roles without copies
  if (x.n_iter > 0) {
    cep_load_stats(p, x, 0, A, ring, sm);
    cep_publish(p, x, 0, A, sm);  // phase 0
  }
  for (int64_t i = 0; i < x.n_iter; i += 2) {
    cep_step<TOut>(p, x, i, A, B, ring, sm);
    if (i + 1 < x.n_iter) cep_step<TOut>(p, x, i + 1, B, A, ring, sm);
  }
  // Every issued copy was waited for above; after a timed-out wait, make
  // sure none is still landing before shared memory is released.
  if (tid == 0 && x.has_body)
    for (int64_t j = x.n_iter > CEP_NBUF ? x.n_iter - CEP_NBUF : 0; j < x.n_iter; ++j)
      mbar_wait_drain(&sm.full[j % CEP_NBUF], static_cast<uint32_t>((j / CEP_NBUF) & 1), p.err);
  cluster_sync();  // no CTA leaves while another may still write into its stat_in
}

// ------------------------------------------------------------ two-pass path
// Grid (parts, T): rank r's (m_r, s_r) for token t with an online max/sum
// (one read of the shard), the label's logit and owner.
__global__ void __launch_bounds__(256) ce_stats_kernel(const CeParams p) {
  __shared__ float red_m[32], red_s[32];
  const int32_t r = blockIdx.x;
  const int64_t t = blockIdx.y;
  const int64_t beg = shard_offset(p.V, p.parts, r);
  const int64_t end = imin64(shard_offset(p.V, p.parts, r + 1), p.vreal);  // padding stays out
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
    const int kind = label_kind(p, y);
    if (kind == 0 && y >= beg && y < end) {
      p.zy[t] = zrow[y];
      if (p.owner) p.owner[t] = r;
      if (p.count) atomicAdd(p.count, 1);
    } else if (kind == 1 && r == 0) {
      p.zy[t] = 0.0f;
      if (p.owner) p.owner[t] = -1;
    } else if (kind == 2 && r == 0) {
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
    if (blockIdx.x == 0)  // NaN propagates for a bad label
      p.loss[t] = label_kind(p, load_label(p, t)) == 1 ? 0.0f : logf(s) + m - p.zy[t];
  }
  __syncthreads();
  const int64_t y = load_label(p, t);
  const bool ignored = label_kind(p, y) == 1;
  const float sc = grad_scale(p);
  const float m = comb[0], inv_s = ignored ? 0.0f : sc / comb[1], hot = ignored ? 0.0f : sc;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * CE_GRAD_CHUNK;
  const int64_t c1 = imin64(p.V, c0 + CE_GRAD_CHUNK);
  const float* zrow = p.z + t * p.ldz;
  TOut* grow = static_cast<TOut*>(p.dlog) + t * p.ldg;
  for (int64_t j = c0 + threadIdx.x; j < c1; j += blockDim.x)
    store_grad(grow + j, j < p.vreal ? __expf(zrow[j] - m) * inv_s - (j == y ? hot : 0.0f) : 0.0f);
}

// One block: the divisor D of a mean (the caller's denominator if > 0,
// else the number of supervised labels, at least 1; D = 1 for a sum), the
// gradient scale 1 / D, and the reduced loss sum_t loss_t / D.
__global__ void __launch_bounds__(1024) ce_finalize_kernel(const float* loss, int64_t T, const int32_t* count,
                                                           int reduction, double denominator, float* scale,
                                                           float* loss_reduced) {
  __shared__ double red[32];
  double D = 1.0;
  if (reduction == TPS_REDUCE_MEAN) D = denominator > 0.0 ? denominator : (*count > 0 ? double(*count) : 1.0);
  if (scale != nullptr && threadIdx.x == 0) *scale = static_cast<float>(1.0 / D);
  if (loss_reduced == nullptr) return;
  double acc = 0.0;
  for (int64_t t = threadIdx.x; t < T; t += blockDim.x) acc += loss[t];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double total = 0.0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) total += red[w];
    *loss_reduced = static_cast<float>(total / D);
  }
}

// ------------------------------------------------------------ from tile statistics
// The logits GEMM's epilogue left, per (token, 128-column tile), the
// statistics of the tile's columns in the shard of its first column, and
// per (token, shard) the statistics of the part of the tile in which the
// shard starts, when that is not a tile boundary.  Shard r's (m_r, s_r)
// combines the tiles whose first column lies in r and, when r starts inside
// a tile, that tile's part in r.

constexpr int CEF_TOK_PER_BLOCK = 8;  // one warp per token

__global__ void __launch_bounds__(32 * CEF_TOK_PER_BLOCK) ce_combine_kernel(const CeParams p, const float* ts,
                                                                          int64_t n_tiles, float* ms) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * CEF_TOK_PER_BLOCK + w;
  if (t >= p.T) return;
  const float2* row = reinterpret_cast<const float2*>(ts) + t * n_tiles;
  const float2* row_b = reinterpret_cast<const float2*>(p.stats) + t * p.parts;
  float m = -INFINITY, s = 0.0f;  // running global combine (identical in all lanes)
  for (int32_t r = 0; r < p.parts; ++r) {
    const int64_t beg = shard_offset(p.V, p.parts, r), end = shard_offset(p.V, p.parts, r + 1);
    const int64_t t0 = beg / kStatsTileN, t1 = (end - 1) / kStatsTileN;
    float mr = -INFINITY, sr = 0.0f;
    for (int64_t tt = t0 + lane; tt <= t1; tt += 32) {
      const float2 e = (tt == t0 && beg % kStatsTileN != 0) ? row_b[r] : row[tt];
      ms_combine_acc(mr, sr, e.x, e.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      ms_combine_acc(mr, sr, __shfl_xor_sync(0xffffffffu, mr, o), __shfl_xor_sync(0xffffffffu, sr, o));
    ms_combine_acc(m, s, mr, sr);  // the pages' combine across shards
  }
  if (lane == 0 && ce_dbg_ok(p, t, 0, 0)) {
    const int64_t y = load_label(p, t);
    const int kind = label_kind(p, y);
    // an ignored token gets (m, 1/s) = (+inf, 0): every e^{z - m} / s is 0
    reinterpret_cast<float2*>(ms)[t] = kind == 1 ? make_float2(INFINITY, 0.0f) : make_float2(m, 1.0f / s);
    if (kind == 1) {
      p.loss[t] = 0.0f;
      if (p.owner) p.owner[t] = -1;
    } else if (kind == 0) {
      p.loss[t] = logf(s) + m - p.zy[t];
      if (p.owner) {
        int32_t r = 0;
        while (r + 1 < p.parts && shard_offset(p.V, p.parts, r + 1) <= y) ++r;
        p.owner[t] = r;
      }
      if (p.count) atomicAdd(p.count, 1);
    } else {
      p.loss[t] = __int_as_float(0x7fc00000);  // NaN
      if (p.owner) p.owner[t] = -1;
      atomicOr(p.err, TPS_DEVERR_LABEL);
    }
  }
}

constexpr int CEF_THREADS = 256;
constexpr int CEF_VEC = 4;                                 // 16-byte loads (8 logits) per thread per item
constexpr int64_t CEF_ITEM = CEF_THREADS * 8 * CEF_VEC;   // 8192 columns

// The two bf16 values packed in a 32-bit word, low half first, as floats.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// dlogits = e^{z - m}/s - 1[j = y], streamed over (token, 8192-column item)
// work items by a persistent grid sized to the blocks that fit at once.
// The logits arrive as bf16 z~ = z - c, relative to the shift c of their
// 128-column statistics tile, so e^{z - m} = 2^{z~ log2(e) + (c - m) log2(e)}
// (one FMA and one ex2 per element).  The loads are software-pipelined:
// each thread issues the next item's 16-byte loads before the exponentials
// and stores of the current one, so HBM reads stay in flight through the
// arithmetic.
template <typename TOut>
__global__ void __launch_bounds__(CEF_THREADS) ce_grad_stream_kernel(const CeParams p, const float* ms) {
  const int64_t per_row = (p.V + CEF_ITEM - 1) / CEF_ITEM;
  const int64_t items = p.T * per_row;
  const bool vec = ((p.ldz & 7) == 0) && ((p.ldg & 7) == 0) &&
                   ((reinterpret_cast<uintptr_t>(p.z16) & 15u) == 0) &&
                   ((reinterpret_cast<uintptr_t>(p.dlog) & 15u) == 0);
  const float sc = grad_scale(p);
  struct Item {
    uint4 z[CEF_VEC];   // 8 bf16 logits (relative to their tile's shift) per load
    float c[CEF_VEC];   // the shift of each load's tile
  };
  auto load_item = [&](int64_t it, Item& w) {
    const int64_t t = it / per_row;
    const int64_t c0 = (it - t * per_row) * CEF_ITEM;
    const __nv_bfloat16* zrow = p.z16 + t * p.ldz;
    const unsigned short* zbits = reinterpret_cast<const unsigned short*>(zrow);
    const float* crow = p.zshift + t * p.shift_ld;
#pragma unroll
    for (int k = 0; k < CEF_VEC; ++k) {
      const int64_t e = c0 + 8 * (threadIdx.x + k * CEF_THREADS);
      w.c[k] = (e < p.V) ? crow[e / kStatsTileN] : 0.0f;
      if (vec && e + 7 < p.V) {
        w.z[k] = __ldcs(reinterpret_cast<const uint4*>(zrow + e));
      } else {
        uint32_t q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t lo = (e + 2 * j < p.V) ? zbits[e + 2 * j] : 0u;
          const uint32_t hi = (e + 2 * j + 1 < p.V) ? zbits[e + 2 * j + 1] : 0u;
          q[j] = lo | (hi << 16);
        }
        w.z[k] = make_uint4(q[0], q[1], q[2], q[3]);
      }
    }
  };
  Item v;
  if (blockIdx.x < items) load_item(blockIdx.x, v);
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    const int64_t t = it / per_row;
    const int64_t c0 = (it - t * per_row) * CEF_ITEM;
    const float2 mi = reinterpret_cast<const float2*>(ms)[t];
    const float ml = mi.x * kLog2e, inv = mi.y * sc;
    const int64_t y0 = load_label(p, t);
    const int64_t y = label_kind(p, y0) == 1 ? -1 : y0;  // an ignored row has no one-hot
    TOut* grow = static_cast<TOut*>(p.dlog) + t * p.ldg;
    Item nv;
    if (it + gridDim.x < items) load_item(it + gridDim.x, nv);
#pragma unroll
    for (int k = 0; k < CEF_VEC; ++k) {
      const int64_t e = c0 + 8 * (threadIdx.x + k * CEF_THREADS);
      if (e >= p.V) continue;
      const float adj = fmaf(v.c[k], kLog2e, -ml);  // (c - m) log2(e)
      const uint32_t wd[4] = {v.z[k].x, v.z[k].y, v.z[k].z, v.z[k].w};
      float g[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        g[2 * j] = ex2_approx(fmaf(bf16_lo(wd[j]), kLog2e, adj)) * inv;
        g[2 * j + 1] = ex2_approx(fmaf(bf16_hi(wd[j]), kLog2e, adj)) * inv;
      }
      if (y >= e && y < e + 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] -= (y == e + j) ? sc : 0.0f;
      }
      if (e + 7 >= p.vreal) {  // vocabulary padding
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = (e + j < p.vreal) ? g[j] : 0.0f;
      }
      if (!ce_dbg_ok(p, t, e, imin64(8, p.V - e))) continue;
      if (vec && e + 7 < p.V) {
        if constexpr (sizeof(TOut) == 2) {
          uint32_t q[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 b = __floats2bfloat162_rn(g[2 * j], g[2 * j + 1]);
            q[j] = *reinterpret_cast<uint32_t*>(&b);
          }
          __stcs(reinterpret_cast<uint4*>(grow + e), make_uint4(q[0], q[1], q[2], q[3]));
        } else {
          __stcs(reinterpret_cast<float4*>(grow + e), make_float4(g[0], g[1], g[2], g[3]));
          __stcs(reinterpret_cast<float4*>(grow + e + 4), make_float4(g[4], g[5], g[6], g[7]));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (e + j < p.V) store_grad(grow + e + j, g[j]);
      }
    }
    v = nv;
  }
}

// ------------------------------------------------------------ fused combine + stream
// One persistent kernel for the whole CE core when the shifted bf16 logits
// rows are 16-byte aligned.  Work items are (token, 8192-column chunk) in
// row-major order, and block b takes the contiguous range
// [b I / G, (b + 1) I / G) of the I items (G blocks), so it meets a short run
// of consecutive rows.  Three roles:
//   producer (one thread)   bulk-copies each item's 16 KB of logits and its
//                           64 tile shifts into a ring of CFS_STAGES stages
//   combiner (one warp)     for each row of the range, in order: the pages'
//                           per-shard (m_r, s_r) from the tile statistics of
//                           the logits GEMM, their combine into m and s, and,
//                           in the block that holds the row's first item,
//                           the loss and the owner; (m, scale / s) and the
//                           one-hot column go to a ring of CFS_ROWS rows
//   consumers (8 warps)     dlogits = e^{z - m} scale / s - scale 1[j = y]
//                           from the staged logits, 16-byte streaming stores
// The combiner runs up to CFS_ROWS rows ahead, so the statistics of the
// next rows are read while the current ones stream, and the separate
// combine launch (and its pass over the statistics) disappears.
constexpr int CFS_CONSUMERS = 8;
constexpr int CFS_THREADS = 32 * (CFS_CONSUMERS + 2);
constexpr int64_t CFS_CHUNK = 8192;                                  // columns per item
constexpr int CFS_SHIFTS = static_cast<int>(CFS_CHUNK / kStatsTileN);  // 64
// Six stages of 16 KB at two blocks per SM (98 KB of shared memory each):
// measured 0.674-0.677 ms at T=8192, V=128256 against 0.720-0.723 ms with
// four stages at three blocks per SM, and 0.87 ms with eight at one.
constexpr int CFS_STAGES = 6;
constexpr int CFS_ROWS = 4;
static_assert(CFS_CHUNK == 8 * 4 * 32 * CFS_CONSUMERS, "each consumer thread takes four 8-column vectors per item");

struct CfsShared {
  uint16_t z[CFS_STAGES][CFS_CHUNK];   // shifted bf16 logits of one item per stage
  float c[CFS_STAGES][CFS_SHIFTS];     // the item's tile shifts
  float2 row_ms[CFS_ROWS];             // (m log2 e, scale / s); ignored rows (+inf, 0)
  long long row_y[CFS_ROWS];           // one-hot column (-1: none)
  uint64_t full[CFS_STAGES], empty[CFS_STAGES], row_full[CFS_ROWS], row_empty[CFS_ROWS];
  uint32_t abort;
};

template <typename TOut>
__global__ void __launch_bounds__(CFS_THREADS) ce_fused_stream_kernel(const CeParams p, const float* ts) {
  extern __shared__ __align__(128) uint8_t cfs_raw[];
  CfsShared& sh = *reinterpret_cast<CfsShared*>(cfs_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t per_row = (p.V + CFS_CHUNK - 1) / CFS_CHUNK;
  const int64_t items = p.T * per_row;
  const int64_t it0 = items * blockIdx.x / gridDim.x, it1 = items * (blockIdx.x + 1) / gridDim.x;
  if (threadIdx.x == 0) {
    for (int i = 0; i < CFS_STAGES; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], CFS_CONSUMERS);
    }
    for (int i = 0; i < CFS_ROWS; ++i) {
      mbar_init(&sh.row_full[i], 1);
      mbar_init(&sh.row_empty[i], CFS_CONSUMERS);
    }
    sh.abort = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  if (it0 >= it1) return;
  const float sc = grad_scale(p);

  if (warp == CFS_CONSUMERS) {
    // ---------------------------------------------------- producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      for (int64_t it = it0; it < it1; ++it) {
        if (!mbar_wait(&sh.empty[stage], phase ^ 1u, &sh.abort, p.err)) break;
        const int64_t t = it / per_row, c0 = (it - t * per_row) * CFS_CHUNK;
        const int64_t n = imin64(CFS_CHUNK, p.V - c0);          // a multiple of 8
        const int64_t nt = ((n + kStatsTileN - 1) / kStatsTileN + 3) & ~int64_t(3);
        const uint32_t zb = static_cast<uint32_t>(n * 2), cb = static_cast<uint32_t>(nt * 4);
        mbar_expect_tx(&sh.full[stage], zb + cb);
        bulk_load(sh.z[stage], p.z16 + t * p.ldz + c0, zb, &sh.full[stage]);
        bulk_load(sh.c[stage], p.zshift + t * p.shift_ld + c0 / kStatsTileN, cb, &sh.full[stage]);
        ++issued;
        if (++stage == CFS_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // the copies still in flight land before the block may exit
      const int64_t first = issued > CFS_STAGES ? issued - CFS_STAGES : 0;
      for (int64_t i = first; i < issued; ++i)
        mbar_wait_drain(&sh.full[i % CFS_STAGES], static_cast<uint32_t>((i / CFS_STAGES) & 1), p.err);
    }
  } else if (warp == CFS_CONSUMERS + 1) {
    // ---------------------------------------------------- combiner
    const int64_t t_first = it0 / per_row, t_last = (it1 - 1) / per_row;
    uint32_t slot = 0, phase = 0;
    for (int64_t t = t_first; t <= t_last; ++t) {
      if (!mbar_wait(&sh.row_empty[slot], phase ^ 1u, &sh.abort, p.err)) break;
      const float2* row = reinterpret_cast<const float2*>(ts) + t * p.n_tiles;
      const float2* row_b = reinterpret_cast<const float2*>(p.stats) + t * p.parts;
      float m = -INFINITY, s = 0.0f;
      for (int32_t r = 0; r < p.parts; ++r) {
        const int64_t beg = shard_offset(p.V, p.parts, r), end = shard_offset(p.V, p.parts, r + 1);
        const int64_t t0 = beg / kStatsTileN, t1 = (end - 1) / kStatsTileN;
        const bool split0 = beg % kStatsTileN != 0;  // shard r starts inside tile t0: its part in r
        float mr = -INFINITY, sr = 0.0f;
        for (int64_t tt = t0 + lane; tt <= t1; tt += 4 * 32) {
          float2 e[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int64_t u = tt + 32 * k;
            e[k] = u > t1 ? make_float2(-INFINITY, 0.0f) : ((u == t0 && split0) ? row_b[r] : __ldg(row + u));
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) ms_combine_acc(mr, sr, e[k].x, e[k].y);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
          ms_combine_acc(mr, sr, __shfl_xor_sync(0xffffffffu, mr, o), __shfl_xor_sync(0xffffffffu, sr, o));
        ms_combine_acc(m, s, mr, sr);  // the pages' combine across shards
      }
      if (lane == 0) {
        const int64_t y = load_label(p, t);
        const int kind = label_kind(p, y);
        sh.row_ms[slot] = kind == 1 ? make_float2(INFINITY, 0.0f) : make_float2(m * kLog2e, sc / s);
        sh.row_y[slot] = kind == 1 ? -1 : y;
        if (t * per_row >= it0 && ce_dbg_ok(p, t, 0, 0)) {  // this block holds the row's first item
          if (kind == 1) {
            p.loss[t] = 0.0f;
            if (p.owner) p.owner[t] = -1;
          } else if (kind == 0) {
            p.loss[t] = logf(s) + m - p.zy[t];
            if (p.owner) {
              int32_t r = 0;
              while (r + 1 < p.parts && shard_offset(p.V, p.parts, r + 1) <= y) ++r;
              p.owner[t] = r;
            }
          } else {
            p.loss[t] = __int_as_float(0x7fc00000);  // NaN
            if (p.owner) p.owner[t] = -1;
            atomicOr(p.err, TPS_DEVERR_LABEL);
          }
        }
        mbar_arrive(&sh.row_full[slot]);
      }
      __syncwarp();
      if (++slot == CFS_ROWS) {
        slot = 0;
        phase ^= 1u;
      }
    }
  } else {
    // ---------------------------------------------------- consumers
    const bool vec = ((p.ldg & 7) == 0) && ((reinterpret_cast<uintptr_t>(p.dlog) & 15u) == 0);
    uint32_t stage = 0, phase = 0, slot = 0, rphase = 0;
    int64_t cur = -1, y = -1;
    float ml = 0.0f, inv = 0.0f;
    for (int64_t it = it0; it < it1; ++it) {
      const int64_t t = it / per_row, c0 = (it - t * per_row) * CFS_CHUNK;
      if (t != cur) {
        if (cur >= 0) {  // done with the previous row: free its slot
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.row_empty[slot]);
          if (++slot == CFS_ROWS) {
            slot = 0;
            rphase ^= 1u;
          }
        }
        if (!mbar_wait(&sh.row_full[slot], rphase, &sh.abort, p.err)) break;
        const float2 r = sh.row_ms[slot];
        ml = r.x;
        inv = r.y;
        y = sh.row_y[slot];
        cur = t;
      }
      if (!mbar_wait(&sh.full[stage], phase, &sh.abort, p.err)) break;
      const int64_t n = imin64(CFS_CHUNK, p.V - c0);
      TOut* grow = static_cast<TOut*>(p.dlog) + t * p.ldg + c0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = 8 * (static_cast<int>(threadIdx.x) + k * 32 * CFS_CONSUMERS);
        if (e >= n) continue;
        const uint4 q = *reinterpret_cast<const uint4*>(&sh.z[stage][e]);
        const float adj = fmaf(sh.c[stage][e / kStatsTileN], kLog2e, -ml);  // (c - m) log2(e)
        const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
        float g[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          g[2 * j] = ex2_approx(fmaf(bf16_lo(wd[j]), kLog2e, adj)) * inv;
          g[2 * j + 1] = ex2_approx(fmaf(bf16_hi(wd[j]), kLog2e, adj)) * inv;
        }
        const int64_t col = c0 + e;
        if (y >= col && y < col + 8) {
#pragma unroll
          for (int j = 0; j < 8; ++j) g[j] -= (y == col + j) ? sc : 0.0f;
        }
        if (col + 7 >= p.vreal) {  // vocabulary padding
#pragma unroll
          for (int j = 0; j < 8; ++j) g[j] = (col + j < p.vreal) ? g[j] : 0.0f;
        }
        if (!ce_dbg_ok(p, t, col, 8)) continue;
        if (vec) {
          if constexpr (sizeof(TOut) == 2) {
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              __nv_bfloat162 b = __floats2bfloat162_rn(g[2 * j], g[2 * j + 1]);
              o[j] = *reinterpret_cast<uint32_t*>(&b);
            }
            __stcs(reinterpret_cast<uint4*>(grow + e), make_uint4(o[0], o[1], o[2], o[3]));
          } else {
            __stcs(reinterpret_cast<float4*>(grow + e), make_float4(g[0], g[1], g[2], g[3]));
            __stcs(reinterpret_cast<float4*>(grow + e + 4), make_float4(g[4], g[5], g[6], g[7]));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) store_grad(grow + e + j, g[j]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[stage]);
      if (++stage == CFS_STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
}

// Extended form, before the fused kernel: the number of supervised labels
// and the gradient scale 1 / D (one block; D as in ce_finalize_kernel).
__global__ void __launch_bounds__(1024) ce_count_scale_kernel(const CeParams p, int reduction, double denominator) {
  __shared__ int red[32];
  int n = 0;
  for (int64_t t = threadIdx.x; t < p.T; t += blockDim.x) n += label_kind(p, load_label(p, t)) == 0 ? 1 : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = n;
  __syncthreads();
  if (threadIdx.x == 0) {
    int total = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) total += red[w];
    *p.count = total;
    double D = 1.0;
    if (reduction == TPS_REDUCE_MEAN) D = denominator > 0.0 ? denominator : (total > 0 ? double(total) : 1.0);
    if (p.scale != nullptr) *const_cast<float*>(p.scale) = static_cast<float>(1.0 / D);
  }
}

bool ce_tile_stats_supported(int64_t V, int32_t parts) { return parts >= 1 && V / parts >= kStatsTileN; }

static CeParams make_params(const CeDesc& c, uint32_t* dev_err) {
  CeParams p;
  p.T = c.T;
  p.V = c.V;
  p.parts = c.parts;
  p.z = c.logits;
  p.ldz = c.ldz;
  p.z16 = static_cast<const __nv_bfloat16*>(c.logits16);
  p.zshift = c.shift;
  p.shift_ld = c.shift_ld;
  p.n_tiles = 0;
  p.labels = c.labels;
  p.label_is_i64 = (c.label_dtype == TPS_I64);
  p.loss = c.loss;
  p.dlog = c.dlogits;
  p.ldg = c.ldg;
  p.owner = c.owner;
  p.stats = c.stats;
  p.zy = c.zy;
  p.err = dev_err;
  p.ignore_index = c.options ? c.ignore_index : TPS_NO_IGNORE;
  p.vreal = c.options ? c.vreal : c.V;
  p.scale = (c.options && c.reduction == TPS_REDUCE_MEAN) ? c.scale : nullptr;
  p.count = c.options ? c.count : nullptr;
  return p;
}

// The divisor's scale (before the gradient) and / or the reduced loss
// (once every loss is written) of the extended form.
static int launch_finalize(const CeDesc& c, bool want_scale, bool want_reduced, cudaStream_t stream) {
  float* scale = (want_scale && c.reduction == TPS_REDUCE_MEAN) ? c.scale : nullptr;
  float* red = (want_reduced && c.reduction != TPS_REDUCE_NONE) ? c.loss_reduced : nullptr;
  if (scale == nullptr && red == nullptr) return TPS_OK;
  ProfScope prof("ce_finalize", "ce_core", 0.0, double(c.T) * 4.0, stream);
  ce_finalize_kernel<<<1, 1024, 0, stream>>>(c.loss, c.T, c.count, c.reduction, c.denominator, scale, red);
  note_launch();
  return cudaPeekAtLastError() == cudaSuccess ? TPS_OK : TPS_ERR_CUDA;
}

int launch_ce_from_tile_stats(const CeDesc& c, const float* tile_stats, int64_t n_tiles, float* ms,
                              uint32_t* dev_err, cudaStream_t stream) {
  if (c.T == 0) return TPS_OK;
  if (c.logits16 == nullptr || c.shift == nullptr || c.zy == nullptr) return TPS_ERR_ARG;
  CeParams p = make_params(c, dev_err);
  p.stats = c.stats;  // statistics of the tiles in which a shard starts
  p.n_tiles = n_tiles;
  const int64_t gsize = c.dlogits_dtype == TPS_F32 ? 4 : 2;
  const double bytes = double(c.T) * double(c.V) * (2.0 + gsize) + double(c.T) * double(n_tiles) * 4.0 +
                       double(c.T) * (8.0 + 4.0);
  ProfScope prof("ce_stream", "ce_core", 0.0, bytes, stream);
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // One fused kernel when every item's logits and shifts can be bulk-copied:
  // 16-byte aligned logits rows and shift rows.
  const bool one_kernel = (c.V % 8 == 0) && (c.ldz % 8 == 0) && (reinterpret_cast<uintptr_t>(c.logits16) & 15u) == 0 &&
                          (c.shift_ld % 4 == 0) && (reinterpret_cast<uintptr_t>(c.shift) & 15u) == 0 &&
                          getenv("TPS_CE_TWO_KERNELS") == nullptr;
  if (one_kernel) {
    if (c.options) {  // the divisor of a mean needs every label: count them first
      ce_count_scale_kernel<<<1, 1024, 0, stream>>>(p, c.reduction, c.denominator);
      note_launch();
      if (cudaPeekAtLastError() != cudaSuccess) return TPS_ERR_CUDA;
    }
    static int occ_f = 0, occ_b = 0;
    static cudaError_t attr_err = cudaSuccess;
    static std::once_flag once;
    std::call_once(once, [] {
      const int smem = static_cast<int>(sizeof(CfsShared));
      attr_err = cudaFuncSetAttribute(ce_fused_stream_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (attr_err == cudaSuccess)
        attr_err = cudaFuncSetAttribute(ce_fused_stream_kernel<__nv_bfloat16>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_f, ce_fused_stream_kernel<float>, CFS_THREADS, smem);
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_b, ce_fused_stream_kernel<__nv_bfloat16>, CFS_THREADS, smem);
    });
    if (attr_err != cudaSuccess) return TPS_ERR_CUDA;
    const int occ = c.dlogits_dtype == TPS_F32 ? occ_f : occ_b;
    const int64_t items = c.T * ((c.V + CFS_CHUNK - 1) / CFS_CHUNK);
    const int64_t want = static_cast<int64_t>(sms) * (occ > 0 ? occ : 1);
    const unsigned grid = static_cast<unsigned>(items < want ? items : want);
    CeParams q = p;
    q.count = nullptr;  // counted above
    if (c.dlogits_dtype == TPS_F32)
      ce_fused_stream_kernel<float><<<grid, CFS_THREADS, sizeof(CfsShared), stream>>>(q, tile_stats);
    else
      ce_fused_stream_kernel<__nv_bfloat16><<<grid, CFS_THREADS, sizeof(CfsShared), stream>>>(q, tile_stats);
    note_launch();
    if (cudaPeekAtLastError() != cudaSuccess) return TPS_ERR_CUDA;
    return c.options ? launch_finalize(c, false, true, stream) : TPS_OK;  // the reduced loss
  }
  const int64_t nb = (c.T + CEF_TOK_PER_BLOCK - 1) / CEF_TOK_PER_BLOCK;
  if (nb > 0x7FFFFFFF) return TPS_ERR_SHAPE;
  if (c.options && cudaMemsetAsync(c.count, 0, sizeof(int32_t), stream) != cudaSuccess) return TPS_ERR_CUDA;
  ce_combine_kernel<<<static_cast<unsigned>(nb), 32 * CEF_TOK_PER_BLOCK, 0, stream>>>(p, tile_stats, n_tiles, ms);
  note_launch();
  if (cudaPeekAtLastError() != cudaSuccess) return TPS_ERR_CUDA;
  if (c.options) {  // every loss and the count are known after the combine
    const int rc = launch_finalize(c, true, true, stream);
    if (rc != TPS_OK) return rc;
  }
  // exactly the blocks that fit at once: a larger grid would run as a
  // second, partial wave
  static int occ_f = 0, occ_b = 0;
  static std::once_flag occ_once;
  std::call_once(occ_once, [] {
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_f, ce_grad_stream_kernel<float>, CEF_THREADS, 0);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_b, ce_grad_stream_kernel<__nv_bfloat16>, CEF_THREADS, 0);
  });
  const int occ = (c.dlogits_dtype == TPS_F32 ? occ_f : occ_b);
  const unsigned grid = static_cast<unsigned>(sms * (occ > 0 ? occ : 1));
  if (c.dlogits_dtype == TPS_F32)
    ce_grad_stream_kernel<float><<<grid, CEF_THREADS, 0, stream>>>(p, ms);
  else
    ce_grad_stream_kernel<__nv_bfloat16><<<grid, CEF_THREADS, 0, stream>>>(p, ms);
  note_launch();
  return cudaPeekAtLastError() == cudaSuccess ? TPS_OK : TPS_ERR_CUDA;
}

// The combine alone, for the path whose dlogits are formed inside the
// dHidden GEMM (CeGradOperand): the loss, the owner and each row's
// (m, 1/s).  Plain form only (no options).
int launch_ce_combine(const CeDesc& c, const float* tile_stats, int64_t n_tiles, float* ms, uint32_t* dev_err,
                      cudaStream_t stream) {
  if (c.T == 0) return TPS_OK;
  if (c.options || c.zy == nullptr) return TPS_ERR_ARG;
  CeParams p = make_params(c, dev_err);
  p.stats = c.stats;  // statistics of the tiles in which a shard starts
  p.n_tiles = n_tiles;
  const int64_t nb = (c.T + CEF_TOK_PER_BLOCK - 1) / CEF_TOK_PER_BLOCK;
  if (nb > 0x7FFFFFFF) return TPS_ERR_SHAPE;
  const double bytes = double(c.T) * double(n_tiles) * 8.0 + double(c.T) * 20.0;
  ProfScope prof("ce_combine", "ce_core", 0.0, bytes, stream);
  ce_combine_kernel<<<static_cast<unsigned>(nb), 32 * CEF_TOK_PER_BLOCK, 0, stream>>>(p, tile_stats, n_tiles, ms);
  note_launch();
  return cudaPeekAtLastError() == cudaSuccess ? TPS_OK : TPS_ERR_CUDA;
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
  const bool z_aligned = ((reinterpret_cast<uintptr_t>(p.z) & 15u) == 0) && ((p.ldz & 3) == 0);
  if (z_aligned && max_len + 3 <= CEP_BUF_FLOATS) {
    // persistent clusters, as many as can be resident at once
    const size_t smem = size_t(CEP_NBUF) * CEP_BUF_FLOATS * sizeof(float);
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [smem] {
      attr_err = cudaFuncSetAttribute(ce_persistent_kernel<TOut>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem));
    });
    if (attr_err != cudaSuccess) return TPS_ERR_CUDA;
    cfg.blockDim = dim3(CEP_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    int clusters = 0;
    cfg.gridDim = dim3(static_cast<unsigned>(p.parts), 1, 1);
    if (cudaOccupancyMaxActiveClusters(&clusters, ce_persistent_kernel<TOut>, &cfg) != cudaSuccess || clusters < 1)
      clusters = 1;
    const int64_t C = p.T < clusters ? p.T : clusters;
    cfg.gridDim = dim3(static_cast<unsigned>(p.parts), static_cast<unsigned>(C), 1);
    e = cudaLaunchKernelEx(&cfg, ce_persistent_kernel<TOut>, p);
  } else if (max_len <= CE_THREADS * 4 * 2) {
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

static int launch_stats(const CeParams& p, cudaStream_t stream) {
  ProfScope prof("ce_stats", "ce_core", 0.0, double(p.T) * double(p.V) * 4.0, stream);
  ce_stats_kernel<<<dim3(static_cast<unsigned>(p.parts), static_cast<unsigned>(p.T)), 256, 0, stream>>>(p);
  note_launch();
  return cudaPeekAtLastError() == cudaSuccess ? TPS_OK : TPS_ERR_CUDA;
}

template <typename TOut>
static int launch_grad(const CeParams& p, cudaStream_t stream) {
  const int64_t chunks = (p.V + CE_GRAD_CHUNK - 1) / CE_GRAD_CHUNK;
  ProfScope prof("ce_grad", "ce_core", 0.0, double(p.T) * double(p.V) * (4.0 + sizeof(TOut)), stream);
  ce_grad_kernel<TOut><<<dim3(static_cast<unsigned>(chunks), static_cast<unsigned>(p.T)), 256, 0, stream>>>(p);
  note_launch();
  return cudaPeekAtLastError() == cudaSuccess ? TPS_OK : TPS_ERR_CUDA;
}

// Tokens [t0, t0 + min(65535, T - t0)) of `p`: tokens go on grid.y.
static CeParams slab(const CeParams& p, int64_t t0, size_t gsize) {
  CeParams q = p;
  q.T = imin64(65535, p.T - t0);
  q.z = p.z + t0 * p.ldz;
  q.labels = p.label_is_i64 ? static_cast<const void*>(static_cast<const int64_t*>(p.labels) + t0)
                            : static_cast<const void*>(static_cast<const int32_t*>(p.labels) + t0);
  q.loss = p.loss + t0;
  q.dlog = static_cast<char*>(p.dlog) + t0 * p.ldg * gsize;
  q.owner = p.owner ? p.owner + t0 : nullptr;
  q.stats = p.stats ? p.stats + t0 * p.parts * 2 : nullptr;
  q.zy = p.zy ? p.zy + t0 : nullptr;
  return q;
}

int launch_ce(const CeDesc& c, uint32_t* dev_err, cudaStream_t stream, bool* used_cluster) {
  const CeParams p = make_params(c, dev_err);
  // The cluster kernels serve the plain form only.
  const bool cl = !c.options && ce_cluster_supported(c.V, c.parts, c.dlogits_dtype);
  if (used_cluster) *used_cluster = cl;
  const bool f32 = c.dlogits_dtype == TPS_F32;
  const size_t gsize = f32 ? 4 : 2;
  if (cl) {
    for (int64_t t0 = 0; t0 < c.T; t0 += 65535) {
      const CeParams q = slab(p, t0, gsize);
      const int rc = f32 ? launch_cluster<float>(q, stream) : launch_cluster<__nv_bfloat16>(q, stream);
      if (rc != TPS_OK) return rc;
    }
    return TPS_OK;
  }
  if (c.options && c.T > 0 && cudaMemsetAsync(c.count, 0, sizeof(int32_t), stream) != cudaSuccess)
    return TPS_ERR_CUDA;
  for (int64_t t0 = 0; t0 < c.T; t0 += 65535) {
    const int rc = launch_stats(slab(p, t0, gsize), stream);
    if (rc != TPS_OK) return rc;
  }
  if (c.options && c.T > 0) {  // the mean's divisor needs every count
    const int rc = launch_finalize(c, true, false, stream);
    if (rc != TPS_OK) return rc;
  }
  for (int64_t t0 = 0; t0 < c.T; t0 += 65535) {
    const CeParams q = slab(p, t0, gsize);
    const int rc = f32 ? launch_grad<float>(q, stream) : launch_grad<__nv_bfloat16>(q, stream);
    if (rc != TPS_OK) return rc;
  }
  if (c.options && c.T > 0) return launch_finalize(c, false, true, stream);  // every loss is written
  return TPS_OK;
}

}  // namespace tps
