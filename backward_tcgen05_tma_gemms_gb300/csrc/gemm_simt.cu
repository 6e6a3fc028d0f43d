// gemm_simt.cu -- shard-aware GEMM with plain fp32 FMA arithmetic.
//
// Used for fp32 operands (the tensor cores' tf32 mode would round operands
// to 10 mantissa bits) and for bf16 operands whose layout TMA cannot
// describe.  It follows the pages' rank simulation literally: when the
// contraction dimension is sharded over `kparts` logical ranks
// ("Sharded GEMM与Backprop：行、列、内维三种切分", 解题路线 steps 2-4: a
// result that needs sum/all-reduce), each rank's partial product over its
// array_split segment of K is accumulated separately and the partials are
// then added in rank order, inside the kernel.  Further contraction
// segments (D = A B + A2 B2 + A3 B3) add each rank's segment of every
// further pair to the same rank partial.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "epilogue.cuh"
#include "internal.cuh"

namespace tps {

constexpr int SG_BM = 64, SG_BN = 64, SG_BK = 16, SG_THREADS = 256;

struct SimtParams {
  int64_t M, N, K, K2, K3;
  const void* a;
  int64_t a_sm, a_sk;
  const void* b;
  int64_t b_sk, b_sn;
  const void* a2;
  int64_t a2_sm, a2_sk;
  const void* b2;
  int64_t b2_sk, b2_sn;
  const void* a3;
  int64_t a3_sm, a3_sk;
  const void* b3;
  int64_t b3_sk, b3_sn;
  int32_t kparts;
  Epilogue epi;
};

template <typename T>
__device__ __forceinline__ float ld_as_float(const void* base, int64_t idx) {
  if constexpr (sizeof(T) == 4)
    return static_cast<const float*>(base)[idx];
  else
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
}

// part += A[m0.., kb..ke) B[kb..ke, n0..) for this thread's 4 x 4 outputs.
template <typename T>
__device__ __forceinline__ void simt_segment(const void* a, int64_t a_sm, int64_t a_sk, const void* b, int64_t b_sk,
                                             int64_t b_sn, int64_t M, int64_t N, int64_t m0, int64_t n0, int64_t kb,
                                             int64_t ke, float (&As)[SG_BK][SG_BM + 4], float (&Bs)[SG_BK][SG_BN + 4],
                                             float (&part)[4][4]) {
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  for (int64_t k0 = kb; k0 < ke; k0 += SG_BK) {
    for (int e = tid; e < SG_BM * SG_BK; e += SG_THREADS) {
      int mm, kk;
      if (a_sk == 1) {
        mm = e / SG_BK;
        kk = e % SG_BK;
      } else {
        mm = e % SG_BM;
        kk = e / SG_BM;
      }
      const int64_t m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < M && k < ke) ? ld_as_float<T>(a, m * a_sm + k * a_sk) : 0.0f;
    }
    for (int e = tid; e < SG_BN * SG_BK; e += SG_THREADS) {
      int nn, kk;
      if (b_sk == 1) {
        nn = e / SG_BK;
        kk = e % SG_BK;
      } else {
        nn = e % SG_BN;
        kk = e / SG_BN;
      }
      const int64_t n = n0 + nn, k = k0 + kk;
      Bs[kk][nn] = (n < N && k < ke) ? ld_as_float<T>(b, k * b_sk + n * b_sn) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) part[i][j] = fmaf(av[i], bv[j], part[i][j]);
    }
    __syncthreads();
  }
}

template <typename T>
__global__ void __launch_bounds__(SG_THREADS) gemm_simt_kernel(const SimtParams p) {
  __shared__ float As[SG_BK][SG_BM + 4];
  __shared__ float Bs[SG_BK][SG_BN + 4];
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * SG_BM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * SG_BN;

  float total[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) total[i][j] = 0.0f;

  for (int32_t r = 0; r < p.kparts; ++r) {
    float part[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) part[i][j] = 0.0f;
    simt_segment<T>(p.a, p.a_sm, p.a_sk, p.b, p.b_sk, p.b_sn, p.M, p.N, m0, n0, shard_offset(p.K, p.kparts, r),
                    shard_offset(p.K, p.kparts, r + 1), As, Bs, part);
    if (p.K2 > 0)
      simt_segment<T>(p.a2, p.a2_sm, p.a2_sk, p.b2, p.b2_sk, p.b2_sn, p.M, p.N, m0, n0,
                      shard_offset(p.K2, p.kparts, r), shard_offset(p.K2, p.kparts, r + 1), As, Bs, part);
    if (p.K3 > 0)
      simt_segment<T>(p.a3, p.a3_sm, p.a3_sk, p.b3, p.b3_sk, p.b3_sn, p.M, p.N, m0, n0,
                      shard_offset(p.K3, p.kparts, r), shard_offset(p.K3, p.kparts, r + 1), As, Bs, part);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) total[i][j] += part[i][j];
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= p.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx * 4 + j;
      if (n < p.N) epilogue_elem(p.epi, m, n, total[i][j]);
    }
  }
}

int launch_gemm_simt(const GemmDesc& g, uint32_t* /*dev_err*/, cudaStream_t stream) {
  SimtParams p;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.a = g.a;
  p.a_sm = g.a_sm;
  p.a_sk = g.a_sk;
  p.b = g.b;
  p.b_sk = g.b_sk;
  p.b_sn = g.b_sn;
  p.K2 = g.K2;
  p.a2 = g.a2;
  p.a2_sm = g.a2_sm;
  p.a2_sk = g.a2_sk;
  p.b2 = g.b2;
  p.b2_sk = g.b2_sk;
  p.b2_sn = g.b2_sn;
  p.K3 = g.K3;
  p.a3 = g.a3;
  p.a3_sm = g.a3_sm;
  p.a3_sk = g.a3_sk;
  p.b3 = g.b3;
  p.b3_sk = g.b3_sk;
  p.b3_sn = g.b3_sn;
  p.kparts = g.kparts < 1 ? 1 : g.kparts;
  // the fused gate/up form, the CE statistics form and column segments are
  // tensor-core only
  if (g.epi.mode == EPI_GLU_FWD || g.epi.mode == EPI_CE_STATS || g.n_segs > 1) return TPS_ERR_ARG;
  p.epi = g.epi;
  const int64_t gx = (g.N + SG_BN - 1) / SG_BN, gy = (g.M + SG_BM - 1) / SG_BM;
  if (gx > 0x7FFFFFFF || gy > 65535) return TPS_ERR_SHAPE;
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  ProfScope prof("gemm_simt", g.name, 2.0 * double(g.M) * double(g.N) * double(g.K + g.K2 + g.K3), 0.0, stream);
  if (g.in_dtype == TPS_F32)
    gemm_simt_kernel<float><<<grid, SG_THREADS, 0, stream>>>(p);
  else
    gemm_simt_kernel<__nv_bfloat16><<<grid, SG_THREADS, 0, stream>>>(p);
  note_launch();
  return cudaPeekAtLastError() == cudaSuccess ? TPS_OK : TPS_ERR_CUDA;
}

}  // namespace tps
