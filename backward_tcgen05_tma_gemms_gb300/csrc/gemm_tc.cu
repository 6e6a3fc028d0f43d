// gemm_tc.cu -- persistent, warp-specialised bf16 GEMM on the sm_103a
// tensor cores: TMA loads tiles into 128-byte-swizzled shared memory,
// one thread issues tcgen05.mma (cta_group::1, M=128, N=256, K=16) into a
// double-buffered fp32 accumulator in tensor memory, and four epilogue warps
// drain the other buffer with tcgen05.ld and apply the fused epilogue.
//
// This is the shard GEMM of "Sharded GEMM与Backprop：行、列、内维三种切分"
// (解题路线 steps 2-4) and of the column/row-parallel layers of
// "第 6 课：张量并行 TP" (core concept 1): a result the pages concatenate is
// a range of D, and a result they sum over ranks is the K loop of one tile,
// which walks the ranks' shard segments of K in rank order and accumulates
// them in tensor memory.
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer (one thread)
//   warp 1      TMEM allocator + MMA issuer (one thread)
//   warps 2..5  epilogue; warp w may only read TMEM lanes 32*(w%4)..+31
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "epilogue.cuh"
#include "internal.cuh"
#include "ptx.cuh"

namespace tps {

constexpr int TC_BM = 128;
constexpr int TC_BN = 256;
static_assert(TC_BN == kTileN, "CE tile statistics assume the GEMM's N tile");
constexpr int TC_BK = 64;  // one 128-byte swizzle row of bf16
constexpr int TC_STAGES = 4;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;  // 16 KB
constexpr int TC_B_BYTES = TC_BN * TC_BK * 2;  // 32 KB
constexpr int TC_STAGE_BYTES = TC_A_BYTES + TC_B_BYTES;
constexpr int TC_THREADS = 192;
constexpr int TC_EPI_THREADS = 128;
constexpr uint32_t TC_TMEM_COLS = 2 * TC_BN;  // two fp32 accumulators of BN columns
constexpr int TC_GROUP_M = 16;                // tile raster: groups of 16 M-tiles
// A box of an MN-major operand: 64 MN elements (128 B) x 64 K rows.
constexpr int TC_MN_BOX_BYTES = 64 * TC_BK * 2;  // 8 KB
// Epilogue staging for TMA stores, per epilogue warp: a 32 x 32 fp32 box
// (128-byte swizzle) and a 32 x 32 bf16 box (64-byte swizzle).
constexpr int TC_STG_F32_BYTES = 32 * 32 * 4;
constexpr int TC_STG_BF16_BYTES = 32 * 32 * 2;
constexpr int TC_STAGING_BYTES = 4 * (TC_STG_F32_BYTES + TC_STG_BF16_BYTES);

struct TcBarriers {
  uint64_t full[TC_STAGES];
  uint64_t empty[TC_STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_slot;
  uint32_t abort;
};

constexpr size_t TC_SMEM_BYTES =
    1024 /*alignment slack*/ + TC_STAGES * TC_STAGE_BYTES + TC_STAGING_BYTES + sizeof(TcBarriers);

struct TcParams {
  int M, N, K;
  int m_tiles, n_tiles, k_tiles, num_tiles;
  int tma_store;  // 1: outputs leave through swizzled staging + TMA stores
  Epilogue epi;
  uint32_t* err;
};

// Row `r` of a warp's staging box, in the layout the TMA unit expects for
// 128-byte (fp32, 8 chunks of 16 B per row) and 64-byte (bf16, 4 chunks per
// row) swizzling: chunk i of row r sits at chunk i ^ f(r).  Consecutive rows
// land in different bank groups, so the per-lane row writes do not conflict.
__device__ __forceinline__ void stage_f32_sw128(uint8_t* buf, int r, const float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    *reinterpret_cast<float4*>(buf + r * 128 + ((i ^ (r & 7)) << 4)) =
        make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}
__device__ __forceinline__ void stage_bf16_sw64(uint8_t* buf, int r, const float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b0 = __floats2bfloat162_rn(v[8 * i + 0], v[8 * i + 1]);
    __nv_bfloat162 b1 = __floats2bfloat162_rn(v[8 * i + 2], v[8 * i + 3]);
    __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * i + 4], v[8 * i + 5]);
    __nv_bfloat162 b3 = __floats2bfloat162_rn(v[8 * i + 6], v[8 * i + 7]);
    uint4 w;
    w.x = *reinterpret_cast<uint32_t*>(&b0);
    w.y = *reinterpret_cast<uint32_t*>(&b1);
    w.z = *reinterpret_cast<uint32_t*>(&b2);
    w.w = *reinterpret_cast<uint32_t*>(&b3);
    *reinterpret_cast<uint4*>(buf + r * 64 + ((i ^ ((r >> 1) & 3)) << 4)) = w;
  }
}

__device__ __forceinline__ void tc_tile_coords(int tile, int m_tiles, int n_tiles, int& mt, int& nt) {
  const int group_size = TC_GROUP_M * n_tiles;
  const int group = tile / group_size;
  const int first_m = group * TC_GROUP_M;
  const int gm = min(m_tiles - first_m, TC_GROUP_M);
  const int in_group = tile - group * group_size;
  mt = first_m + in_group % gm;
  nt = in_group / gm;
}

// ---- vocabulary-CE statistics in the logits epilogue --------------------
// Each epilogue thread owns one output row of the tile, so the statistics
// of the tile's 256 columns need no cross-thread reduction: the thread folds
// its 8 chunks of 32 columns into (max, sum of e^{z - max}) for the part of
// the tile in shard a (the shard of the tile's first column) and the part in
// shard b (the next one).
constexpr float kTcLog2e = 1.4426950408889634f;

// Fold elements [i0, i1) of v into (m, s); the range is a compile-time-free
// runtime interval, so each element is predicated.
__device__ __forceinline__ void ce_fold(const float (&v)[32], int i0, int i1, float& m, float& s) {
  float cm = -INFINITY;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i >= i0 && i < i1) cm = fmaxf(cm, v[i]);
  if (cm == -INFINITY) return;
  if (cm > m) {
    s = (m == -INFINITY) ? 0.0f : s * ex2_approx((m - cm) * kTcLog2e);
    m = cm;
  }
  const float ml = m * kTcLog2e;
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i >= i0 && i < i1) acc += ex2_approx(fmaf(v[i], kTcLog2e, -ml));
  s += acc;
}

// The shard owning column c under the array_split of n into p parts.
__device__ __forceinline__ int64_t shard_of(int64_t c, int64_t n, int64_t p) {
  const int64_t q = n / p, r = n % p, big = r * (q + 1);
  return c < big ? c / (q + 1) : r + (c - big) / q;
}

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD2,
                   const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzling repeats every 1024 bytes: align the stage buffers.
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* staging = smem + TC_STAGES * TC_STAGE_BYTES;  // 1024-aligned
  TcBarriers* bars = reinterpret_cast<TcBarriers*>(staging + TC_STAGING_BYTES);
  volatile uint32_t* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->tmem_full[b], 1);
      mbar_init(&bars->tmem_empty[b], TC_EPI_THREADS);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, TC_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        int mt, nt;
        tc_tile_coords(tile, p.m_tiles, p.n_tiles, mt, nt);
        const int m0 = mt * TC_BM, n0 = nt * TC_BN;
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * TC_STAGE_BYTES;
          uint8_t* sb = sa + TC_A_BYTES;
          uint64_t* fb = &bars->full[stage];
          mbar_expect_tx(fb, TC_STAGE_BYTES);
          const int k0 = kt * TC_BK;
          if (!A_MN) {
            tma_load_2d(sa, &tmA, fb, k0, m0);
          } else {
#pragma unroll
            for (int j = 0; j < TC_BM / 64; ++j) tma_load_2d(sa + j * TC_MN_BOX_BYTES, &tmA, fb, m0 + 64 * j, k0);
          }
          if (!B_MN) {
            tma_load_2d(sb, &tmB, fb, k0, n0);
          } else {
#pragma unroll
            for (int j = 0; j < TC_BN / 64; ++j) tma_load_2d(sb + j * TC_MN_BOX_BYTES, &tmB, fb, n0 + 64 * j, k0);
          }
          ++issued;
          if (++stage == TC_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: every issued load must land before the CTA may exit.
      const int64_t first = issued > TC_STAGES ? issued - TC_STAGES : 0;
      for (int64_t i = first; i < issued; ++i)
        mbar_wait_drain(&bars->full[i % TC_STAGES], static_cast<uint32_t>((i / TC_STAGES) & 1), p.err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(TC_BM, TC_BN, A_MN, B_MN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        if (!mbar_wait(&bars->tmem_empty[acc], acc_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * TC_BN;
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          if (!mbar_wait(&bars->full[stage], phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * TC_STAGE_BYTES);
          const uint32_t sb = sa + TC_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk) {
            // K-major: the 16-element K step is 32 bytes inside the swizzled
            // 128-byte row; rows are 128 B apart, 8-row groups 1024 B apart.
            // MN-major: the K step is 16 rows = two 1024-byte 8-row groups;
            // 64-element MN groups are one 8 KB box apart.
            const uint64_t ad = A_MN ? smem_desc_sw128(sa + kk * 2048, TC_MN_BOX_BYTES, 1024)
                                     : smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(sb + kk * 2048, TC_MN_BOX_BYTES, 1024)
                                     : smem_desc_sw128(sb + kk * 32, 16, 1024);
            tc_mma_f16(d_tmem, ad, bd, idesc, (kt | kk) != 0 ? 1u : 0u);
          }
          tc_commit(&bars->empty[stage]);  // frees the stage once these MMAs finish
          if (++stage == TC_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&bars->tmem_full[acc]);  // accumulator complete
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Drain: all issued MMAs complete before TMEM is released.
      tc_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, p.err);
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    uint8_t* stg_f32 = staging + (warp - 2) * TC_STG_F32_BYTES;
    uint8_t* stg_bf16 = staging + 4 * TC_STG_F32_BYTES + (warp - 2) * TC_STG_BF16_BYTES;
    const Epilogue& e = p.epi;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      int mt, nt;
      tc_tile_coords(tile, p.m_tiles, p.n_tiles, mt, nt);
      const int m0 = mt * TC_BM, n0 = nt * TC_BN;
      if (!mbar_wait(&bars->tmem_full[acc], acc_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const int row0 = m0 + q * 32;
      const int64_t row = row0 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * TC_BN;
      // act-bwd: the pre-activation of the next 32 columns is loaded while
      // the current ones are processed
      float a_next[32];
      const bool bwd = p.tma_store && e.mode == EPI_ACT_BWD;
      if (bwd) {
        if (row < p.M) {
          load_run32(e.aux + row * e.ld_aux + n0, min(32, p.N - n0), a_next);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) a_next[i] = 0.0f;
        }
      }
      // CE statistics: columns < split belong to shard a, the rest to b
      const bool ce = (e.mode == EPI_CE_STATS);
      int64_t split = 0;
      float ma = -INFINITY, sa = 0.0f, mb = -INFINITY, sb = 0.0f;
      if (ce) split = shard_offset(p.N, e.ce_parts, shard_of(n0, p.N, e.ce_parts) + 1);
      for (int c = 0; c < TC_BN / 32; ++c) {
        const int col0 = n0 + c * 32;
        if (col0 >= p.N) break;  // warp-uniform
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        float a[32];
        if (bwd) {
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = a_next[i];
          if (row < p.M && col0 + 32 < p.N && c + 1 < TC_BN / 32)
            load_run32(e.aux + row * e.ld_aux + col0 + 32, min(32, p.N - col0 - 32), a_next);
        }
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        const int n = min(32, p.N - col0);
        if (ce) {
          const int na = static_cast<int>(split - col0 < 0 ? 0 : (split - col0 > n ? n : split - col0));
          ce_fold(v, 0, na, ma, sa);
          if (na < n) ce_fold(v, na, n, mb, sb);
        }
        if (!p.tma_store) {
          if (row < p.M) epilogue_run32(e, row, col0, n, v);
          continue;
        }
        // TMA store path: the box (32 rows x 32 columns) is clipped to the
        // tensor by the TMA unit, so rows >= M and columns >= N are dropped.
        if (lane == 0) bulk_wait_read0();  // previous boxes have left staging
        __syncwarp();
        if (e.mode == EPI_STORE || e.mode == EPI_CE_STATS) {
          if (e.d_dtype == TPS_F32)
            stage_f32_sw128(stg_f32, lane, v);
          else
            stage_bf16_sw64(stg_bf16, lane, v);
        } else if (e.mode == EPI_ACT_FWD) {
          if (e.d != nullptr) stage_f32_sw128(stg_f32, lane, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = act_fwd(e.act, v[i]);
          stage_bf16_sw64(stg_bf16, lane, v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= act_grad(e.act, a[i]);
          if (e.d_dtype == TPS_F32)
            stage_f32_sw128(stg_f32, lane, v);
          else
            stage_bf16_sw64(stg_bf16, lane, v);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (e.mode == EPI_ACT_FWD) {
            if (e.d != nullptr) tma_store_2d(&tmD, stg_f32, col0, row0);
            tma_store_2d(&tmD2, stg_bf16, col0, row0);
          } else {
            tma_store_2d(&tmD, e.d_dtype == TPS_F32 ? stg_f32 : stg_bf16, col0, row0);
          }
          bulk_commit();
        }
      }
      if (ce && row < p.M)
        *reinterpret_cast<float4*>(e.stats + (row * e.n_tiles + nt) * 4) = make_float4(ma, sa, mb, sb);
      tc_fence_before();
      mbar_arrive(&bars->tmem_empty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (p.tma_store && lane == 0) bulk_wait0();  // stores complete before exit
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TC_TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major bf16 matrix view: `rows` x `cols`, `cols` contiguous, row pitch
// `ld` elements.  Box: `box_cols` x `box_rows`, 128-byte swizzle, OOB -> 0.
static bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                     int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output view for TMA stores: rows x cols row-major with pitch `ld`
// elements, box 32 x 32, swizzle matching the staging layout.
static bool make_out_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int dtype) {
  auto fn = encode_fn();
  if (fn == nullptr || base == nullptr) return false;
  const int es = (dtype == TPS_F32) ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || (ld * es) % 16 != 0 || ld < cols) return false;
  if (rows >= (1ll << 31) || cols >= (1ll << 31)) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * es)};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype == TPS_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  dtype == TPS_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The tensor-core path needs bf16 operands that TMA can describe: 16-byte
// aligned base, unit stride in one dimension and a pitch that is a multiple
// of 16 bytes.
bool gemm_tc_supported(const GemmDesc& g) {
  if (g.in_dtype != TPS_BF16) return false;
  if (g.M < 1 || g.N < 1 || g.K < 1) return false;
  if (g.M >= (1ll << 31) || g.N >= (1ll << 31) || g.K >= (1ll << 31)) return false;
  auto ok_operand = [](const void* ptr, int64_t s_outer, int64_t s_inner, int64_t inner_extent) {
    if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return false;
    if (s_inner != 1) return false;
    if ((s_outer * 2) % 16 != 0 || s_outer < inner_extent) return false;
    return s_outer * 2 < (1ll << 40);
  };
  const bool a_ok = (g.a_sk == 1) ? ok_operand(g.a, g.a_sm, g.a_sk, g.K) : ok_operand(g.a, g.a_sk, g.a_sm, g.M);
  const bool b_ok = (g.b_sk == 1) ? ok_operand(g.b, g.b_sn, g.b_sk, g.K) : ok_operand(g.b, g.b_sk, g.b_sn, g.N);
  return a_ok && b_ok;
}

template <bool A_MN, bool B_MN>
static int launch_typed(const GemmDesc& g, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td,
                        const CUtensorMap& td2, const TcParams& p, int grid, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_tc_kernel<A_MN, B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(TC_SMEM_BYTES));
  });
  if (attr_err != cudaSuccess) return TPS_ERR_CUDA;
  ProfScope prof("gemm_tc", g.name, 2.0 * double(g.M) * double(g.N) * double(g.K), 0.0, stream);
  gemm_tc_kernel<A_MN, B_MN><<<grid, TC_THREADS, TC_SMEM_BYTES, stream>>>(ta, tb, td, td2, p);
  note_launch();
  return cudaPeekAtLastError() == cudaSuccess ? TPS_OK : TPS_ERR_CUDA;
}

static int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

int launch_gemm_tc(const GemmDesc& g, uint32_t* dev_err, cudaStream_t stream) {
  const bool a_mn = (g.a_sk != 1);
  const bool b_mn = (g.b_sk != 1);
  CUtensorMap ta, tb;
  bool ok = a_mn ? make_map(&ta, g.a, g.K, g.M, g.a_sk, 64, TC_BK)     // stored K x M
                 : make_map(&ta, g.a, g.M, g.K, g.a_sm, TC_BK, TC_BM);  // stored M x K
  ok = ok && (b_mn ? make_map(&tb, g.b, g.K, g.N, g.b_sk, 64, TC_BK)    // stored K x N
                   : make_map(&tb, g.b, g.N, g.K, g.b_sn, TC_BK, TC_BN)); // stored N x K
  if (!ok) return TPS_ERR_CUDA;

  TcParams p;
  p.M = static_cast<int>(g.M);
  p.N = static_cast<int>(g.N);
  p.K = static_cast<int>(g.K);
  p.m_tiles = static_cast<int>((g.M + TC_BM - 1) / TC_BM);
  p.n_tiles = static_cast<int>((g.N + TC_BN - 1) / TC_BN);
  p.k_tiles = static_cast<int>((g.K + TC_BK - 1) / TC_BK);
  p.num_tiles = p.m_tiles * p.n_tiles;
  p.epi = g.epi;
  p.err = dev_err;
  // TMA stores when every output can be described (else direct stores).
  CUtensorMap td, td2;
  memset(&td, 0, sizeof(td));
  memset(&td2, 0, sizeof(td2));
  bool tma = true;
  if (g.epi.mode == EPI_ACT_FWD) {
    if (g.epi.d != nullptr) tma = make_out_map(&td, g.epi.d, g.M, g.N, g.epi.ldd, TPS_F32);
    tma = tma && g.epi.d2_dtype == TPS_BF16 && make_out_map(&td2, g.epi.d2, g.M, g.N, g.epi.ldd2, TPS_BF16);
  } else {
    tma = make_out_map(&td, g.epi.d, g.M, g.N, g.epi.ldd, g.epi.d_dtype);
  }
  p.tma_store = tma ? 1 : 0;
  const int grid = p.num_tiles < num_sms() ? p.num_tiles : num_sms();

  if (!a_mn && !b_mn) return launch_typed<false, false>(g, ta, tb, td, td2, p, grid, stream);
  if (!a_mn && b_mn) return launch_typed<false, true>(g, ta, tb, td, td2, p, grid, stream);
  if (a_mn && !b_mn) return launch_typed<true, false>(g, ta, tb, td, td2, p, grid, stream);
  return launch_typed<true, true>(g, ta, tb, td, td2, p, grid, stream);
}

}  // namespace tps
