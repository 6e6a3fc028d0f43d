// gemm_tc.cu -- persistent, warp-specialised bf16 GEMM on the sm_103a
// tensor cores, one CTA per 128 x 256 output tile: TMA loads tiles into
// 128-byte-swizzled shared memory, one thread issues tcgen05.mma
// (cta_group::1, M=128, N=256, K=16) into a double-buffered fp32
// accumulator in tensor memory, and four epilogue warps drain the other
// buffer with tcgen05.ld and apply the fused epilogue.  gemm_tc2.cu holds
// the CTA-pair variant; this file also holds the host code both share.
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
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "tc_common.cuh"

namespace tps {

constexpr int TC_BM = 128;
constexpr int TC_BN = 256;
constexpr int TC_STAGES = 4;
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2;  // 16 KB
constexpr int TC_B_BYTES = TC_BN * TC_BK * 2;  // 32 KB
constexpr int TC_STAGE_BYTES = TC_A_BYTES + TC_B_BYTES;
constexpr int TC_THREADS = 192;
constexpr int TC_EPI_THREADS = 128;
constexpr uint32_t TC_TMEM_COLS = 2 * TC_BN;  // two fp32 accumulators of BN columns
constexpr int TC_GROUP_M = 16;                // default tile raster: groups of 16 M-tiles
constexpr int TC_STAGING_BYTES = 4 * (TC_STG_F32_BYTES + TC_STG_BF16_BYTES);
static_assert(TC_BN % kStatsTileN == 0, "CE statistics tiles must divide the N tile");

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
  int raster_n, group;  // tile order (tc_raster)
  int pol_a, pol_b;     // L2 policy per operand: 0 normal, 1 evict-first, 2 evict-last
  int tma_store;        // 1: outputs leave through swizzled staging + TMA stores
  Epilogue epi;
  uint32_t* err;
};

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
      const uint64_t pa = tc_policy(p.pol_a), pb = tc_policy(p.pol_b);
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        int mt, nt;
        tc_raster(p.raster_n, p.group, p.m_tiles, p.n_tiles, tile, mt, nt);
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
            tma_load_maybe_hint(sa, &tmA, fb, k0, m0, p.pol_a, pa);
          } else {
#pragma unroll
            for (int j = 0; j < TC_BM / 64; ++j)
              tma_load_maybe_hint(sa + j * TC_MN_BOX_BYTES, &tmA, fb, m0 + 64 * j, k0, p.pol_a, pa);
          }
          if (!B_MN) {
            tma_load_maybe_hint(sb, &tmB, fb, k0, n0, p.pol_b, pb);
          } else {
#pragma unroll
            for (int j = 0; j < TC_BN / 64; ++j)
              tma_load_maybe_hint(sb + j * TC_MN_BOX_BYTES, &tmB, fb, n0 + 64 * j, k0, p.pol_b, pb);
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
    const bool ce = (e.mode == EPI_CE_STATS);
    const bool bwd = p.tma_store && (e.mode == EPI_ACT_BWD || e.mode == EPI_GLU_UP);  // AUX prefetch
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
      int mt, nt;
      tc_raster(p.raster_n, p.group, p.m_tiles, p.n_tiles, tile, mt, nt);
      const int m0 = mt * TC_BM, n0 = nt * TC_BN;
      if (!mbar_wait(&bars->tmem_full[acc], acc_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const int row0 = m0 + q * 32;
      const int64_t row = row0 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * TC_BN;
      // act-bwd: the pre-activation of the next 32 columns is loaded while
      // the current ones are processed
      float a_next[32];
      if (bwd) {
        if (row < p.M) {
          load_pre32(e, row, n0, min(32, p.N - n0), a_next);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) a_next[i] = 0.0f;
        }
      }
      if (ce) {  // the warp's 256 columns are two statistics tiles
        const int64_t y = row < p.M ? ce_row_label(e, row) : -1;
        float zy = 0.0f, a[32];
        bool have = false;
        for (int tt = 0; tt < TC_BN / kStatsTileN; ++tt) {
          const int tc0 = n0 + tt * kStatsTileN;
          if (tc0 >= p.N) break;  // warp-uniform
          ce_stats_tile(e, t_row + tt * kStatsTileN, tc0, p.N, row < p.M, row, y, zy, have,
                        [&](int64_t col0, int n, float(&v)[32]) {
                          if (!p.tma_store) {
                            if (row < p.M) epilogue_run32(e, row, col0, n, v);
                            return;
                          }
                          tc_store_chunk<0>(e, &tmD, &tmD2, stg_f32, stg_bf16, lane, row0, static_cast<int>(col0), v,
                                            a);
                        });
        }
        if (have) e.ce_zy[row] = zy;
      }
      for (int c = 0; !ce && c < TC_BN / 32; ++c) {
        const int col0 = n0 + c * 32;
        if (col0 >= p.N) break;  // warp-uniform
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        float a[32];
        if (bwd) {
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = a_next[i];
          if (row < p.M && col0 + 32 < p.N && c + 1 < TC_BN / 32)
            load_pre32(e, row, col0 + 32, min(32, p.N - col0 - 32), a_next);
        }
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        const int n = min(32, p.N - col0);
        if (!p.tma_store) {
          if (row < p.M) epilogue_run32(e, row, col0, n, v);
          continue;
        }
        // TMA store path: the box (32 rows x 32 columns) is clipped to the
        // tensor by the TMA unit, so rows >= M and columns >= N are dropped.
        tc_store_chunk<0>(e, &tmD, &tmD2, stg_f32, stg_bf16, lane, row0, col0, v, a);
      }
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

bool tc_make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_cols,
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

bool tc_make_out_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int dtype) {
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

int tc_num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// Tile order and L2 policy.  Consecutive tiles walk groups of 16 M-tiles
// (M fastest), so a wave of tiles touches a compact block of A rows and B
// columns and consecutive waves share the group's A slabs.
// TPS_GEMM_GROUP overrides the group size.  TPS_GEMM_L2_HINTS=1 marks A (the
// operand a group revisits) evict-last and B evict-first; two digits "ab"
// choose each operand's policy (0 none, 1 evict-first, 2 evict-last).  The
// default carries no hint: every hinted form measured slower.
void tc_raster_choice(int m_tiles, int* raster_n, int* group, int* pol_a, int* pol_b) {
  const char* gv = getenv("TPS_GEMM_GROUP");
  const char* hv = getenv("TPS_GEMM_L2_HINTS");
  const int g = (gv && atoi(gv) > 0) ? atoi(gv) : TC_GROUP_M;
  *raster_n = 0;
  *group = g < m_tiles ? g : m_tiles;
  *pol_a = 0;
  *pol_b = 0;
  if (hv == nullptr) return;
  if (hv[0] >= '0' && hv[0] <= '2' && hv[1] >= '0' && hv[1] <= '2' && hv[2] == '\0') {
    *pol_a = hv[0] - '0';
    *pol_b = hv[1] - '0';
  } else if (atoi(hv) != 0) {
    *pol_a = 2;
    *pol_b = 1;
  }
}

// The tensor-core path needs bf16 operands that TMA can describe: 16-byte
// aligned base, unit stride in one dimension and a pitch that is a multiple
// of 16 bytes.
// The gated forms need their second operands to qualify too, with the same
// contiguous dimension.
bool gemm_tc_supported(const GemmDesc& g) {
  if (g.in_dtype != TPS_BF16) return false;
  if (g.M < 1 || g.N < 1 || g.K < 1 || g.K2 < 0 || g.K3 < 0) return false;
  if (g.M >= (1ll << 31) || g.N >= (1ll << 31) || g.K + g.K2 + g.K3 >= (1ll << 31)) return false;
  const bool k_segs = g.K2 > 0 || g.K3 > 0;
  if (g.epi.mode == EPI_GLU_FWD && (g.b_up == nullptr || k_segs || g.n_segs > 1)) return false;
  if (g.epi.mode == EPI_CE_STATS && (g.epi.d_dtype != TPS_BF16 || g.epi.stats == nullptr || g.epi.stats_b == nullptr ||
                                     g.epi.ce_shift == nullptr ||
                                     g.epi.ce_labels == nullptr || g.epi.ce_zy == nullptr))
    return false;
  if (g.n_segs < 1 || g.n_segs > 3 || (g.n_segs > 1 && k_segs)) return false;
  if ((g.n_segs > 1 || k_segs) && g.epi.mode != EPI_STORE) return false;  // segments: plain stores only
  auto ok_operand = [](const void* ptr, int64_t s_outer, int64_t s_inner, int64_t inner_extent) {
    if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return false;
    if (s_inner != 1) return false;
    if ((s_outer * 2) % 16 != 0 || s_outer < inner_extent) return false;
    return s_outer * 2 < (1ll << 40);
  };
  const bool a_ok = (g.a_sk == 1) ? ok_operand(g.a, g.a_sm, g.a_sk, g.K) : ok_operand(g.a, g.a_sk, g.a_sm, g.M);
  if (!a_ok) return false;
  if (g.n_segs > 1) {  // each segment's B and output, boundaries on 128-column blocks
    int64_t n = 0;
    for (int s = 0; s < g.n_segs; ++s) {
      const int64_t c = g.n_cols[s];
      if (c < 1 || (s + 1 < g.n_segs && c % 128 != 0)) return false;
      if ((g.nb_sk[s] == 1) != (g.b_sk == 1)) return false;
      if (!((g.nb_sk[s] == 1) ? ok_operand(g.nb[s], g.nb_sn[s], 1, g.K) : ok_operand(g.nb[s], g.nb_sk[s], g.nb_sn[s], c)))
        return false;
      const int es = g.epi.d_dtype == TPS_F32 ? 4 : 2;
      if ((reinterpret_cast<uintptr_t>(g.nd[s]) & 15u) != 0 || (g.nldd[s] * es) % 16 != 0 || g.nldd[s] < c)
        return false;
      n += c;
    }
    return n == g.N;
  }
  const bool b_ok = (g.b_sk == 1) ? ok_operand(g.b, g.b_sn, g.b_sk, g.K) : ok_operand(g.b, g.b_sk, g.b_sn, g.N);
  if (!b_ok) return false;
  if (g.epi.mode == EPI_GLU_FWD &&
      !((g.b_sk == 1) ? ok_operand(g.b_up, g.b_sn, g.b_sk, g.K) : ok_operand(g.b_up, g.b_sk, g.b_sn, g.N)))
    return false;
  const void* as[2] = {g.a2, g.a3};
  const void* bs[2] = {g.b2, g.b3};
  const int64_t ks[2] = {g.K2, g.K3}, asm_[2] = {g.a2_sm, g.a3_sm}, ask[2] = {g.a2_sk, g.a3_sk};
  const int64_t bsk[2] = {g.b2_sk, g.b3_sk}, bsn[2] = {g.b2_sn, g.b3_sn};
  for (int s = 0; s < 2; ++s) {
    if (ks[s] == 0) continue;
    if ((ask[s] == 1) != (g.a_sk == 1) || (bsk[s] == 1) != (g.b_sk == 1)) return false;
    const bool ao = (ask[s] == 1) ? ok_operand(as[s], asm_[s], 1, ks[s]) : ok_operand(as[s], ask[s], asm_[s], g.M);
    const bool bo = (bsk[s] == 1) ? ok_operand(bs[s], bsn[s], 1, ks[s]) : ok_operand(bs[s], bsk[s], bsn[s], g.N);
    if (!ao || !bo) return false;
  }
  return true;
}

// Output maps for the TMA-store epilogue; false when an output cannot be
// described (the kernels then store directly).  `td3` (U of EPI_GLU_FWD)
// may be null for the other modes.
bool tc_make_output_maps(const GemmDesc& g, CUtensorMap* td, CUtensorMap* td2, CUtensorMap* td3) {
  memset(td, 0, sizeof(*td));
  memset(td2, 0, sizeof(*td2));
  if (td3) memset(td3, 0, sizeof(*td3));
  if (g.n_segs > 1) {  // one map per column segment, in td, td2, td3
    CUtensorMap* maps[3] = {td, td2, td3};
    for (int s = 0; s < g.n_segs; ++s)
      if (maps[s] == nullptr || !tc_make_out_map(maps[s], g.nd[s], g.M, g.n_cols[s], g.nldd[s], g.epi.d_dtype))
        return false;
    return true;
  }
  if (g.epi.mode == EPI_GLU_FWD) {  // Hg and U fp32, A bf16, 128-wide hidden-unit tiles
    return td3 != nullptr && g.epi.d2_dtype == TPS_BF16 &&
           tc_make_out_map(td, g.epi.d, g.M, g.N, g.epi.ldd, TPS_F32) &&
           tc_make_out_map(td3, g.epi.d3, g.M, g.N, g.epi.ldd3, TPS_F32) &&
           tc_make_out_map(td2, g.epi.d2, g.M, g.N, g.epi.ldd2, TPS_BF16);
  }
  if (g.epi.mode == EPI_GLU_BWD) {  // dHg and dU leave as two bf16 boxes
    return g.epi.d_dtype == TPS_BF16 && g.epi.d2_dtype == TPS_BF16 &&
           tc_make_out_map(td, g.epi.d, g.M, g.N, g.epi.ldd, TPS_BF16) &&
           tc_make_out_map(td2, g.epi.d2, g.M, g.N, g.epi.ldd2, TPS_BF16);
  }
  if (g.epi.mode == EPI_ACT_FWD || g.epi.mode == EPI_GLU_UP) {
    bool ok = true;
    const int pre_dtype = g.epi.mode == EPI_ACT_FWD ? g.epi.d_dtype : TPS_F32;  // U of EPI_GLU_UP is fp32
    if (g.epi.d != nullptr) ok = tc_make_out_map(td, g.epi.d, g.M, g.N, g.epi.ldd, pre_dtype);
    return ok && g.epi.d2_dtype == TPS_BF16 && tc_make_out_map(td2, g.epi.d2, g.M, g.N, g.epi.ldd2, TPS_BF16);
  }
  return tc_make_out_map(td, g.epi.d, g.M, g.N, g.epi.ldd, g.epi.d_dtype);
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

int launch_gemm_tc1(const GemmDesc& g, uint32_t* dev_err, cudaStream_t stream) {
  // the gated forms and a second K segment exist on CTA pairs only
  if (g.epi.mode == EPI_GLU_FWD || g.epi.mode == EPI_GLU_BWD || g.K2 > 0 || g.K3 > 0 || g.n_segs > 1)
    return TPS_ERR_ARG;
  const bool a_mn = (g.a_sk != 1);
  const bool b_mn = (g.b_sk != 1);
  CUtensorMap ta, tb;
  bool ok = a_mn ? tc_make_map(&ta, g.a, g.K, g.M, g.a_sk, 64, TC_BK)     // stored K x M
                 : tc_make_map(&ta, g.a, g.M, g.K, g.a_sm, TC_BK, TC_BM);  // stored M x K
  ok = ok && (b_mn ? tc_make_map(&tb, g.b, g.K, g.N, g.b_sk, 64, TC_BK)    // stored K x N
                   : tc_make_map(&tb, g.b, g.N, g.K, g.b_sn, TC_BK, TC_BN)); // stored N x K
  if (!ok) return TPS_ERR_CUDA;

  TcParams p;
  p.M = static_cast<int>(g.M);
  p.N = static_cast<int>(g.N);
  p.K = static_cast<int>(g.K);
  p.m_tiles = static_cast<int>((g.M + TC_BM - 1) / TC_BM);
  p.n_tiles = static_cast<int>((g.N + TC_BN - 1) / TC_BN);
  p.k_tiles = static_cast<int>((g.K + TC_BK - 1) / TC_BK);
  p.num_tiles = p.m_tiles * p.n_tiles;
  tc_raster_choice(p.m_tiles, &p.raster_n, &p.group, &p.pol_a, &p.pol_b);
  p.epi = g.epi;
  p.err = dev_err;
  CUtensorMap td, td2;
  p.tma_store = tc_make_output_maps(g, &td, &td2, nullptr) ? 1 : 0;
  const int sms = tc_num_sms();
  const int grid = p.num_tiles < sms ? p.num_tiles : sms;

  if (!a_mn && !b_mn) return launch_typed<false, false>(g, ta, tb, td, td2, p, grid, stream);
  if (!a_mn && b_mn) return launch_typed<false, true>(g, ta, tb, td, td2, p, grid, stream);
  if (a_mn && !b_mn) return launch_typed<true, false>(g, ta, tb, td, td2, p, grid, stream);
  return launch_typed<true, true>(g, ta, tb, td, td2, p, grid, stream);
}

// Kernel choice: CTA pairs (gemm_tc2.cu) when M spans at least one 256-row
// pair tile, else single CTAs.  TPS_GEMM_KERNEL=1 or 2 forces one, except
// that the gated forms and contraction or column segments always run on
// CTA pairs.
int launch_gemm_tc(const GemmDesc& g, uint32_t* dev_err, cudaStream_t stream) {
  const char* kv = getenv("TPS_GEMM_KERNEL");
  const int forced = kv ? atoi(kv) : 0;
  const bool pair_only =
      g.epi.mode == EPI_GLU_FWD || g.epi.mode == EPI_GLU_BWD || g.K2 > 0 || g.K3 > 0 || g.n_segs > 1;
  const bool pair = pair_only || forced == 2 || (forced != 1 && g.M >= 256);
  return pair ? launch_gemm_tc2(g, dev_err, stream) : launch_gemm_tc1(g, dev_err, stream);
}

}  // namespace tps
