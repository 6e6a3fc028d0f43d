// gemm_tc2.cu -- the tensor-core GEMM on CTA pairs (tcgen05 cta_group::2).
//
// A cluster of two CTAs on neighbouring SMs computes one 256 x 256 output
// tile: each CTA stages its own 128 rows of A and its own 128 columns of B
// (so B is loaded once per pair, halving B's shared-memory footprint and
// L2->SM traffic per SM against the one-CTA kernel), the even CTA issues
// tcgen05.mma with M=256, and each CTA's tensor memory receives its 128
// rows of the fp32 accumulator.  The shared memory this frees holds eight
// epilogue warps with double-buffered TMA-store staging.
//
// Same GEMM, shard semantics and epilogues as gemm_tc.cu ("Sharded GEMM与
// Backprop", 解题路线 steps 2-4; "第 6 课：张量并行 TP", core concept 1).
//
// Synchronisation (barriers live at the same offsets in both CTAs):
//   full[s]       even CTA only: its producer expects both CTAs' bytes and
//                 both CTAs' TMA loads complete on it
//   empty[s]      each CTA: arrived by the MMA commit multicast to the pair
//   tmem_full[b]  each CTA: arrived by the MMA commit multicast to the pair
//   tmem_empty[b] even CTA only: one arrival per epilogue warp of each CTA
//
// Gated MLP forward (EPI_GLU_FWD): the even CTA stages 128 columns of the
// gate weight and the odd CTA the same 128 columns of the up weight, so each
// CTA's accumulator holds, for its 128 rows, the gate (columns 0..127) and
// the up projection (128..255) of the same 128 hidden units, and the
// epilogue forms phi(gate) * up without leaving the SM.  A pair tile then
// covers 128 hidden units.
//
// Further contraction segments (GemmDesc::K2, K3) continue the K loop with
// the operands A2, B2 (and A3, B3) into the same accumulator:
// D = A B + A2 B2 + A3 B3.  Column segments (GemmDesc::n_segs) run up to
// three GEMMs that share A as one launch over their concatenated columns:
// each CTA's 128 B columns, and each epilogue warp's 128 output columns,
// lie in one segment, whose own B and output maps they use.
//
// Warp roles (320 threads, one CTA per SM):
//   warp 0      TMA producer (one thread)
//   warp 1      TMEM allocator; MMA issuer on the even CTA (one thread)
//   warps 2..9  epilogue: warp w reads TMEM lanes 32*(w%4)..+31 and
//               columns 128*((w-2)/4)..+127 of the accumulator (gated:
//               hidden units 64*((w-2)/4)..+63, gate and up)
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "tc_common.cuh"

namespace tps {

constexpr int T2_BM = 128;      // rows per CTA (256 per pair)
constexpr int T2_BN = 256;      // columns per pair tile
constexpr int T2_BN_CTA = 128;  // B columns staged by each CTA
constexpr int T2_MAX_STAGES = 5;
constexpr int T2_A_BYTES = T2_BM * TC_BK * 2;      // 16 KB
constexpr int T2_B_BYTES = T2_BN_CTA * TC_BK * 2;  // 16 KB
constexpr int T2_STAGE_BYTES = T2_A_BYTES + T2_B_BYTES;
constexpr int T2_THREADS = 320;
constexpr int T2_EPI_WARPS = 8;
constexpr uint32_t T2_TMEM_COLS = 2 * T2_BN;  // two fp32 accumulators
constexpr int T2_STG_BUF = TC_STG_F32_BYTES + TC_STG_BF16_BYTES;  // 6 KB, one buffer
static_assert(T2_BN / 2 == kStatsTileN, "each epilogue warp covers one CE statistics tile");

struct T2Barriers {
  uint64_t full[T2_MAX_STAGES];
  uint64_t empty[T2_MAX_STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint64_t sched_full[kUnitRing];  // PairUnits ring (dynamic schedule)
  uint64_t sched_empty[kUnitRing];
  int32_t sched_unit[kUnitRing];
  uint32_t tmem_slot;
  uint32_t abort;
};
// Readers of each unit the dynamic schedule publishes: the even CTA's MMA
// thread, both CTAs' epilogue warps and the odd CTA's producer.
constexpr int T2_SCHED_READERS = 2 + 2 * T2_EPI_WARPS;


// Tensor maps of one launch: a[s], b[s] are the operands of contraction
// segment s (b[1] is the up weight of the gated forward); with column
// segments b[s] and d[s] belong to column segment s; otherwise d[0], d[1],
// d[2] are the outputs D, D2 and D3.
struct T2Maps {
  CUtensorMap a[3], b[3], d[3];
};

struct T2Params {
  int M, N, K;
  int m_tiles, n_tiles, k_tiles, num_tiles;  // m_tiles counts 256-row pair tiles
  // K split (GemmDesc::ksplit): work unit u is tile u % num_tiles and run
  // u / num_tiles of kt_run K tiles; num_units = num_tiles * ksplit
  int ksplit, kt_run, num_units;
  uint32_t* kflags;
  uint32_t* unit_counter;  // dynamic schedule (GemmDesc::unit_counter), else nullptr
  int k_end[3];                              // cumulative K tiles of the contraction segments
  int n_segs, n_end[3];                      // column segments: cumulative column ends
  int glu;                                   // EPI_GLU_FWD: b[1] is the up weight
  int raster_n, group;
  int pol_a, pol_b;  // L2 policy kinds of the operand loads (0 none, 1 evict-first, 2 evict-last)
  int tma_store;
  Epilogue epi;
  uint32_t* err;
};

// Epilogue families, compiled as separate kernels so that one form's extra
// live registers and staging do not cost another its registers or stages.
//   T2_PLAIN    EPI_STORE, EPI_CE_STATS (one output box per chunk)
//   T2_ACT16    EPI_ACT_FWD, EPI_ACT_BWD with a bf16 pre-activation
//   T2_ACT      EPI_ACT_FWD, EPI_ACT_BWD with an fp32 pre-activation, EPI_GLU_UP
//   T2_GLU_FWD  EPI_GLU_FWD
//   T2_GLU_BWD  EPI_GLU_BWD
//   T2_SEG      EPI_STORE with contraction or column segments
enum T2Family : int { T2_PLAIN = 0, T2_GLU_FWD = 1, T2_GLU_BWD = 2, T2_SEG = 3, T2_ACT = 4, T2_ACT16 = 5 };

// Shared-memory layout per family: five operand stages of 32 KB and the
// epilogue's staging.  With four stages the mainloop measured latency-bound
// (the MLP GEMMs ran 8 % and the CE GEMMs 4-5 % slower than with five at
// the Llama shapes); a sixth stage, where it fits, measured slower again.
//   plain, segmented  one 4 KB box per warp (fp32 and bf16 share it),
//                     double-buffered                       -> 5 stages
//   act, bf16 pre     two bf16 boxes (4 KB), double-buffered -> 5 stages
//   act, fp32 pre     fp32 + bf16 boxes (6 KB), single       -> 5 stages
//   gated backward    two bf16 boxes (4 KB), double-buffered -> 5 stages
//   gated forward     Hg then U through one fp32 box, A bf16
//                     (6 KB), single-buffered                -> 5 stages
template <int FAM>
struct T2Layout {
  static constexpr bool kStoreOnly = FAM == T2_PLAIN || FAM == T2_SEG;
  static constexpr int kStages = 5;
  static constexpr bool kTwoBf16 = FAM == T2_GLU_BWD || FAM == T2_ACT16;  // two bf16 boxes per buffer
  static constexpr int kBufBytes = kStoreOnly ? TC_STG_F32_BYTES : (kTwoBf16 ? 2 * TC_STG_BF16_BYTES : T2_STG_BUF);
  static constexpr int kBufs = (kTwoBf16 || kStoreOnly) ? 2 : 1;
  // offset of the second (activation) box of an activation-family buffer
  static constexpr int kSecondBox = kTwoBf16 ? TC_STG_BF16_BYTES : TC_STG_F32_BYTES;
  static constexpr int kWarpStaging = kBufs * kBufBytes;
  static constexpr size_t kSmem =
      1024 + kStages * T2_STAGE_BYTES + T2_EPI_WARPS * kWarpStaging + sizeof(T2Barriers);
  static_assert(kStages <= T2_MAX_STAGES, "barrier arrays hold T2_MAX_STAGES stages");
  static_assert(kSmem <= 232448, "exceeds the opt-in shared memory per block");
};

// A paired operand load that carries an L2 policy only when one was chosen.
__device__ __forceinline__ void pair_load(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int32_t c0,
                                          int32_t c1, int kind, uint64_t policy) {
  if (kind != 0)
    tma_load_2d_pair_hint(dst, map, bar_cluster, c0, c1, policy);
  else
    tma_load_2d_pair(dst, map, bar_cluster, c0, c1);
}

template <bool A_MN, bool B_MN, int FAM>
__global__ void __launch_bounds__(T2_THREADS, 1)
    gemm_tc2_kernel(const __grid_constant__ T2Maps m, const T2Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  using L = T2Layout<FAM>;
  constexpr int T2_STAGES = L::kStages;
  uint8_t* staging = smem + T2_STAGES * T2_STAGE_BYTES;  // 1024-aligned
  T2Barriers* bars = reinterpret_cast<T2Barriers*>(staging + T2_EPI_WARPS * L::kWarpStaging);
  volatile uint32_t* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < T2_STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->tmem_full[b], 1);
      mbar_init(&bars->tmem_empty[b], 2 * T2_EPI_WARPS);
    }
    mbar_init(&bars->drain, 1);
    for (int s = 0; s < kUnitRing; ++s) {
      mbar_init(&bars->sched_full[s], 1);
      mbar_init(&bars->sched_empty[s], T2_SCHED_READERS);
    }
    bars->abort = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < 3; ++s) {
      const bool k_used = s == 0 || p.k_end[s] > p.k_end[s - 1];
      if (k_used) tma_prefetch_desc(&m.a[s]);
      if (k_used || s < p.n_segs || (s == 1 && p.glu)) tma_prefetch_desc(&m.b[s]);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(&bars->tmem_slot, T2_TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_slot;
  const uint32_t full0_leader = cluster_map(smem_u32(&bars->full[0]), 0);
  const uint32_t tmem_empty0_leader = cluster_map(smem_u32(&bars->tmem_empty[0]), 0);
  PairUnits units;
  units.init(bars->sched_full, bars->sched_empty, bars->sched_unit, abort_flag, p.err, p.unit_counter, pair, npairs,
             p.num_units, warp == 0 && rank == 0);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      bool ok = true;
      const uint64_t pa = tc_policy(p.pol_a), pb = tc_policy(p.pol_b);
      for (int u = units.take(); ok && u >= 0; u = units.take()) {
        const int tile = u % p.num_tiles, run = u / p.num_tiles;
        const int kt_begin = run * p.kt_run, kt_end = min(p.k_tiles, kt_begin + p.kt_run);
        int mt, nt;
        tc_raster(p.raster_n, p.group, p.m_tiles, p.n_tiles, tile, mt, nt);
        const int m0 = mt * 2 * T2_BM + static_cast<int>(rank) * T2_BM;
        // gated: both CTAs stage the same 128 hidden units, gate or up
        int nb0 = p.glu ? nt * T2_BN_CTA : nt * T2_BN + static_cast<int>(rank) * T2_BN_CTA;
        int nseg = 0;  // column segment of this CTA's 128 B columns
        if constexpr (FAM == T2_SEG) {
          while (nseg < p.n_segs - 1 && nb0 >= p.n_end[nseg]) ++nseg;
          if (nseg > 0) nb0 -= p.n_end[nseg - 1];
        }
        const CUtensorMap* mb0 = (p.glu && rank == 1) ? &m.b[1] : &m.b[nseg];
        for (int kt = kt_begin; kt < kt_end; ++kt) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * T2_STAGE_BYTES;
          uint8_t* sb = sa + T2_A_BYTES;
          if (rank == 0) mbar_expect_tx(&bars->full[stage], 2 * T2_STAGE_BYTES);
          const uint32_t fb = full0_leader + stage * static_cast<uint32_t>(sizeof(uint64_t));
          int ks = 0;  // contraction segment of this K tile
          if constexpr (FAM == T2_SEG)
            while (ks < 2 && kt >= p.k_end[ks]) ++ks;
          const CUtensorMap* ma = &m.a[ks];
          const CUtensorMap* mb = ks > 0 ? &m.b[ks] : mb0;
          const int k0 = (kt - (ks > 0 ? p.k_end[ks - 1] : 0)) * TC_BK;
          if (!A_MN) {
            pair_load(sa, ma, fb, k0, m0, p.pol_a, pa);
          } else {
#pragma unroll
            for (int j = 0; j < T2_BM / 64; ++j)
              pair_load(sa + j * TC_MN_BOX_BYTES, ma, fb, m0 + 64 * j, k0, p.pol_a, pa);
          }
          if (!B_MN) {
            pair_load(sb, mb, fb, k0, nb0, p.pol_b, pb);
          } else {
#pragma unroll
            for (int j = 0; j < T2_BN_CTA / 64; ++j)
              pair_load(sb + j * TC_MN_BOX_BYTES, mb, fb, nb0 + 64 * j, k0, p.pol_b, pb);
          }
          ++issued;
          if (++stage == T2_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain (even CTA: the full barriers count both CTAs' bytes).
      if (rank == 0) {
        const int64_t first = issued > T2_STAGES ? issued - T2_STAGES : 0;
        for (int64_t i = first; i < issued; ++i)
          mbar_wait_drain(&bars->full[i % T2_STAGES], static_cast<uint32_t>((i / T2_STAGES) & 1), p.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(2 * T2_BM, T2_BN, A_MN, B_MN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int u = units.take(); ok && u >= 0; u = units.take()) {
        const int run = u / p.num_tiles;
        const int kt_begin = run * p.kt_run, kt_end = min(p.k_tiles, kt_begin + p.kt_run);
        if (!mbar_wait(&bars->tmem_empty[acc], acc_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * T2_BN;
        for (int kt = kt_begin; kt < kt_end; ++kt) {
          if (!mbar_wait(&bars->full[stage], phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * T2_STAGE_BYTES);
          const uint32_t sb = sa + T2_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk) {
            const uint64_t ad = A_MN ? smem_desc_sw128(sa + kk * 2048, TC_MN_BOX_BYTES, 1024)
                                     : smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(sb + kk * 2048, TC_MN_BOX_BYTES, 1024)
                                     : smem_desc_sw128(sb + kk * 32, 16, 1024);
            tc_mma_f16_pair(d_tmem, ad, bd, idesc, (kt != kt_begin || kk != 0) ? 1u : 0u);
          }
          tc_commit_pair_mc(&bars->empty[stage], 0x3);  // frees the stage in both CTAs
          if (++stage == T2_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(&bars->tmem_full[acc], 0x3);  // both CTAs' accumulators complete
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      tc_commit_pair(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, p.err);
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int ew = warp - 2;       // 0..7
    const int q = warp & 3;        // TMEM lane quadrant
    const int h = ew >> 2;         // column half of the 256-column tile
    uint8_t* stg = staging + ew * L::kWarpStaging;
    const Epilogue& e = p.epi;
    const bool ce = FAM == T2_PLAIN && e.mode == EPI_CE_STATS;
    const bool bwd = (FAM == T2_ACT || FAM == T2_ACT16) && p.tma_store &&
                     (e.mode == EPI_ACT_BWD || e.mode == EPI_GLU_UP);  // AUX prefetch
    constexpr bool glu = FAM == T2_GLU_FWD;
    constexpr bool gbwd = FAM == T2_GLU_BWD;
    // accumulator columns this warp drains: 128 (gated: 64 gate + 64 up)
    const int warp_cols = glu ? T2_BN_CTA / 2 : T2_BN / 2;
    uint32_t acc = 0, acc_phase = 0, chunk = 0;
    for (int u = units.take_warp(lane); u >= 0; u = units.take_warp(lane)) {
      const int tile = u % p.num_tiles, run = u / p.num_tiles;
      int mt, nt;
      tc_raster(p.raster_n, p.group, p.m_tiles, p.n_tiles, tile, mt, nt);
      const int m0 = mt * 2 * T2_BM + static_cast<int>(rank) * T2_BM;
      // first output column of this warp's part of the tile
      const int nh0 = glu ? nt * T2_BN_CTA + h * warp_cols : nt * T2_BN + h * warp_cols;
      int oseg = 0, ocol0 = 0;  // column segment of these columns: its output map and first column
      if constexpr (FAM == T2_SEG) {
        while (oseg < p.n_segs - 1 && nh0 >= p.n_end[oseg]) ++oseg;
        ocol0 = oseg > 0 ? p.n_end[oseg - 1] : 0;
      }
      const int row0 = m0 + q * 32;
      const int64_t row = row0 + lane;
      // The first chunk's AUX input does not depend on the accumulator: it
      // is loaded before waiting for it.
      float a_next[32];
      if (bwd) {
        if (row < p.M && nh0 < p.N) {
          load_pre32(e, row, nh0, min(32, p.N - nh0), a_next);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) a_next[i] = 0.0f;
        }
      }
      if (p.ksplit > 1 && run > 0) {
        // K split: the previous run of this tile (all 2 x 8 epilogue warps
        // of its pair) must be in memory before this run adds to it.
        uint32_t ready = 1u;
        if (lane == 0) {
          const uint32_t need = static_cast<uint32_t>(2 * T2_EPI_WARPS * run);
          const uint64_t t0 = globaltimer_ns();
          while (ld_acquire_gpu(p.kflags + tile) < need) {
            if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
              if (!*abort_flag) {
                *abort_flag = 1u;
                atomicOr(p.err, TPS_DEVERR_TIMEOUT);
              }
              ready = 0u;
              break;
            }
            __nanosleep(256);
          }
          fence_async_global();
        }
        if (!__shfl_sync(0xffffffffu, ready, 0)) break;
      }
      if (!mbar_wait(&bars->tmem_full[acc], acc_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t t_row =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * T2_BN + static_cast<uint32_t>(h * warp_cols);
      bool ce_done = false;
      if constexpr (FAM == T2_PLAIN) {
        if (ce) {  // the warp's 128 columns are one statistics tile
          ce_done = true;
          if (nh0 < p.N) {
            const int64_t y = row < p.M ? ce_row_label(e, row) : -1;
            float zy = 0.0f, a[32];
            bool have = false;
            ce_stats_tile(e, t_row, nh0, p.N, row < p.M, row, y, zy, have, [&](int64_t col0, int n, float(&v)[32]) {
              if (!p.tma_store) {
                if (row < p.M) epilogue_run32(e, row, col0, n, v);
                return;
              }
              uint8_t* buf = stg + (L::kBufs == 2 ? (chunk & 1u) * L::kBufBytes : 0u);
              tc_store_chunk<L::kBufs - 1, true>(e, &m.d[0], &m.d[1], buf, buf, lane, row0, static_cast<int>(col0),
                                                 v, a);
              ++chunk;
            });
            if (have) e.ce_zy[row] = zy;
          }
        }
      }
      for (int c = 0; !ce_done && c < warp_cols / 32; ++c) {
        const int col0 = nh0 + c * 32;
        if (col0 >= p.N) break;  // warp-uniform
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        if constexpr (glu) {  // gate in r, the same hidden units' up projection 128 columns on
          uint32_t r2[32];
          tmem_ld_32x32b_x32(t_row + T2_BN_CTA + c * 32, r2);
          tmem_ld_wait();
          float hg[32], u[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            hg[i] = __uint_as_float(r[i]);
            u[i] = __uint_as_float(r2[i]);
          }
          if (!p.tma_store) {
            if (row < p.M) epilogue_glu_run32(e, row, col0, min(32, p.N - col0), hg, u);
          } else {
            tc_store_glu_chunk(e, &m.d[0], &m.d[1], &m.d[2], stg, lane, row0, col0, hg, u);
          }
          continue;
        }
        if constexpr (gbwd) {
          if (p.tma_store) {
            float hg[32], u[32];  // Hg and U of these 32 columns
            if (row < p.M) {
              load_run32(e.aux + row * e.ld_aux + col0, min(32, p.N - col0), hg);
              load_run32(e.aux2 + row * e.ld_aux2 + col0, min(32, p.N - col0), u);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) hg[i] = u[i] = 0.0f;
            }
            tmem_ld_wait();
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
            uint8_t* buf = stg + (chunk & 1u) * L::kBufBytes;  // dU box, then the dHg box
            tc_store_glu_bwd_chunk(e, &m.d[0], &m.d[1], buf, buf + TC_STG_BF16_BYTES, lane, row0, col0, v, hg, u);
            ++chunk;
          } else {
            tmem_ld_wait();
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
            if (row < p.M) epilogue_glu_bwd_run32(e, row, col0, min(32, p.N - col0), v);
          }
          continue;
        }
        float a[32];
        if (bwd) {
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = a_next[i];
          if (row < p.M && col0 + 32 < p.N && c + 1 < warp_cols / 32)
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
        // the fp32 and bf16 slots (store-only: one shared box), single- or double-buffered
        uint8_t* buf = stg + (L::kBufs == 2 ? (chunk & 1u) * L::kBufBytes : 0u);
        if constexpr (FAM == T2_PLAIN) {
          if (run > 0) {  // K split: add this run's partial tile to the output
            tc_store_chunk<L::kBufs - 1, true, true>(e, &m.d[0], &m.d[1], buf, buf, lane, row0, col0, v, a);
            ++chunk;
            continue;
          }
        }
        tc_store_chunk<L::kBufs - 1, L::kStoreOnly>(e, &m.d[oseg], &m.d[1], buf,
                                                    L::kStoreOnly ? buf : buf + L::kSecondBox, lane, row0,
                                                    col0 - ocol0, v, a);
        ++chunk;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tmem_empty0_leader + acc * static_cast<uint32_t>(sizeof(uint64_t)));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
      if (p.ksplit > 1) {  // K split: this warp's part of the run is in memory
        if (lane == 0) {
          bulk_wait0();
          fence_async_global();
          red_release_gpu_add(p.kflags + tile, 1u);
        }
        __syncwarp();
      }
    }
    if (p.tma_store && lane == 0) bulk_wait0();
  }

  tc_fence_before();
  cluster_sync();  // the pair's MMAs, loads and epilogues are all finished
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, T2_TMEM_COLS);
}

// ------------------------------------------------------------------ host

bool tc_make_output_maps(const GemmDesc& g, CUtensorMap* td, CUtensorMap* td2, CUtensorMap* td3);

template <bool A_MN, bool B_MN, int FAM>
static int launch_pair_typed(const GemmDesc& g, const T2Maps& m, const T2Params& p, int pairs,
                             cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_tc2_kernel<A_MN, B_MN, FAM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(T2Layout<FAM>::kSmem));
  });
  if (attr_err != cudaSuccess) return TPS_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.blockDim = dim3(T2_THREADS, 1, 1);
  cfg.dynamicSmemBytes = T2Layout<FAM>::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.ksplit > 1) {
    // Under a K split an epilogue waits for a run that another pair holds:
    // launch only as many pairs as can be resident at once, so that every
    // run it waits for belongs to a running pair.
    static std::once_flag cl_once;
    static int max_clusters = 0;
    std::call_once(cl_once, [&cfg] {
      if (cudaOccupancyMaxActiveClusters(&max_clusters, gemm_tc2_kernel<A_MN, B_MN, FAM>, &cfg) != cudaSuccess)
        max_clusters = 0;
    });
    if (max_clusters < 1) return TPS_ERR_CUDA;
    if (pairs > max_clusters) cfg.gridDim = dim3(static_cast<unsigned>(2 * max_clusters), 1, 1);
  }
  const double flops = 2.0 * double(g.M) * double(g.N) * double(g.K + g.K2 + g.K3) * (p.glu ? 2.0 : 1.0);
  ProfScope prof("gemm_tc", g.name, flops, 0.0, stream);
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, gemm_tc2_kernel<A_MN, B_MN, FAM>, m, p);
  note_launch();
  return e == cudaSuccess ? TPS_OK : TPS_ERR_CUDA;
}

template <int FAM>
static int launch_pair_majors(const GemmDesc& g, const T2Maps& m, const T2Params& p, int pairs, bool a_mn,
                              bool b_mn, cudaStream_t stream) {
  if (!a_mn && !b_mn) return launch_pair_typed<false, false, FAM>(g, m, p, pairs, stream);
  if (!a_mn && b_mn) return launch_pair_typed<false, true, FAM>(g, m, p, pairs, stream);
  if (a_mn && !b_mn) return launch_pair_typed<true, false, FAM>(g, m, p, pairs, stream);
  return launch_pair_typed<true, true, FAM>(g, m, p, pairs, stream);
}

static int launch_pair_family(const GemmDesc& g, const T2Maps& m, const T2Params& p, int pairs, bool a_mn,
                              bool b_mn, cudaStream_t stream) {
  if (g.epi.mode == EPI_GLU_FWD) return launch_pair_majors<T2_GLU_FWD>(g, m, p, pairs, a_mn, b_mn, stream);
  if (g.epi.mode == EPI_GLU_BWD) return launch_pair_majors<T2_GLU_BWD>(g, m, p, pairs, a_mn, b_mn, stream);
  if (g.n_segs > 1 || g.K2 > 0 || g.K3 > 0) {
    if (g.epi.mode != EPI_STORE) return TPS_ERR_ARG;
    return launch_pair_majors<T2_SEG>(g, m, p, pairs, a_mn, b_mn, stream);
  }
  const bool pre16 = (g.epi.mode == EPI_ACT_FWD && (g.epi.d == nullptr || g.epi.d_dtype == TPS_BF16)) ||
                     (g.epi.mode == EPI_ACT_BWD && g.epi.aux_bf16 != nullptr && g.epi.d_dtype == TPS_BF16);
  if (pre16) return launch_pair_majors<T2_ACT16>(g, m, p, pairs, a_mn, b_mn, stream);
  if (g.epi.mode == EPI_ACT_FWD || g.epi.mode == EPI_ACT_BWD || g.epi.mode == EPI_GLU_UP)
    return launch_pair_majors<T2_ACT>(g, m, p, pairs, a_mn, b_mn, stream);
  return launch_pair_majors<T2_PLAIN>(g, m, p, pairs, a_mn, b_mn, stream);
}

static bool pair_operand_map(CUtensorMap* map, const void* base, bool mn, int64_t K, int64_t MN, int64_t ld,
                             int box_mn) {
  return mn ? tc_make_map(map, base, K, MN, ld, 64, TC_BK)       // stored K x MN
            : tc_make_map(map, base, MN, K, ld, TC_BK, box_mn);  // stored MN x K
}

int launch_gemm_tc2(const GemmDesc& g, uint32_t* dev_err, cudaStream_t stream) {
  const bool a_mn = (g.a_sk != 1);
  const bool b_mn = (g.b_sk != 1);
  const bool glu = g.epi.mode == EPI_GLU_FWD;
  const int64_t ks[3] = {g.K, g.K2, g.K3};
  const void* as[3] = {g.a, g.a2, g.a3};
  const void* bs[3] = {g.b, g.b2, g.b3};
  const int64_t a_sm[3] = {g.a_sm, g.a2_sm, g.a3_sm}, a_sk[3] = {g.a_sk, g.a2_sk, g.a3_sk};
  const int64_t b_sk[3] = {g.b_sk, g.b2_sk, g.b3_sk}, b_sn[3] = {g.b_sn, g.b2_sn, g.b3_sn};
  const bool k_segs = g.K2 > 0 || g.K3 > 0;
  const bool n_segs = g.n_segs > 1;
  if (g.n_segs < 1 || g.n_segs > 3) return TPS_ERR_ARG;
  if (glu && (k_segs || n_segs || g.b_up == nullptr)) return TPS_ERR_ARG;
  if ((n_segs || k_segs) && g.epi.mode != EPI_STORE) return TPS_ERR_ARG;  // segments: plain stores only
  if (n_segs && k_segs) return TPS_ERR_ARG;
  for (int s = 1; s < 3; ++s)
    if (ks[s] > 0 && ((a_sk[s] != 1) != a_mn || (b_sk[s] != 1) != b_mn)) return TPS_ERR_LAYOUT;
  T2Maps m;
  memset(&m, 0, sizeof(m));
  bool ok = true;
  for (int s = 0; s < 3; ++s) {
    if (s > 0 && ks[s] == 0) continue;
    ok = ok && pair_operand_map(&m.a[s], as[s], a_mn, ks[s], g.M, a_mn ? a_sk[s] : a_sm[s], T2_BM);
    if (!n_segs) ok = ok && pair_operand_map(&m.b[s], bs[s], b_mn, ks[s], g.N, b_mn ? b_sk[s] : b_sn[s], T2_BN_CTA);
  }
  if (glu) ok = ok && pair_operand_map(&m.b[1], g.b_up, b_mn, g.K, g.N, b_mn ? g.b_sk : g.b_sn, T2_BN_CTA);
  if (n_segs)
    for (int s = 0; s < g.n_segs; ++s)
      ok = ok && ((g.nb_sk[s] != 1) == b_mn) &&
           pair_operand_map(&m.b[s], g.nb[s], b_mn, g.K, g.n_cols[s], b_mn ? g.nb_sk[s] : g.nb_sn[s], T2_BN_CTA);
  if (!ok) return TPS_ERR_CUDA;

  T2Params p;
  p.M = static_cast<int>(g.M);
  p.N = static_cast<int>(g.N);
  p.K = static_cast<int>(g.K);
  p.glu = glu ? 1 : 0;
  p.m_tiles = static_cast<int>((g.M + 2 * T2_BM - 1) / (2 * T2_BM));
  p.n_tiles = static_cast<int>(glu ? (g.N + T2_BN_CTA - 1) / T2_BN_CTA : (g.N + T2_BN - 1) / T2_BN);
  int kt = 0;
  for (int s = 0; s < 3; ++s) {
    kt += static_cast<int>((ks[s] + TC_BK - 1) / TC_BK);
    p.k_end[s] = kt;
  }
  p.k_tiles = kt;
  p.n_segs = g.n_segs;
  int64_t nc = 0;
  for (int s = 0; s < 3; ++s) {
    if (s < g.n_segs && n_segs) {
      if (s + 1 < g.n_segs && g.n_cols[s] % T2_BN_CTA != 0) return TPS_ERR_ARG;
      nc += g.n_cols[s];
    } else {
      nc = g.N;
    }
    p.n_end[s] = static_cast<int>(nc);
  }
  if (n_segs && nc != g.N) return TPS_ERR_ARG;
  p.num_tiles = p.m_tiles * p.n_tiles;
  p.ksplit = 1;
  p.kflags = nullptr;
  p.unit_counter = g.unit_counter;
  // groups of pair tiles cover the same rows as twice as many single tiles
  tc_raster_choice(2 * p.m_tiles, &p.raster_n, &p.group, &p.pol_a, &p.pol_b);
  p.group = (p.group + 1) / 2;
  // A wider group pays while its A panels (group x 256 rows x K) stay in
  // L2 from one wave of tiles to the next: B then streams once per group,
  // and fewer groups mean fewer passes over B (the vocabulary head of the
  // logits GEMM: 6.6 GB read with 8 pair rows per group, 3.4 GB with 16).
  // Longer panels are evicted within a wave anyway, and there the wave's
  // count of distinct panels, about group + 76 / group, is smallest at 8.
  if (getenv("TPS_GEMM_GROUP") == nullptr) {
    const int64_t k_total = static_cast<int64_t>(g.K) + g.K2 + g.K3;
    if (16ll * 2 * T2_BM * k_total * 2 <= (40ll << 20)) p.group = 16;
  }
  if (p.group < 1) p.group = 1;
  if (p.group > p.m_tiles) p.group = p.m_tiles;
  p.epi = g.epi;
  p.err = dev_err;
  p.tma_store = tc_make_output_maps(g, &m.d[0], &m.d[1], &m.d[2]) ? 1 : 0;
  if (n_segs && !p.tma_store) return TPS_ERR_LAYOUT;  // column segments leave through TMA stores only
  // K split: plain fp32 stores through TMA, at least one K tile per run
  if (g.ksplit > 1 && g.kflags != nullptr && g.epi.mode == EPI_STORE && g.epi.d_dtype == TPS_F32 && p.tma_store &&
      !glu && !k_segs && !n_segs && p.k_tiles >= g.ksplit)
    p.ksplit = g.ksplit;
  p.kt_run = (p.k_tiles + p.ksplit - 1) / p.ksplit;
  p.ksplit = (p.k_tiles + p.kt_run - 1) / p.kt_run;  // every run holds at least one K tile
  p.num_units = p.num_tiles * p.ksplit;
  if (p.ksplit > 1) p.kflags = g.kflags;
  const int max_pairs = tc_num_sms() / 2;
  const int pairs = p.num_units < max_pairs ? p.num_units : max_pairs;

  return launch_pair_family(g, m, p, pairs, a_mn, b_mn, stream);
}

}  // namespace tps
