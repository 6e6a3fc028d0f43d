// gemm_wide.cu -- the CTA-pair tensor-core GEMM with 256 x 512 output tiles,
// for long contractions: the dHidden GEMM of the vocabulary-parallel
// cross-entropy ("多卡张量：拆开计算，再合回同一结果", 04 VOCABULARY SHARDS:
// dHidden = sum over shards of dlogits_r Whead_r^T), whose K is the whole
// vocabulary.
//
// Each pair tile is twice as wide as in gemm_tc2.cu: each CTA stages 128
// rows of A and two 128-column boxes of B per K step, and the even CTA
// issues two M=256, N=256 MMAs per 16-deep slice into the two halves of a
// single 512-column accumulator.  Per staged byte a CTA does a third more
// MMA work than with 256-wide tiles, and the output's tile count halves, so
// each block of A rows is staged half as often.  The price is the second
// accumulator: the next tile's MMAs wait until the epilogue has drained
// this one, which costs little when a tile runs thousands of K steps.
//
// Optionally (GemmDesc::ce_grad) A is not read as stored: the loads bring
// the logits GEMM's shifted bf16 logits, and the eight epilogue warps of
// each CTA, idle during the main loop, turn each staged A tile into the
// cross-entropy gradient e^{z - m}/s - 1[j = y] in shared memory before
// the MMAs read it; the passes over the output's first column block also
// write it to dlogits, so the gradient makes no separate trip through HBM.
// That form measured 2.2 times slower than the CE core plus this GEMM
// reading dlogits (the per-stage proxy fence and cluster release wait for
// the transforming warps' stores, a latency inside the stage ring that four
// stages cannot cover), and the library only runs it when asked
// (TPS_CE_GRAD_IN_GEMM=1).
//
// Synchronisation (barriers at the same offsets in both CTAs):
//   full[s]      even CTA: expects both CTAs' bytes (only B's when A is
//                transformed, plus one arrival per transforming warp of
//                both CTAs); both CTAs' loads complete on it
//   a_full[s]    each CTA, transformed A only: its own A load
//   empty[s]     each CTA: the MMA commit, multicast to the pair
//   tmem_full    each CTA: the MMA commit after a tile's last K step
//   tmem_empty   even CTA: one arrival per epilogue warp of each CTA
//
// Warp roles (320 threads, one CTA per SM): warp 0 TMA producer, warp 1
// TMEM allocator and (even CTA) MMA issuer, warps 2..9 A transform and
// epilogue (warp w drains TMEM lanes 32*(w%4)..+31 and accumulator columns
// 256*((w-2)/4)..+255).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "tc_common.cuh"

namespace tps {

constexpr int W_BM = 128;                             // rows per CTA (256 per pair)
constexpr int W_BN = 512;                             // columns per pair tile
constexpr int W_BN_BOX = 128;                         // columns per B box; each CTA stages two
constexpr int W_STAGES = 4;
constexpr int W_A_BYTES = W_BM * TC_BK * 2;           // 16 KB
constexpr int W_B_BOX_BYTES = W_BN_BOX * TC_BK * 2;   // 16 KB
constexpr int W_B_BYTES = 2 * W_B_BOX_BYTES;          // 32 KB
constexpr int W_STAGE_BYTES = W_A_BYTES + W_B_BYTES;  // 48 KB
constexpr int W_THREADS = 320;
constexpr int W_EPI_WARPS = 8;
constexpr uint32_t W_TMEM_COLS = 512;                 // one fp32 accumulator, 256 columns per MMA
constexpr int W_STG = TC_STG_F32_BYTES;               // one 4 KB box per epilogue warp
// Readers of each unit the dynamic schedule publishes (PairUnits): the even
// CTA's MMA thread, both CTAs' epilogue warps and the odd CTA's producer.
constexpr int W_SCHED_READERS = 2 + 2 * W_EPI_WARPS;

struct WBarriers {
  uint64_t full[W_STAGES];
  uint64_t a_full[W_STAGES];
  uint64_t empty[W_STAGES];
  uint64_t tmem_full;
  uint64_t tmem_empty;
  uint64_t drain;
  uint64_t sched_full[kUnitRing];   // PairUnits ring
  uint64_t sched_empty[kUnitRing];
  int32_t sched_unit[kUnitRing];
  uint32_t tmem_slot;
  uint32_t abort;
};
constexpr size_t W_SMEM = 1024 + W_STAGES * W_STAGE_BYTES + W_EPI_WARPS * W_STG + sizeof(WBarriers);
static_assert(W_SMEM <= 232448, "exceeds the opt-in shared memory per block");

struct WMaps {
  CUtensorMap a, b, d;
};

struct WParams {
  int M, N, K;
  int m_tiles, n_tiles, k_tiles, num_tiles;
  // K split as in gemm_tc2.cu: unit u is tile u % num_tiles, run u / num_tiles
  int ksplit, kt_run, num_units;
  uint32_t* kflags;
  uint32_t* unit_counter;  // dynamic schedule (GemmDesc::unit_counter), else nullptr
  int group;
  Epilogue epi;
  CeGradOperand xf;
  uint32_t* err;
};

// The two bf16 values of a 32-bit word, low half first, as floats.
__device__ __forceinline__ float w_bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float w_bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t w_pack_bf16(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

// Debug builds: a dlogits store of n columns at (row, col) must lie inside
// the M x K gradient.
__device__ __forceinline__ bool w_dbg_ok(const WParams& p, int64_t row, int64_t col, int n) {
#if TPS_DEBUG
  if (row < 0 || row >= p.M || col < 0 || col + n > p.K) {
    atomicOr(p.err, TPS_DEVERR_BOUNDS);
    return false;
  }
#endif
  (void)p; (void)row; (void)col; (void)n;
  return true;
}

template <bool B_MN, bool XF>
__global__ void __launch_bounds__(W_THREADS, 1) gemm_wide_kernel(const __grid_constant__ WMaps m, const WParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* staging = smem + W_STAGES * W_STAGE_BYTES;  // 1024-aligned
  WBarriers* bars = reinterpret_cast<WBarriers*>(staging + W_EPI_WARPS * W_STG);
  volatile uint32_t* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < W_STAGES; ++s) {
      mbar_init(&bars->full[s], XF ? 1 + 2 * W_EPI_WARPS : 1);
      mbar_init(&bars->a_full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->tmem_full, 1);
    mbar_init(&bars->tmem_empty, 2 * W_EPI_WARPS);
    mbar_init(&bars->drain, 1);
    for (int s = 0; s < kUnitRing; ++s) {
      mbar_init(&bars->sched_full[s], 1);
      mbar_init(&bars->sched_empty[s], W_SCHED_READERS);
    }
    bars->abort = 0u;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&m.a);
    tma_prefetch_desc(&m.b);
  }
  if (warp == 1) {
    tmem_alloc_pair(&bars->tmem_slot, W_TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_slot;
  const uint32_t full0_leader = cluster_map(smem_u32(&bars->full[0]), 0);
  const uint32_t tmem_empty_leader = cluster_map(smem_u32(&bars->tmem_empty), 0);
  PairUnits units;
  units.init(bars->sched_full, bars->sched_empty, bars->sched_unit, abort_flag, p.err, p.unit_counter, pair, npairs,
             p.num_units, warp == 0 && rank == 0);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int u = units.take(); ok && u >= 0; u = units.take()) {
        const int tile = u % p.num_tiles, run = u / p.num_tiles;
        const int kt_begin = run * p.kt_run, kt_end = min(p.k_tiles, kt_begin + p.kt_run);
        int mt, nt;
        tc_raster(0, p.group, p.m_tiles, p.n_tiles, tile, mt, nt);
        const int m0 = mt * 2 * W_BM + static_cast<int>(rank) * W_BM;
        // this CTA's B columns: one 128-column box in each 256-column half
        const int nb0 = nt * W_BN + static_cast<int>(rank) * W_BN_BOX;
        for (int kt = kt_begin; kt < kt_end; ++kt) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * W_STAGE_BYTES;
          uint8_t* sb = sa + W_A_BYTES;
          const uint32_t fb = full0_leader + stage * static_cast<uint32_t>(sizeof(uint64_t));
          const int k0 = kt * TC_BK;
          if constexpr (XF) {  // A lands on this CTA's own barrier, for its transforming warps
            mbar_expect_tx(&bars->a_full[stage], W_A_BYTES);
            tma_load_2d(sa, &m.a, &bars->a_full[stage], k0, m0);
            if (rank == 0) mbar_expect_tx(&bars->full[stage], 2 * W_B_BYTES);
          } else {
            if (rank == 0) mbar_expect_tx(&bars->full[stage], 2 * W_STAGE_BYTES);
            tma_load_2d_pair(sa, &m.a, fb, k0, m0);
          }
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            uint8_t* dst = sb + hb * W_B_BOX_BYTES;
            const int n0 = nb0 + hb * (W_BN / 2);
            if (!B_MN) {
              tma_load_2d_pair(dst, &m.b, fb, k0, n0);
            } else {
#pragma unroll
              for (int j = 0; j < W_BN_BOX / 64; ++j) tma_load_2d_pair(dst + j * TC_MN_BOX_BYTES, &m.b, fb, n0 + 64 * j, k0);
            }
          }
          ++issued;
          if (++stage == W_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain the loads still in flight before the CTA exits.
      const int64_t first = issued > W_STAGES ? issued - W_STAGES : 0;
      for (int64_t i = first; i < issued; ++i) {
        const uint32_t par = static_cast<uint32_t>((i / W_STAGES) & 1);
        if (XF) mbar_wait_drain(&bars->a_full[i % W_STAGES], par, p.err);
        if (rank == 0) mbar_wait_drain(&bars->full[i % W_STAGES], par, p.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(2 * W_BM, W_BN / 2, false, B_MN);
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = units.take(); ok && u >= 0; u = units.take()) {
        const int run = u / p.num_tiles;
        const int kt_begin = run * p.kt_run, kt_end = min(p.k_tiles, kt_begin + p.kt_run);
        if (!mbar_wait(&bars->tmem_empty, acc_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        for (int kt = kt_begin; kt < kt_end; ++kt) {
          // the transformed A tiles were written by threads of both CTAs
          const bool got = XF ? mbar_wait_cluster(&bars->full[stage], phase, abort_flag, p.err)
                              : mbar_wait(&bars->full[stage], phase, abort_flag, p.err);
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * W_STAGE_BYTES);
          const uint32_t sb = sa + W_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint32_t accum = (kt != kt_begin || kk != 0) ? 1u : 0u;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              const uint32_t b0 = sb + hb * W_B_BOX_BYTES;
              const uint64_t bd = B_MN ? smem_desc_sw128(b0 + kk * 2048, TC_MN_BOX_BYTES, 1024)
                                       : smem_desc_sw128(b0 + kk * 32, 16, 1024);
              tc_mma_f16_pair(tmem_base + hb * (W_BN / 2), ad, bd, idesc, accum);
            }
          }
          tc_commit_pair_mc(&bars->empty[stage], 0x3);  // frees the stage in both CTAs
          if (++stage == W_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(&bars->tmem_full, 0x3);  // both CTAs' accumulators complete
        acc_phase ^= 1u;
      }
      tc_commit_pair(&bars->drain);
      mbar_wait_drain(&bars->drain, 0, p.err);
    }
  } else {
    // -------------------------------------------- A transform and epilogue
    const int ew = warp - 2;  // 0..7
    const int q = warp & 3;   // TMEM lane quadrant
    const int h = ew >> 2;    // 256-column half of the tile
    uint8_t* stg = staging + ew * W_STG;
    const Epilogue& e = p.epi;
    // Transform: this thread's rows of the CTA's 128-row A tile and the
    // 16-byte chunk it owns in each (8 lanes cover one 128-byte row).
    const int pch = lane & 7;
    int rr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) rr[i] = ew * 16 + (lane >> 3) + 4 * i;
    uint32_t stage = 0, phase = 0, acc_phase = 0;
    bool ok = true;
    for (int u = units.take_warp(lane); ok && u >= 0; u = units.take_warp(lane)) {
      const int tile = u % p.num_tiles, run = u / p.num_tiles;
      const int kt_begin = run * p.kt_run, kt_end = min(p.k_tiles, kt_begin + p.kt_run);
      int mt, nt;
      tc_raster(0, p.group, p.m_tiles, p.n_tiles, tile, mt, nt);
      const int m0 = mt * 2 * W_BM + static_cast<int>(rank) * W_BM;
      if constexpr (XF) {
        const CeGradOperand& x = p.xf;
        float ml[4], inv[4], c_cur[4], c_nxt[4];
        int64_t y[4], row[4];
        bool live[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          row[i] = m0 + rr[i];
          live[i] = row[i] < p.M;
          ml[i] = 0.0f;
          inv[i] = 0.0f;  // rows past M: the gradient is 0
          y[i] = -1;
          c_cur[i] = 0.0f;
          c_nxt[i] = 0.0f;
          if (live[i]) {
            const float2 mi = reinterpret_cast<const float2*>(x.ms)[row[i]];
            ml[i] = mi.x * kTcLog2e;
            inv[i] = mi.y;
            y[i] = x.label_i64 ? static_cast<const int64_t*>(x.labels)[row[i]]
                               : static_cast<int64_t>(static_cast<const int32_t*>(x.labels)[row[i]]);
            c_cur[i] = x.shift[row[i] * x.shift_ld + (kt_begin >> 1)];
          }
        }
        const bool store_g = nt == 0;  // one pass over each A tile writes dlogits
        for (int kt = kt_begin; kt < kt_end; ++kt) {
          // the next statistics tile's shifts, read while this K tile is formed
          const bool next_shift = kt + 1 < kt_end && ((kt + 1) & 1) == 0;
          if (next_shift) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (live[i]) c_nxt[i] = x.shift[row[i] * x.shift_ld + ((kt + 1) >> 1)];
          }
          if (!mbar_wait(&bars->a_full[stage], phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * W_STAGE_BYTES;
          const int k0 = kt * TC_BK;
          const bool tail = k0 + TC_BK > p.K;  // warp-uniform
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = rr[i];
            uint4* slot = reinterpret_cast<uint4*>(sa + r * 128 + pch * 16);
            const int64_t col = k0 + 8 * (pch ^ (r & 7));  // the chunk's first column (128-byte swizzle)
            const uint4 zw = *slot;
            const uint32_t wd[4] = {zw.x, zw.y, zw.z, zw.w};
            // (c - m) log2(e): e^{z - m} = 2^{(z - c) log2(e) + (c - m) log2(e)}
            const float adj = fmaf(c_cur[i], kTcLog2e, -ml[i]);
            float g[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              g[2 * j] = ex2_approx(fmaf(w_bf16_lo(wd[j]), kTcLog2e, adj)) * inv[i];
              g[2 * j + 1] = ex2_approx(fmaf(w_bf16_hi(wd[j]), kTcLog2e, adj)) * inv[i];
            }
            if (y[i] >= col && y[i] < col + 8) {
#pragma unroll
              for (int j = 0; j < 8; ++j) g[j] -= (y[i] == col + j) ? 1.0f : 0.0f;
            }
            if (tail) {  // columns past K: the loads filled zeros, the gradient is 0 there
#pragma unroll
              for (int j = 0; j < 8; ++j) g[j] = (col + j < p.K) ? g[j] : 0.0f;
            }
            const uint4 ow = make_uint4(w_pack_bf16(g[0], g[1]), w_pack_bf16(g[2], g[3]), w_pack_bf16(g[4], g[5]),
                                        w_pack_bf16(g[6], g[7]));
            *slot = ow;
            if (store_g && live[i] && col < p.K) {
              __nv_bfloat16* grow = static_cast<__nv_bfloat16*>(x.dlogits) + row[i] * x.ldg;
              if (col + 8 <= p.K) {
                if (w_dbg_ok(p, row[i], col, 8)) __stcs(reinterpret_cast<uint4*>(grow + col), ow);
              } else {
                const uint32_t ows[4] = {ow.x, ow.y, ow.z, ow.w};
                unsigned short* gb = reinterpret_cast<unsigned short*>(grow);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  if (col + j < p.K && w_dbg_ok(p, row[i], col + j, 1))
                    gb[col + j] = static_cast<unsigned short>((j & 1) ? (ows[j >> 1] >> 16) : (ows[j >> 1] & 0xffffu));
              }
            }
          }
          fence_async_smem();  // the MMA reads these tiles through the async proxy
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(full0_leader + stage * static_cast<uint32_t>(sizeof(uint64_t)));
          if (next_shift) {
#pragma unroll
            for (int i = 0; i < 4; ++i) c_cur[i] = c_nxt[i];
          }
          if (++stage == W_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      // ---- epilogue
      if (p.ksplit > 1 && run > 0) {
        // K split: the previous run of this tile (all 2 x 8 epilogue warps
        // of its pair) must be in memory before this run adds to it.
        uint32_t ready = 1u;
        if (lane == 0) {
          const uint32_t need = static_cast<uint32_t>(2 * W_EPI_WARPS * run);
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
      if (!mbar_wait(&bars->tmem_full, acc_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const int row0 = m0 + q * 32;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(h * (W_BN / 2));
      const float none[32] = {};
      for (int c = 0; c < W_BN / 2 / 32; ++c) {
        const int col0 = nt * W_BN + h * (W_BN / 2) + c * 32;
        if (col0 >= p.N) break;  // warp-uniform
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        tmem_ld_wait();
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        if (run > 0)  // K split: add this run's partial tile to the output
          tc_store_chunk<0, true, true>(e, &m.d, &m.d, stg, stg, lane, row0, col0, v, none);
        else
          tc_store_chunk<0, true>(e, &m.d, &m.d, stg, stg, lane, row0, col0, v, none);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tmem_empty_leader);
      acc_phase ^= 1u;
      if (p.ksplit > 1) {  // K split: this warp's part of the run is in memory
        if (lane == 0) {
          bulk_wait0();
          fence_async_global();
          red_release_gpu_add(p.kflags + tile, 1u);
        }
        __syncwarp();
      }
    }
    if (lane == 0) bulk_wait0();
  }

  tc_fence_before();
  cluster_sync();  // the pair's MMAs, loads and epilogues are all finished
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, W_TMEM_COLS);
}

// ------------------------------------------------------------------ host

bool gemm_wide_supported(const GemmDesc& g) {
  if (!gemm_tc_supported(g)) return false;
  if (g.epi.mode != EPI_STORE || g.epi.d_dtype != TPS_F32) return false;
  if (g.a_sk != 1 || g.n_segs > 1 || g.K2 > 0 || g.K3 > 0) return false;
  if (g.epi.d == nullptr || (reinterpret_cast<uintptr_t>(g.epi.d) & 15u) != 0 || (g.epi.ldd * 4) % 16 != 0 ||
      g.epi.ldd < g.N)
    return false;
  const CeGradOperand& x = g.ce_grad;
  if (x.ms != nullptr) {
    if (x.shift == nullptr || x.labels == nullptr || x.dlogits == nullptr || x.shift_ld < (g.K + 127) / 128) return false;
    if ((reinterpret_cast<uintptr_t>(x.dlogits) & 15u) != 0 || x.ldg % 8 != 0 || x.ldg < g.K) return false;
  }
  return true;
}

template <bool B_MN, bool XF>
static int launch_wide_typed(const WMaps& m, const WParams& p, int pairs, double flops, const char* name,
                             cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.blockDim = dim3(W_THREADS, 1, 1);
  cfg.dynamicSmemBytes = W_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  std::call_once(once, [&cfg] {
    attr_err = cudaFuncSetAttribute(gemm_wide_kernel<B_MN, XF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(W_SMEM));
    if (attr_err == cudaSuccess &&
        cudaOccupancyMaxActiveClusters(&max_clusters, gemm_wide_kernel<B_MN, XF>, &cfg) != cudaSuccess)
      max_clusters = 0;
  });
  if (attr_err != cudaSuccess) return TPS_ERR_CUDA;
  // Under a K split an epilogue waits for a run that another pair holds:
  // launch only as many pairs as can be resident at once.
  if (p.ksplit > 1) {
    if (max_clusters < 1) return TPS_ERR_CUDA;
    if (pairs > max_clusters) cfg.gridDim = dim3(static_cast<unsigned>(2 * max_clusters), 1, 1);
  }
  ProfScope prof("gemm_tc", name, flops, 0.0, stream);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_wide_kernel<B_MN, XF>, m, p);
  note_launch();
  return e == cudaSuccess ? TPS_OK : TPS_ERR_CUDA;
}

int launch_gemm_wide(const GemmDesc& g, uint32_t* dev_err, cudaStream_t stream) {
  if (!gemm_wide_supported(g)) return TPS_ERR_ARG;
  const bool b_mn = g.b_sk != 1;
  const bool xf = g.ce_grad.ms != nullptr;
  WMaps m;
  memset(&m, 0, sizeof(m));
  bool ok = tc_make_map(&m.a, g.a, g.M, g.K, g.a_sm, TC_BK, W_BM);                     // stored M x K
  ok = ok && (b_mn ? tc_make_map(&m.b, g.b, g.K, g.N, g.b_sk, 64, TC_BK)               // stored K x N
                   : tc_make_map(&m.b, g.b, g.N, g.K, g.b_sn, TC_BK, W_BN_BOX));       // stored N x K
  ok = ok && tc_make_out_map(&m.d, g.epi.d, g.M, g.N, g.epi.ldd, TPS_F32);
  if (!ok) return TPS_ERR_CUDA;

  WParams p;
  p.M = static_cast<int>(g.M);
  p.N = static_cast<int>(g.N);
  p.K = static_cast<int>(g.K);
  p.m_tiles = static_cast<int>((g.M + 2 * W_BM - 1) / (2 * W_BM));
  p.n_tiles = static_cast<int>((g.N + W_BN - 1) / W_BN);
  p.k_tiles = static_cast<int>((g.K + TC_BK - 1) / TC_BK);
  p.num_tiles = p.m_tiles * p.n_tiles;
  // Groups of eight pair rows (TPS_GEMM_GROUP counts 128-row tiles, as on
  // the other kernels).  On the dHidden GEMM at T = 8192 with the units
  // taken in order: 1, 2, 4, 8, 16 pair rows took 4.37-4.41, 4.30-4.32,
  // 4.26-4.28, 4.24-4.25, 4.29-4.33 ms (with the static round-robin four
  // had been 1-2 % faster than eight).
  int raster_n = 0, group = 0, pa = 0, pb = 0;
  tc_raster_choice(2 * p.m_tiles, &raster_n, &group, &pa, &pb);
  p.group = getenv("TPS_GEMM_GROUP") != nullptr ? (group + 1) / 2 : 8;
  if (p.group < 1) p.group = 1;
  if (p.group > p.m_tiles) p.group = p.m_tiles;
  p.ksplit = 1;
  p.kflags = nullptr;
  if (g.ksplit > 1 && g.kflags != nullptr && p.k_tiles >= g.ksplit) p.ksplit = g.ksplit;
  p.unit_counter = g.unit_counter;
  p.kt_run = (p.k_tiles + p.ksplit - 1) / p.ksplit;
  if (xf && (p.kt_run & 1) && p.ksplit > 1) ++p.kt_run;  // runs start on a statistics tile (two K tiles)
  p.ksplit = (p.k_tiles + p.kt_run - 1) / p.kt_run;     // every run holds at least one K tile
  p.num_units = p.num_tiles * p.ksplit;
  if (p.ksplit > 1) p.kflags = g.kflags;
  p.epi = g.epi;
  p.xf = g.ce_grad;
  p.err = dev_err;
  const int max_pairs = tc_num_sms() / 2;
  const int pairs = p.num_units < max_pairs ? p.num_units : max_pairs;
  const double flops = 2.0 * double(g.M) * double(g.N) * double(g.K);
  if (!b_mn)
    return xf ? launch_wide_typed<false, true>(m, p, pairs, flops, g.name, stream)
              : launch_wide_typed<false, false>(m, p, pairs, flops, g.name, stream);
  return xf ? launch_wide_typed<true, true>(m, p, pairs, flops, g.name, stream)
            : launch_wide_typed<true, false>(m, p, pairs, flops, g.name, stream);
}

}  // namespace tps
