// tc_common.cuh -- pieces shared by the two tensor-core GEMM kernels
// (gemm_tc.cu: one CTA per 128 x 256 tile; gemm_tc2.cu: a CTA pair per
// 256 x 256 tile): output staging for TMA stores, the fused epilogue of one
// 32-column chunk, the vocabulary-CE tile statistics, the tile raster and
// the host-side tensor-map helpers.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include "epilogue.cuh"
#include "internal.cuh"
#include "ptx.cuh"

namespace tps {

constexpr int TC_BK = 64;  // one 128-byte swizzle row of bf16
// A box of an MN-major operand: 64 MN elements (128 B) x 64 K rows.
constexpr int TC_MN_BOX_BYTES = 64 * TC_BK * 2;  // 8 KB
// Epilogue staging per warp and buffer: a 32 x 32 fp32 box (128-byte
// swizzle) and a 32 x 32 bf16 box (64-byte swizzle).
constexpr int TC_STG_F32_BYTES = 32 * 32 * 4;
constexpr int TC_STG_BF16_BYTES = 32 * 32 * 2;
constexpr float kTcLog2e = 1.4426950408889634f;

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

// Fused epilogue of one 32 x 32 chunk (lane = row) through TMA stores.  The
// TMA unit clips every box to its tensor map, whose extent is the output's
// (M, N): a box of a ragged tile that starts past the output writes
// nothing, so these stores need no bounds check in debug builds.
// `v` holds the accumulators, `a` the pre-activation for EPI_ACT_BWD (Hg
// for EPI_GLU_UP).  EPI_ACT_FWD stages its pre-activation in `stg_f32` (a
// 32 x 32 bf16 box there when d_dtype is bf16) and the activation in
// `stg_bf16`.  PENDING is the number of this warp's earlier
// bulk-store groups that may still be reading staging when the buffers are
// overwritten (0 for one staging buffer, 1 when the caller alternates two).
// STORE_ONLY: the caller guarantees EPI_STORE.  REDUCE (EPI_STORE, fp32):
// add the box into the output with a TMA reduction instead of storing it.
template <int PENDING, bool STORE_ONLY = false, bool REDUCE = false>
__device__ __forceinline__ void tc_store_chunk(const Epilogue& e, const CUtensorMap* tmD, const CUtensorMap* tmD2,
                                               uint8_t* stg_f32, uint8_t* stg_bf16, int lane, int row0, int col0,
                                               float (&v)[32], const float (&a)[32]) {
  if (lane == 0) {
    if constexpr (PENDING == 0)
      bulk_wait_read0();
    else
      asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
  }
  __syncwarp();
  if (STORE_ONLY || e.mode == EPI_STORE || e.mode == EPI_CE_STATS) {
    if (e.d_dtype == TPS_F32)
      stage_f32_sw128(stg_f32, lane, v);
    else
      stage_bf16_sw64(stg_bf16, lane, v);
  } else if (e.mode == EPI_ACT_FWD) {
    if (e.d != nullptr) {  // the pre-activation, fp32 or bf16, from the first slot
      if (e.d_dtype == TPS_F32)
        stage_f32_sw128(stg_f32, lane, v);
      else
        stage_bf16_sw64(stg_f32, lane, v);
    }
    act_dispatch(e.act, [&](auto A) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = act_fwd_c<decltype(A)::value>(v[i]);
    });
    stage_bf16_sw64(stg_bf16, lane, v);
  } else if (e.mode == EPI_GLU_UP) {
    if (e.d != nullptr) stage_f32_sw128(stg_f32, lane, v);
    act_dispatch(e.act, [&](auto A) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= act_fwd_c<decltype(A)::value>(a[i]);
    });
    stage_bf16_sw64(stg_bf16, lane, v);
  } else {
    act_dispatch(e.act, [&](auto A) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= act_grad_c<decltype(A)::value>(a[i]);
    });
    if (e.d_dtype == TPS_F32)
      stage_f32_sw128(stg_f32, lane, v);
    else
      stage_bf16_sw64(stg_bf16, lane, v);
  }
  fence_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (!STORE_ONLY && (e.mode == EPI_ACT_FWD || e.mode == EPI_GLU_UP)) {
      if (e.d != nullptr) tma_store_2d(tmD, stg_f32, col0, row0);
      tma_store_2d(tmD2, stg_bf16, col0, row0);
    } else if (REDUCE) {
      tma_reduce_add_2d(tmD, stg_f32, col0, row0);
    } else {
      tma_store_2d(tmD, e.d_dtype == TPS_F32 ? stg_f32 : stg_bf16, col0, row0);
    }
    bulk_commit();
  }
}

// EPI_GLU_BWD chunk through TMA stores, double-buffered like
// tc_store_chunk<1>: dHg = v * U * phi'(Hg) leaves from the bf16 slot and
// dU = v * phi(Hg) from the start of the fp32 slot, both as bf16 boxes.
// `u` is overwritten with dU.
__device__ __forceinline__ void tc_store_glu_bwd_chunk(const Epilogue& e, const CUtensorMap* tmD,
                                                       const CUtensorMap* tmD2, uint8_t* stg_f32, uint8_t* stg_bf16,
                                                       int lane, int row0, int col0, float (&v)[32],
                                                       const float (&hg)[32], float (&u)[32]) {
  if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
  __syncwarp();
  act_dispatch(e.act, [&](auto A) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      float f, g;
      act_fwd_grad_c<decltype(A)::value>(hg[i], f, g);
      const float da = v[i];
      v[i] = da * u[i] * g;
      u[i] = da * f;
    }
  });
  stage_bf16_sw64(stg_bf16, lane, v);
  stage_bf16_sw64(stg_f32, lane, u);
  fence_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmD, stg_bf16, col0, row0);
    tma_store_2d(tmD2, stg_f32, col0, row0);
    bulk_commit();
  }
}

// EPI_GLU_FWD chunk through TMA stores from a 6 KB staging buffer: Hg and
// then U (fp32) pass through the same 4 KB box at +0 -- U is staged once
// the Hg store has read the box -- and A = phi(Hg) * U (bf16) through the
// 2 KB box at +4 KB.  The buffer is reused only after this warp's earlier
// stores have read it.
__device__ __forceinline__ void tc_store_glu_chunk(const Epilogue& e, const CUtensorMap* tmHg, const CUtensorMap* tmA,
                                                   const CUtensorMap* tmU, uint8_t* stg, int lane, int row0,
                                                   int col0, const float (&hg)[32], float (&u)[32]) {
  if (lane == 0) bulk_wait_read0();
  __syncwarp();
  stage_f32_sw128(stg, lane, hg);
  fence_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmHg, stg, col0, row0);
    bulk_commit();
  }
  float a[32];
  act_dispatch(e.act, [&](auto A) {
#pragma unroll
    for (int i = 0; i < 32; ++i) a[i] = u[i] * act_fwd_c<decltype(A)::value>(hg[i]);
  });
  stage_bf16_sw64(stg + TC_STG_F32_BYTES, lane, a);
  if (lane == 0) bulk_wait_read0();  // the Hg store has read the fp32 box
  __syncwarp();
  stage_f32_sw128(stg, lane, u);
  fence_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmU, stg, col0, row0);
    tma_store_2d(tmA, stg + TC_STG_F32_BYTES, col0, row0);
    bulk_commit();
  }
}

// ---- vocabulary-CE statistics in the logits epilogue ----------------------
// Each epilogue thread owns one output row, so the statistics of a
// kStatsTileN-column tile need no cross-thread reduction.  The tile is read
// from tensor memory twice: the first pass finds the max of the part of the
// tile in shard a (the shard of the tile's first column) and of the part in
// shard b (the next one); the second sums e^{z - max} for each part, takes
// the logit at the row's label, and stores the tile relative to its max
// (the larger of the two).  bf16 rounds z - max to within 2^-8 of its
// magnitude, so a softmax weight p = e^{z - m} / s is off by at most
// p (max - z) 2^-8 <= 2^-8 / e in absolute terms, and the weights near the
// max, which dominate, are nearly exact.

// Max of elements [i0, i1) of v (-inf for an empty range).
__device__ __forceinline__ float ce_chunk_max(const float (&v)[32], int i0, int i1) {
  float cm = -INFINITY;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i >= i0 && i < i1) cm = fmaxf(cm, v[i]);
  return cm;
}
// Sum of e^{v - m} over elements [i0, i1) of v (m finite when the range is not empty).
__device__ __forceinline__ float ce_chunk_sum(const float (&v)[32], int i0, int i1, float m) {
  const float ml = m * kTcLog2e;
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i >= i0 && i < i1) acc += ex2_approx(fmaf(v[i], kTcLog2e, -ml));
  return acc;
}

// Max of all 32 elements, and sum of e^{v - m} over all 32, for the chunks
// that lie entirely in one shard's real columns (all but a few per row): no
// per-element range tests, and a tree / four partial sums instead of one
// serial chain.
__device__ __forceinline__ float ce_max32(const float (&v)[32]) {
  float m[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) m[i] = fmaxf(v[i], v[i + 16]);
#pragma unroll
  for (int w = 8; w > 0; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
  return m[0];
}
__device__ __forceinline__ float ce_sum32(const float (&v)[32], float m) {
  const float ml = m * kTcLog2e;
  float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i & 3] += ex2_approx(fmaf(v[i], kTcLog2e, -ml));
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// The shard owning column c under the array_split of n into p parts.
__device__ __forceinline__ int64_t shard_of(int64_t c, int64_t n, int64_t p) {
  const int64_t q = n / p, r = n % p, big = r * (q + 1);
  return c < big ? c / (q + 1) : r + (c - big) / q;
}

struct CeTileAcc {
  int64_t split;  // first column of shard b
  int64_t b;      // shard b: the one after the shard of the tile's first column
  bool has_b;     // shard b starts inside the tile
  float ma, sa, mb, sb;
  __device__ __forceinline__ void reset(const Epilogue& e, int64_t N, int64_t tile_col0) {
    b = shard_of(tile_col0, N, e.ce_parts) + 1;
    split = shard_offset(N, e.ce_parts, b);
    has_b = b < e.ce_parts && split > tile_col0 && split < tile_col0 + kStatsTileN;
    ma = -INFINITY;
    sa = 0.0f;
    mb = -INFINITY;
    sb = 0.0f;
  }
  // Of the chunk [col0, col0 + n): the real columns (those below vreal;
  // the rest are vocabulary padding) end at chunk index nn, shard a's at na.
  __device__ __forceinline__ void parts(int64_t col0, int n, int64_t vreal, int& na, int& nn) const {
    nn = (vreal - col0 < n) ? static_cast<int>(vreal - col0 < 0 ? 0 : vreal - col0) : n;
    na = static_cast<int>(split - col0 < 0 ? 0 : (split - col0 > nn ? nn : split - col0));
  }
  __device__ __forceinline__ void fold_max(const float (&v)[32], int64_t col0, int n, int64_t vreal) {
    int na, nn;
    parts(col0, n, vreal, na, nn);
    if (na == 32) {  // the whole chunk is real and in shard a
      ma = fmaxf(ma, ce_max32(v));
      return;
    }
    ma = fmaxf(ma, ce_chunk_max(v, 0, na));
    mb = fmaxf(mb, ce_chunk_max(v, na, nn));
  }
  __device__ __forceinline__ void fold_sum(const float (&v)[32], int64_t col0, int n, int64_t vreal) {
    int na, nn;
    parts(col0, n, vreal, na, nn);
    if (na == 32) {
      sa += ce_sum32(v, ma);
      return;
    }
    if (na > 0) sa += ce_chunk_sum(v, 0, na, ma);
    if (nn > na) sb += ce_chunk_sum(v, na, nn, mb);
  }
  __device__ __forceinline__ float shift() const {
    const float m = fmaxf(ma, mb);
    return m == -INFINITY ? 0.0f : m;
  }
  __device__ __forceinline__ void flush(const Epilogue& e, int64_t row, int64_t stat_tile) const {
    if (!dbg_store_ok(e, row, stat_tile * kStatsTileN, 1)) return;
    reinterpret_cast<float2*>(e.stats)[row * e.n_tiles + stat_tile] = make_float2(ma, sa);
    if (has_b) reinterpret_cast<float2*>(e.stats_b)[row * e.ce_parts + b] = make_float2(mb, sb);
    e.ce_shift[row * e.ce_shift_ld + stat_tile] = shift();
  }
};

// The label of row `row` (int32 or int64 labels).
__device__ __forceinline__ int64_t ce_row_label(const Epilogue& e, int64_t row) {
  return e.ce_label_i64 ? static_cast<const int64_t*>(e.ce_labels)[row]
                        : static_cast<int64_t>(static_cast<const int32_t*>(e.ce_labels)[row]);
}

// EPI_CE_STATS over the statistics tile that starts at column tc0 (TMEM
// address t_col), for the row this thread owns (row_ok: row < M; label y).
// Each 32-column chunk leaves through store(col0, n, v) with v relative to
// the tile's shift; zy receives the label's logit when the label lies in
// the tile (have = true).
template <class Store>
__device__ __forceinline__ void ce_stats_tile(const Epilogue& e, uint32_t t_col, int64_t tc0, int64_t N, bool row_ok,
                                              int64_t row, int64_t y, float& zy, bool& have, Store&& store) {
  constexpr int kChunks = kStatsTileN / 32;
  const int chunks = static_cast<int>((N - tc0) / 32 < kChunks ? (N - tc0 + 31) / 32 : kChunks);
  CeTileAcc st;
  st.reset(e, N, tc0);
  for (int c = 0; c < chunks; ++c) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_col + c * 32, r);
    tmem_ld_wait();
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
    const int64_t col0 = tc0 + 32 * c;
    st.fold_max(v, col0, static_cast<int>(N - col0 < 32 ? N - col0 : 32), e.ce_vreal);
  }
  const float sh = st.shift();
  for (int c = 0; c < chunks; ++c) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_col + c * 32, r);
    tmem_ld_wait();
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
    const int64_t col0 = tc0 + 32 * c;
    const int n = static_cast<int>(N - col0 < 32 ? N - col0 : 32);
    st.fold_sum(v, col0, n, e.ce_vreal);
    const int64_t dy = y - col0;
    if (dy >= 0 && dy < n) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i == dy) zy = v[i];
      have = true;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] -= sh;
    store(col0, n, v);
  }
  if (row_ok) st.flush(e, row, tc0 / kStatsTileN);
}

// ---- work units of a CTA pair ---------------------------------------------
// The units one role of a CTA pair processes, in order.  Static: pair p
// takes units p, p + pairs, p + 2 pairs, ...  Dynamic (a zeroed global
// counter given): the even CTA's producer takes each next unit from the
// counter when it starts on it and publishes it through a ring of
// kUnitRing slots in both CTAs' shared memory, where the other roles read
// it; a unit past the end tells them to stop.  Units are taken in
// increasing order and every pair works through its own in order, so a
// K-split run only ever waits for a unit that a running pair took earlier.
// Each slot's `empty` barrier (even CTA) counts `readers` arrivals.
constexpr int kUnitRing = 4;
struct PairUnits {
  uint64_t* full;   // [kUnitRing], this CTA: the slot's unit has been written
  uint64_t* empty;  // [kUnitRing], this CTA (used in the even CTA)
  int32_t* unit;    // [kUnitRing], this CTA's copy
  uint32_t empty0_leader, full0_peer, unit0_peer;  // cluster addresses
  volatile uint32_t* abort_flag;
  uint32_t* err;
  uint32_t* counter;
  uint32_t slot, phase;
  int next, step, num_units;
  bool writer;

  __device__ __forceinline__ void init(uint64_t* full_, uint64_t* empty_, int32_t* unit_, volatile uint32_t* abort_,
                                       uint32_t* err_, uint32_t* counter_, int pair, int npairs, int num_units_,
                                       bool writer_) {
    full = full_;
    empty = empty_;
    unit = unit_;
    empty0_leader = cluster_map(smem_u32(empty_), 0);
    full0_peer = cluster_map(smem_u32(full_), 1);
    unit0_peer = cluster_map(smem_u32(unit_), 1);
    abort_flag = abort_;
    err = err_;
    counter = counter_;
    slot = 0;
    phase = 0;
    next = pair;
    step = npairs;
    num_units = num_units_;
    writer = writer_;
  }
  // The next unit, or -1 when there is none left (or a wait timed out).
  __device__ __forceinline__ int take() {
    if (counter == nullptr) {
      const int u = next;
      next += step;
      return u < num_units ? u : -1;
    }
    int u;
    if (writer) {
      // the odd CTA's readers released their copy of the slot from the other CTA
      if (!mbar_wait_cluster(&empty[slot], phase ^ 1u, abort_flag, err)) return -1;
      u = static_cast<int>(atomicAdd(counter, 1u));
      unit[slot] = u;
      st_cluster_u32(unit0_peer + slot * 4u, static_cast<uint32_t>(u));
      mbar_arrive(&full[slot]);
      mbar_arrive_cluster(full0_peer + slot * static_cast<uint32_t>(sizeof(uint64_t)));
    } else {
      if (!mbar_wait_cluster(&full[slot], phase, abort_flag, err)) return -1;
      u = reinterpret_cast<volatile int32_t*>(unit)[slot];
      mbar_arrive_cluster(empty0_leader + slot * static_cast<uint32_t>(sizeof(uint64_t)));
    }
    if (++slot == kUnitRing) {
      slot = 0;
      phase ^= 1u;
    }
    return u < num_units ? u : -1;
  }
  // One reader per warp: lane 0 takes the unit and hands it to the warp.
  __device__ __forceinline__ int take_warp(int lane) {
    if (counter == nullptr) return take();
    int u = 0;
    if (lane == 0) u = take();
    return __shfl_sync(0xffffffffu, u, 0);
  }
};

// ---- tile raster and L2 policy -------------------------------------------
// Tiles are walked in groups of `group` M-tiles, M fastest (raster_n = 0),
// or groups of `group` N-tiles, N fastest (raster_n = 1).
__device__ __forceinline__ void tc_raster(int raster_n, int group, int m_tiles, int n_tiles, int tile, int& mt,
                                          int& nt) {
  const int fast_tiles = raster_n ? n_tiles : m_tiles;
  const int slow_tiles = raster_n ? m_tiles : n_tiles;
  const int group_size = group * slow_tiles;
  const int gi = tile / group_size;
  const int first = gi * group;
  const int g = min(fast_tiles - first, group);
  const int in_group = tile - gi * group_size;
  const int f = first + in_group % g, sl = in_group / g;
  mt = raster_n ? sl : f;
  nt = raster_n ? f : sl;
}

__device__ __forceinline__ uint64_t tc_policy(int kind) {
  return kind == 2 ? l2_policy_evict_last() : (kind == 1 ? l2_policy_evict_first() : l2_policy_evict_normal());
}
// A TMA load that carries an L2 policy only when one was chosen (kind != 0):
// a load without the hint measured faster than one with evict_normal.
__device__ __forceinline__ void tma_load_maybe_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0,
                                                    int32_t c1, int kind, uint64_t policy) {
  if (kind != 0)
    tma_load_2d_hint(dst, map, bar, c0, c1, policy);
  else
    tma_load_2d(dst, map, bar, c0, c1);
}

// ---- host helpers (defined in gemm_tc.cu) --------------------------------
// Row-major bf16 operand view (rows x cols, pitch ld elements) with a
// box_cols x box_rows box, 128-byte swizzle, zero fill out of bounds.
bool tc_make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_cols,
                 int box_rows);
// Row-major output view (fp32 or bf16) with a 32 x 32 box whose swizzle
// matches the staging layout.
bool tc_make_out_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int dtype);
int tc_num_sms();
// Tile group size and L2 policies for the GEMM (environment overrides).
void tc_raster_choice(int m_tiles, int* raster_n, int* group, int* pol_a, int* pol_b);

}  // namespace tps
