// internal.cuh -- declarations shared by the library's translation units
// (never installed, never seen by callers; the public ABI is include/tps.h).
#pragma once
#include <cuda_runtime.h>
#include <cstdint>
#include <type_traits>

#include "tps.h"

namespace tps {

// Device error word bits (read back by tps_last_device_error).
constexpr uint32_t TPS_DEVERR_TIMEOUT = 1u;
constexpr uint32_t TPS_DEVERR_LABEL = 2u;
constexpr uint32_t TPS_DEVERR_BOUNDS = 4u;  // debug builds: a store outside its output

// The debug build (TPS_DEBUG=1) checks every epilogue and cross-entropy
// store against the bounds of its output; a store outside is skipped and
// TPS_DEVERR_BOUNDS recorded.  Release builds compile the checks out.
#ifndef TPS_DEBUG
#define TPS_DEBUG 0
#endif

// ------------------------------------------------------------ epilogues
// EPI_STORE    D = acc                                  (dtype d_dtype)
// EPI_ACT_FWD  D = acc (fp32, may be null), D2 = phi(acc) (dtype d2_dtype)
// EPI_ACT_BWD  D = acc * phi'(AUX), AUX the fp32 pre-activation
// EPI_CE_STATS tensor-core kernels only.  Per (row, 128-column tile): the
//              softmax statistics of the tile's columns, split at the
//              vocabulary-shard boundary (see CeTileAcc), and the shift
//              c = max over the tile's real columns (0 when it has none);
//              D = bf16(acc - c), the logits relative to their tile's max;
//              and, per row, the fp32 logit at the row's label column
// Gated MLP (Hg = X Wg, U = X Wu, A = phi(Hg) * U):
// EPI_GLU_FWD  CTA-pair kernel only: each pair tile holds 128 gate columns
//              (from B) and the same 128 up columns (from the up operand);
//              D = Hg (fp32), D3 = U (fp32), D2 = A (dtype d2_dtype)
// EPI_GLU_UP   acc = U: D = U (fp32, may be null), D2 = phi(AUX) * U with
//              AUX = Hg (the two-GEMM form of EPI_GLU_FWD)
// EPI_GLU_BWD  acc = dA: D = dHg = acc * AUX2 * phi'(AUX), D2 = dU =
//              acc * phi(AUX), with AUX = Hg and AUX2 = U (fp32)
enum EpiMode : int {
  EPI_STORE = 0,
  EPI_ACT_FWD = 1,
  EPI_ACT_BWD = 2,
  EPI_CE_STATS = 3,
  EPI_GLU_FWD = 4,
  EPI_GLU_UP = 5,
  EPI_GLU_BWD = 6
};

// Width of the column tiles the CE statistics are kept for (the GEMM
// epilogue thread that owns a row folds this many columns at a time).
constexpr int kStatsTileN = 128;

struct Epilogue {
  int mode = EPI_STORE;
  int act = TPS_ACT_GELU_ERF;
  void* d = nullptr;          // row-major M x N, leading dimension ldd
  int64_t ldd = 0;
  int d_dtype = TPS_F32;
  void* d2 = nullptr;         // EPI_ACT_FWD activated output, row-major
  int64_t ldd2 = 0;
  int d2_dtype = TPS_BF16;
  const float* aux = nullptr; // EPI_ACT_BWD pre-activation (EPI_GLU_UP: Hg), row-major fp32
  int64_t ld_aux = 0;
  // EPI_ACT_BWD: when set, the pre-activation is read as bf16 from here
  // (row-major, leading dimension ld_aux) instead of from `aux`.  EPI_ACT_FWD
  // stores its pre-activation `d` in d_dtype (fp32 or bf16).
  const uint16_t* aux_bf16 = nullptr;
  void* d3 = nullptr;         // EPI_GLU_FWD: U, row-major fp32
  int64_t ldd3 = 0;
  const float* aux2 = nullptr;  // EPI_GLU_BWD: U, row-major fp32
  int64_t ld_aux2 = 0;
  // EPI_CE_STATS: stats[(row * n_tiles + tile) * 2 + {0, 1}] = (m_a, s_a),
  // the max and sum of e^{z - max} over the tile's columns in the shard that
  // owns the tile's first column.  When shard b starts inside the tile, the
  // same pair over the tile's columns in shard b goes to
  // stats_b[(row * ce_parts + b) * 2 + {0, 1}] (entries of shards that
  // start on a tile boundary are never written).  Shards are the
  // array_split of N into ce_parts; every shard must be at least
  // kStatsTileN wide so that a tile meets at most two.
  float* stats = nullptr;
  float* stats_b = nullptr;
  int64_t n_tiles = 0;
  int32_t ce_parts = 1;
  // Columns at or beyond ce_vreal are vocabulary padding: they are stored
  // but left out of the statistics.
  int64_t ce_vreal = INT64_MAX;
  float* ce_shift = nullptr;        // shift[row * ce_shift_ld + tile]
  int64_t ce_shift_ld = 0;          // >= n_tiles
  const void* ce_labels = nullptr;  // the label of each row, int32 or int64
  int ce_label_i64 = 0;
  float* ce_zy = nullptr;           // zy[row]: the logit at the label (labels in [0, N))
  // Debug builds: the output's extent (rows, columns) and the error word the
  // bounds checks report to.
  int64_t dbg_rows = 0, dbg_cols = 0;
  uint32_t* dbg_err = nullptr;
};

// The vocabulary CE's gradient as the A operand of the dHidden GEMM, formed
// from the logits GEMM's shifted bf16 logits as their tiles arrive in
// shared memory: A(t, j) = e^{z_tj - m_t} / s_t - 1[j = y_t], with z_tj
// stored as bf16(z_tj - c), c the shift of the 128-column statistics tile
// holding column j.  The GEMM's A pointer is then the shifted logits (K =
// the vocabulary), and the tile pass over the output's first column block
// also writes A once to `dlogits` (bf16, leading dimension ldg).  Rows
// whose label lies outside [0, K) get no one-hot term.
struct CeGradOperand {
  const float* ms = nullptr;     // T x 2: (m, 1/s) of each row
  const float* shift = nullptr;  // shift[t * shift_ld + j / kStatsTileN]
  int64_t shift_ld = 0;
  const void* labels = nullptr;  // T labels, int32 or int64
  int label_i64 = 0;
  void* dlogits = nullptr;
  int64_t ldg = 0;
};

// One GEMM D[M x N] = sum_k A(m, k) B(k, n), operands addressed by element
// strides: A(m, k) = a[m * a_sm + k * a_sk], B(k, n) = b[k * b_sk + n * b_sn].
// One stride of each operand is 1 (its contiguous dimension).
struct GemmDesc {
  int64_t M = 0, N = 0, K = 0;
  int in_dtype = TPS_BF16;
  const void* a = nullptr;
  int64_t a_sm = 0, a_sk = 0;
  const void* b = nullptr;
  int64_t b_sk = 0, b_sn = 0;
  Epilogue epi;
  // Number of logical ranks the contraction dimension K is sharded over
  // (array_split plan).  1 when K is not sharded.
  int32_t kparts = 1;
  // EPI_GLU_FWD: the up projection's weight, with b's strides (b is the
  // gate's); N counts gate (= up) columns.
  const void* b_up = nullptr;
  // Optional further contraction segments: D = A B + A2 B2 + A3 B3 over K2
  // and K3 more terms (same operand dtype and contiguous dimensions as A
  // and B).  Under a K split each logical rank owns its array_split segment
  // of every one.
  const void* a2 = nullptr;
  int64_t a2_sm = 0, a2_sk = 0;
  const void* b2 = nullptr;
  int64_t b2_sk = 0, b2_sn = 0;
  int64_t K2 = 0;
  const void* a3 = nullptr;
  int64_t a3_sm = 0, a3_sk = 0;
  const void* b3 = nullptr;
  int64_t b3_sk = 0, b3_sn = 0;
  int64_t K3 = 0;
  // Column segments (EPI_STORE, CTA-pair kernel): the N columns are up to
  // three GEMMs that share A, segment s being n_cols[s] wide (every
  // segment but the last a multiple of 128), with its own B (base nb[s],
  // strides nb_sk[s], nb_sn[s], the same dimension contiguous in every
  // segment) and its own row-major output (base nd[s], leading dimension
  // nldd[s], dtype epi.d_dtype).  b, b_sk, b_sn describe segment 0.
  int n_segs = 1;
  int64_t n_cols[3] = {0, 0, 0};
  const void* nb[3] = {nullptr, nullptr, nullptr};
  int64_t nb_sk[3] = {0, 0, 0}, nb_sn[3] = {0, 0, 0};
  void* nd[3] = {nullptr, nullptr, nullptr};
  int64_t nldd[3] = {0, 0, 0};
  // K split into ksplit equal runs of K tiles (CTA-pair kernel, EPI_STORE
  // to an fp32 output through TMA stores): the work units are (tile, run)
  // pairs, run-major; run 0 stores its partial tile and run s > 0 adds its
  // partial into the output with a TMA reduction once run s - 1 of the same
  // tile is in memory, which `kflags` (one zeroed counter per pair tile,
  // m_tiles x n_tiles) tracks.  The sum is taken in run order, so results
  // are deterministic.  Ignored (one run) when the conditions do not hold.
  int ksplit = 1;
  uint32_t* kflags = nullptr;
  // Wide tiles (gemm_wide.cu): 256 x 512 pair tiles with one accumulator,
  // for long contractions whose epilogue is a small part of each tile
  // (EPI_STORE to fp32 through TMA, A K-major); kflags then has one
  // counter per wide tile (wide_tile_count).  ce_grad.ms set: A is formed
  // as the CE gradient (CeGradOperand), which needs the wide tiles.
  bool wide = false;
  CeGradOperand ce_grad;
  // CTA-pair kernels (wide and 256 x 256 tiles): when set (a zeroed
  // counter), the pairs take their work units in increasing order from this
  // counter as they start on them, instead of the static round-robin (pair
  // p: units p, p + pairs, ...).  Results are the same bits either way.
  uint32_t* unit_counter = nullptr;
  const char* name = "gemm";  // label used by the launch profiler
};
// Pair tiles of a GEMM on the CTA-pair kernel (the size of GemmDesc::kflags).
inline int64_t pair_tile_count(int64_t M, int64_t N) { return ((M + 255) / 256) * ((N + 255) / 256); }
inline int64_t wide_tile_count(int64_t M, int64_t N) { return ((M + 255) / 256) * ((N + 511) / 512); }

// Launchers (return a TPS_* status; asynchronous on `stream`).
int launch_gemm_tc(const GemmDesc& g, uint32_t* dev_err, cudaStream_t stream);   // picks one of:
int launch_gemm_tc1(const GemmDesc& g, uint32_t* dev_err, cudaStream_t stream);  // one CTA per tile
int launch_gemm_tc2(const GemmDesc& g, uint32_t* dev_err, cudaStream_t stream);  // CTA pairs
int launch_gemm_simt(const GemmDesc& g, uint32_t* dev_err, cudaStream_t stream);
int launch_gemm_wide(const GemmDesc& g, uint32_t* dev_err, cudaStream_t stream);  // wide CTA-pair tiles
bool gemm_wide_supported(const GemmDesc& g);
bool gemm_tc_supported(const GemmDesc& g);

struct CeDesc {
  int64_t T = 0, V = 0;
  int32_t parts = 1;
  const float* logits = nullptr;  // T x V fp32, leading dimension ldz
  int64_t ldz = 0;
  // launch_ce_from_tile_stats reads the logits the EPI_CE_STATS epilogue
  // left instead: T x V bf16 relative to their tile's shift (leading
  // dimension ldz), the shifts (T x n_tiles) and the label logits in zy.
  const void* logits16 = nullptr;
  const float* shift = nullptr;
  int64_t shift_ld = 0;           // row stride of `shift`, a multiple of 4 floats
  const void* labels = nullptr;   // T, int32 or int64
  int label_dtype = TPS_I64;
  float* loss = nullptr;          // T fp32
  void* dlogits = nullptr;        // T x V, leading dimension ldg
  int64_t ldg = 0;
  int dlogits_dtype = TPS_BF16;
  int32_t* owner = nullptr;       // T, nullable
  float* stats = nullptr;         // workspace T x parts x 2 (two-pass path)
  float* zy = nullptr;            // workspace T: the logit at each label
  // Extended form (tps_vocab_ce_fwd_bwd_ex); when `options` is false the
  // fields below are ignored and every label must lie in [0, V).
  bool options = false;
  int64_t ignore_index = TPS_NO_IGNORE;  // label value that is not supervised
  int64_t vreal = 0;                     // columns [vreal, V) are padding
  int reduction = TPS_REDUCE_NONE;
  double denominator = 0.0;              // > 0: the mean's divisor
  float* loss_reduced = nullptr;         // 1 float, nullable
  int32_t* count = nullptr;              // workspace: supervised labels
  float* scale = nullptr;                // workspace: 1 / divisor
};
// Vocabulary CE when the logits GEMM already produced per-tile statistics
// (EPI_CE_STATS): each shard's (m_r, s_r), the global log-sum-exp, the loss
// and the owner are formed from them, and dlogits is streamed from the
// shifted bf16 logits -- in one kernel when the logits rows are 16-byte
// aligned, else by a combine kernel and a streaming kernel.
// `tile_stats` is T x n_tiles x 2 floats and c.stats (T x parts x 2) holds
// the statistics of the tiles in which a shard starts (Epilogue::stats_b);
// `ms` is T x 2 floats of scratch; the logits come from c.logits16,
// c.shift and c.zy.
int launch_ce_from_tile_stats(const CeDesc& c, const float* tile_stats, int64_t n_tiles, float* ms,
                              uint32_t* dev_err, cudaStream_t stream);
bool ce_tile_stats_supported(int64_t V, int32_t parts);
// Only the combine of launch_ce_from_tile_stats (loss, owner, (m, 1/s) in
// `ms`), for dlogits formed inside the dHidden GEMM; plain form only.
int launch_ce_combine(const CeDesc& c, const float* tile_stats, int64_t n_tiles, float* ms, uint32_t* dev_err,
                      cudaStream_t stream);

// Picks the one-read cluster kernel when the shard plan allows it, else the
// two-pass kernels.  `used_cluster` reports the choice.
int launch_ce(const CeDesc& c, uint32_t* dev_err, cudaStream_t stream, bool* used_cluster);
bool ce_cluster_supported(int64_t V, int32_t parts, int dlogits_dtype);

// Launch profiler hooks (api.cu).  When profiling is on, each kernel launch
// is bracketed by CUDA events on its stream.
struct ProfScope {
  // `kind` names the kernel, `label` the call site (e.g. "gemm_tc", "mlp_dX").
  ProfScope(const char* kind, const char* label, double flops, double bytes, cudaStream_t s);
  ~ProfScope();
  int slot;
  cudaStream_t stream;
};
void note_launch();
// Device address of the current device's error word (nullptr on failure).
uint32_t* device_error_word();
// Sets the text tps_last_error_detail returns on this host thread.
void set_error_detail(const char* msg);

// array_split plan, closed form: offset(i) = i * (d / P) + min(i, d mod P).
__host__ __device__ inline int64_t shard_offset(int64_t dim, int64_t parts, int64_t i) {
  const int64_t q = dim / parts, r = dim % parts;
  return i * q + (i < r ? i : r);
}

// ------------------------------------------------------------ activations
// 2^x with the hardware approximation (flushes subnormal results to 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// GELU (erf form) x * Phi(x), with CUDA's erff; tanh with CUDA's tanhf.
// GELU tanh approximation 0.5 x (1 + tanh(z)), z = sqrt(2/pi) (x + 0.044715
// x^3), evaluated through the identity 0.5 (1 + tanh(z)) = 1 / (1 + e^{-2z})
// = 1 / (1 + 2^{x (k1 + k3 x^2)}), k1 = -2 sqrt(2/pi) log2(e), k3 = 0.044715
// k1 (one ex2 and one reciprocal, the constants folded so that the
// epilogues spend few instructions per element); the exponent is clamped at
// 80 log2(e), where the sigmoid is already 0 in fp32.  Derivatives are those
// of the definitions: for the tanh form, with s = 1/(1 + e^{-2z}),
// d/dx = s + 2 x s (1 - s) sqrt(2/pi) (1 + 3 * 0.044715 x^2)
//      = s + x (c1 + c3 x^2) (s - s^2), c1 = 2 sqrt(2/pi), c3 = 3 * 0.044715 c1.
constexpr float kGeluK1 = -2.0f * 0.79788456080286536f * 1.4426950408889634f;
constexpr float kGeluK3 = 0.044715f * kGeluK1;
constexpr float kGeluC1 = 2.0f * 0.79788456080286536f;
constexpr float kGeluC3 = 3.0f * 0.044715f * kGeluC1;
constexpr float kExpClampLog2 = 80.0f * 1.4426950408889634f;
__device__ __forceinline__ float gelu_tanh_sigmoid_x2(float x, float x2) {
  return __fdividef(1.0f, 1.0f + ex2_approx(fminf(x * fmaf(kGeluK3, x2, kGeluK1), kExpClampLog2)));
}
__device__ __forceinline__ float gelu_tanh_sigmoid(float x) { return gelu_tanh_sigmoid_x2(x, x * x); }
// Logistic sigma(x) = 1 / (1 + e^{-x}) = 1 / (1 + 2^{-x log2(e)}); the
// exponent is clamped at 80 log2(e) (sigma is already 0 in fp32 there) so the
// division never sees infinity.
__device__ __forceinline__ float logistic(float x) {
  return __fdividef(1.0f, 1.0f + ex2_approx(fminf(x * -1.4426950408889634f, kExpClampLog2)));
}
__device__ __forceinline__ float act_fwd(int act, float x) {
  if (act == TPS_ACT_GELU_ERF) return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
  if (act == TPS_ACT_GELU_TANH) return x * gelu_tanh_sigmoid(x);
  if (act == TPS_ACT_SILU) return x * logistic(x);
  return tanhf(x);
}
__device__ __forceinline__ float act_grad(int act, float x) {
  if (act == TPS_ACT_GELU_ERF) {
    const float cdf = 0.5f * (1.0f + erff(x * 0.70710678118654752f));
    const float pdf = 0.39894228040143268f * expf(-0.5f * x * x);
    return cdf + x * pdf;
  }
  if (act == TPS_ACT_GELU_TANH) {
    const float x2 = x * x;
    const float s = gelu_tanh_sigmoid_x2(x, x2);
    return fmaf(x * fmaf(kGeluC3, x2, kGeluC1), fmaf(-s, s, s), s);
  }
  if (act == TPS_ACT_SILU) {  // d/dx x s(x) = s + x s (1 - s)
    const float s = logistic(x);
    return fmaf(x, fmaf(-s, s, s), s);
  }
  const float h = tanhf(x);
  return 1.0f - h * h;
}
// Compile-time forms: act_dispatch calls f with the activation as a type,
// once per chunk, so the unrolled element loops carry no activation branch.
template <int ACT>
__device__ __forceinline__ float act_fwd_c(float x) { return act_fwd(ACT, x); }
template <int ACT>
__device__ __forceinline__ float act_grad_c(float x) { return act_grad(ACT, x); }
template <typename F>
__device__ __forceinline__ void act_dispatch(int act, F&& f) {
  switch (act) {
    case TPS_ACT_GELU_ERF: f(std::integral_constant<int, TPS_ACT_GELU_ERF>()); break;
    case TPS_ACT_GELU_TANH: f(std::integral_constant<int, TPS_ACT_GELU_TANH>()); break;
    case TPS_ACT_SILU: f(std::integral_constant<int, TPS_ACT_SILU>()); break;
    default: f(std::integral_constant<int, TPS_ACT_TANH>()); break;
  }
}
// phi(x) and phi'(x) together (one exponential for SiLU).
__device__ __forceinline__ void act_fwd_grad(int act, float x, float& f, float& g) {
  if (act == TPS_ACT_SILU) {
    const float s = logistic(x);
    f = x * s;
    g = fmaf(x, fmaf(-s, s, s), s);
  } else {
    f = act_fwd(act, x);
    g = act_grad(act, x);
  }
}
template <int ACT>
__device__ __forceinline__ void act_fwd_grad_c(float x, float& f, float& g) { act_fwd_grad(ACT, x, f, g); }

}  // namespace tps
