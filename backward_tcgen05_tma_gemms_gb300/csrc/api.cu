// api.cu -- the C ABI of include/tps.h: validation, shard planning, launch
// orchestration, the device error word and the launch profiler.
//
// Nothing here allocates device memory: operands, results and workspace all
// belong to the caller.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.cuh"
#include "tps.h"

namespace tps {

// ------------------------------------------------------------ error detail
static thread_local std::string t_detail;

static int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_detail = buf;
  return code;
}

void set_error_detail(const char* msg) { t_detail = msg; }

// ------------------------------------------------------------ device error word
// One word per device; kernels OR TPS_DEVERR_* bits into it.
__device__ uint32_t g_dev_err_word;

static std::mutex g_err_mu;
static std::vector<uint32_t*> g_err_addr;  // indexed by device ordinal

static uint32_t* dev_err_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (static_cast<int>(g_err_addr.size()) <= dev) g_err_addr.resize(dev + 1, nullptr);
  if (g_err_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_err_word) != cudaSuccess) return nullptr;
    g_err_addr[dev] = static_cast<uint32_t*>(p);
  }
  return g_err_addr[dev];
}

uint32_t* device_error_word() { return dev_err_ptr(); }

// ------------------------------------------------------------ profiler
struct ProfRecord {
  std::string name;  // "kind:label"
  double flops, bytes;
  cudaEvent_t start, stop;
};
static std::mutex g_prof_mu;
static bool g_prof_on = false;
static std::vector<ProfRecord> g_prof;
static std::vector<cudaEvent_t> g_event_pool;
static int64_t g_launches = 0;
static std::vector<std::string> g_summary_names;  // storage for tps_profile_summary

static cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

ProfScope::ProfScope(const char* kind, const char* label, double flops, double bytes, cudaStream_t s)
    : slot(-1), stream(s) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on) return;
  ProfRecord r{std::string(kind) + ":" + label, flops, bytes, take_event(), take_event()};
  cudaEventRecord(r.start, s);
  g_prof.push_back(r);
  slot = static_cast<int>(g_prof.size()) - 1;
}
ProfScope::~ProfScope() {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (slot < static_cast<int>(g_prof.size())) cudaEventRecord(g_prof[slot].stop, stream);
}
void note_launch() {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  ++g_launches;
}

// ------------------------------------------------------------ tensor views
struct Mat {  // 2-D strided view
  void* data = nullptr;
  int dtype = 0;
  int64_t rows = 0, cols = 0, sr = 0, sc = 0;
};

static const char* dtname(int d) {
  switch (d) {
    case TPS_F32: return "f32";
    case TPS_BF16: return "bf16";
    case TPS_I32: return "i32";
    case TPS_I64: return "i64";
    default: return "?";
  }
}

// View `t` as a matrix.  flatten: leading dims (all but the last) are
// merged into rows, which requires them to be mutually contiguous.
// The view must have unit stride in one dimension (either one when a
// dimension has extent <= 1).
static int as_mat(const tps_tensor* t, const char* name, bool flatten, Mat* m) {
  if (t == nullptr) return fail(TPS_ERR_ARG, "%s: missing tensor", name);
  if (t->ndim < 1 || t->ndim > 4) return fail(TPS_ERR_SHAPE, "%s: ndim %d", name, t->ndim);
  int64_t numel = 1;
  for (int i = 0; i < t->ndim; ++i) {
    if (t->shape[i] < 0) return fail(TPS_ERR_SHAPE, "%s: negative extent", name);
    numel *= t->shape[i];
  }
  // An empty tensor may have no storage (NULL data); nothing reads it.
  if (t->data == nullptr && numel > 0) return fail(TPS_ERR_ARG, "%s: missing data", name);
  if (!flatten && t->ndim != 2) return fail(TPS_ERR_SHAPE, "%s: expected a 2-D tensor, got %d-D", name, t->ndim);
  if (flatten && t->ndim < 2) return fail(TPS_ERR_SHAPE, "%s: expected (..., n), got 1-D", name);
  m->data = t->data;
  m->dtype = t->dtype;
  const int last = t->ndim - 1;
  m->cols = t->shape[last];
  m->sc = t->stride[last];
  int64_t rows = 1;
  for (int i = 0; i < last; ++i) rows *= t->shape[i];
  m->rows = rows;
  // row stride: the stride of the innermost leading dim; the others must nest
  m->sr = t->stride[last - 1];
  for (int i = 0; i < last - 1; ++i) {
    if (t->shape[i] > 1 && t->stride[i] != t->stride[i + 1] * t->shape[i + 1])
      return fail(TPS_ERR_LAYOUT, "%s: leading dimensions are not contiguous", name);
  }
  if (m->rows <= 1) m->sr = (m->sc == 1) ? (m->cols > 0 ? m->cols : 1) : 1;
  if (m->cols <= 1) m->sc = (m->sr == 1) ? (m->rows > 0 ? m->rows : 1) : 1;
  if (m->rows <= 1 && m->cols <= 1) {
    m->sr = 1;
    m->sc = 1;
  }
  if (m->sr != 1 && m->sc != 1) return fail(TPS_ERR_LAYOUT, "%s: no unit stride (strides %lld, %lld)", name,
                                            (long long)m->sr, (long long)m->sc);
  return TPS_OK;
}

static int expect(const Mat& m, const char* name, int64_t rows, int64_t cols) {
  if (m.rows != rows || m.cols != cols)
    return fail(TPS_ERR_SHAPE, "%s: shape (%lld, %lld), expected (%lld, %lld)", name, (long long)m.rows,
                (long long)m.cols, (long long)rows, (long long)cols);
  return TPS_OK;
}

// ------------------------------------------------------------ fill kernel
__global__ void fill_kernel(void* base, int dtype, int64_t rows, int64_t cols, int64_t sr, int64_t sc, float v) {
  const int64_t n = rows * cols;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / cols, c = i % cols;
    if (dtype == TPS_F32)
      static_cast<float*>(base)[r * sr + c * sc] = v;
    else
      static_cast<__nv_bfloat16*>(base)[r * sr + c * sc] = __float2bfloat16_rn(v);
  }
}

static int launch_fill(void* base, int dtype, int64_t rows, int64_t cols, int64_t sr, int64_t sc,
                       cudaStream_t stream) {
  if (rows <= 0 || cols <= 0 || base == nullptr) return TPS_OK;
  const int64_t n = rows * cols;
  const int blocks = static_cast<int>(n / 256 + 1 < 4096 ? n / 256 + 1 : 4096);
  ProfScope prof("fill", "zero", 0.0, double(n) * (dtype == TPS_F32 ? 4 : 2), stream);
  fill_kernel<<<blocks, 256, 0, stream>>>(base, dtype, rows, cols, sr, sc, 0.0f);
  note_launch();
  return cudaPeekAtLastError() == cudaSuccess ? TPS_OK : TPS_ERR_CUDA;
}

// ------------------------------------------------------------ GEMM dispatch
// Output orientation: the kernels write row-major D.  A column-major output
// (unit stride along M) is produced as D^T = B^T A^T with the roles of the
// operands swapped.  Epilogues other than a plain store only ever target the
// library's own row-major workspace.
static int run_gemm(GemmDesc g, int64_t d_sm, int64_t d_sn, cudaStream_t stream) {
  if (g.M == 0 || g.N == 0) return TPS_OK;
  uint32_t* err = dev_err_ptr();
  if (err == nullptr) return fail(TPS_ERR_CUDA, "cannot resolve the device error word");
  // Drop empty contraction segments (the first non-empty one moves to the front).
  for (int pass = 0; pass < 2; ++pass) {
    if (g.K == 0 && (g.K2 > 0 || g.K3 > 0)) {
      g.a = g.a2; g.a_sm = g.a2_sm; g.a_sk = g.a2_sk;
      g.b = g.b2; g.b_sk = g.b2_sk; g.b_sn = g.b2_sn;
      g.K = g.K2;
      g.a2 = g.a3; g.a2_sm = g.a3_sm; g.a2_sk = g.a3_sk;
      g.b2 = g.b3; g.b2_sk = g.b3_sk; g.b2_sn = g.b3_sn;
      g.K2 = g.K3;
      g.K3 = 0;
    }
  }
  if (g.K2 == 0 && g.K3 > 0) {
    g.a2 = g.a3; g.a2_sm = g.a3_sm; g.a2_sk = g.a3_sk;
    g.b2 = g.b3; g.b2_sk = g.b3_sk; g.b2_sn = g.b3_sn;
    g.K2 = g.K3;
    g.K3 = 0;
  }
  if (g.n_segs > 1) {  // column segments: each output on its own
    if (g.K == 0) {
      for (int s = 0; s < g.n_segs; ++s) {
        const int rc = launch_fill(g.nd[s], g.epi.d_dtype, g.M, g.n_cols[s], g.nldd[s], 1, stream);
        if (rc) return rc;
      }
      return TPS_OK;
    }
    if (!gemm_tc_supported(g)) {  // one GEMM per segment
      for (int s = 0; s < g.n_segs; ++s) {
        GemmDesc t = g;
        t.n_segs = 1;
        t.N = g.n_cols[s];
        t.b = g.nb[s];
        t.b_sk = g.nb_sk[s];
        t.b_sn = g.nb_sn[s];
        t.epi.d = g.nd[s];
        const int rc = run_gemm(t, g.nldd[s], 1, stream);
        if (rc) return rc;
      }
      return TPS_OK;
    }
    g.epi.dbg_rows = g.M;
    g.epi.dbg_cols = g.N;
    g.epi.dbg_err = err;
    const int rc = launch_gemm_tc(g, err, stream);
    if (rc == TPS_ERR_CUDA) return fail(rc, "%s: launch failed: %s", g.name, cudaGetErrorString(cudaGetLastError()));
    return rc;
  }
  if (g.K == 0) {
    // An empty contraction is the zero matrix; phi(0) = 0 and 0 * phi' = 0
    // for every supported activation, and every gated output is a product
    // with a zero factor.
    const int m = g.epi.mode;
    const bool f32_d = (m == EPI_GLU_FWD || m == EPI_GLU_UP);  // Hg, U; EPI_ACT_FWD's Hp is in d_dtype
    int rc = launch_fill(g.epi.d, f32_d ? TPS_F32 : g.epi.d_dtype, g.M, g.N, d_sm, d_sn, stream);
    if (rc == TPS_OK && (m == EPI_ACT_FWD || m == EPI_GLU_FWD || m == EPI_GLU_UP || m == EPI_GLU_BWD))
      rc = launch_fill(g.epi.d2, g.epi.d2_dtype, g.M, g.N, g.epi.ldd2, 1, stream);
    if (rc == TPS_OK && m == EPI_GLU_FWD) rc = launch_fill(g.epi.d3, TPS_F32, g.M, g.N, g.epi.ldd3, 1, stream);
    return rc;
  }
  if (d_sn != 1) {
    if (d_sm != 1 || g.epi.mode != EPI_STORE) return fail(TPS_ERR_LAYOUT, "%s: unsupported output layout", g.name);
    GemmDesc t = g;
    t.M = g.N;
    t.N = g.M;
    t.a = g.b;
    t.a_sm = g.b_sn;
    t.a_sk = g.b_sk;
    t.b = g.a;
    t.b_sk = g.a_sk;
    t.b_sn = g.a_sm;
    t.a2 = g.b2;
    t.a2_sm = g.b2_sn;
    t.a2_sk = g.b2_sk;
    t.b2 = g.a2;
    t.b2_sk = g.a2_sk;
    t.b2_sn = g.a2_sm;
    t.a3 = g.b3;
    t.a3_sm = g.b3_sn;
    t.a3_sk = g.b3_sk;
    t.b3 = g.a3;
    t.b3_sk = g.a3_sk;
    t.b3_sn = g.a3_sm;
    t.epi.ldd = d_sn;
    t.wide = false;
    if (g.ce_grad.ms != nullptr) return fail(TPS_ERR_LAYOUT, "%s: the CE-gradient operand needs a row-major output", g.name);
    g = t;
  } else {
    g.epi.ldd = d_sm;
  }
  g.epi.dbg_rows = g.M;  // the output as the kernels write it (row-major M x N)
  g.epi.dbg_cols = g.N;
  g.epi.dbg_err = err;
  int rc;
  if (g.wide && gemm_wide_supported(g))
    rc = launch_gemm_wide(g, err, stream);
  else if (g.ce_grad.ms != nullptr)
    return fail(TPS_ERR_ARG, "%s: the CE-gradient operand needs the wide-tile kernel", g.name);
  else
    rc = gemm_tc_supported(g) ? launch_gemm_tc(g, err, stream) : launch_gemm_simt(g, err, stream);
  if (rc == TPS_ERR_CUDA) return fail(rc, "%s: launch failed: %s", g.name, cudaGetErrorString(cudaGetLastError()));
  return rc;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace tps

using namespace tps;

// ====================================================================== ABI

extern "C" int tps_plan_shards(int64_t dim, int32_t parts, int64_t* offsets) {
  if (offsets == nullptr) return fail(TPS_ERR_ARG, "offsets is NULL");
  if (parts < 1) return fail(TPS_ERR_PARTITION, "parts must be >= 1 (got %d)", parts);
  if (dim < 0) return fail(TPS_ERR_SHAPE, "dim must be >= 0");
  for (int32_t i = 0; i <= parts; ++i) offsets[i] = shard_offset(dim, parts, i);
  return TPS_OK;
}

extern "C" int tps_matmul_fwd_bwd(const tps_tensor* A, const tps_tensor* B, const tps_tensor* G, int32_t parts,
                                  int32_t axis, const tps_tensor* Y, const tps_tensor* dA, const tps_tensor* dB,
                                  void* cuda_stream) {
  t_detail.clear();
  Mat a, b, g;
  int rc;
  if ((rc = as_mat(A, "A", false, &a)) || (rc = as_mat(B, "B", false, &b)) || (rc = as_mat(G, "G", false, &g)))
    return rc;
  const int64_t M = a.rows, K = a.cols, N = b.cols;
  if (b.rows != K) return fail(TPS_ERR_SHAPE, "A is %lld x %lld but B has %lld rows", (long long)M, (long long)K,
                               (long long)b.rows);
  if ((rc = expect(g, "G", M, N))) return rc;
  if (parts < 1) return fail(TPS_ERR_PARTITION, "parts must be >= 1 (got %d)", parts);
  if (axis != TPS_AXIS_ROWS && axis != TPS_AXIS_COLUMNS && axis != TPS_AXIS_INNER)
    return fail(TPS_ERR_PARTITION, "unknown axis %d", axis);
  if ((a.dtype != TPS_F32 && a.dtype != TPS_BF16) || b.dtype != a.dtype || g.dtype != a.dtype)
    return fail(TPS_ERR_DTYPE, "A, B, G must all be f32 or all bf16 (got %s, %s, %s)", dtname(a.dtype),
                dtname(b.dtype), dtname(g.dtype));
  Mat y, da, db;
  const bool want_y = Y != nullptr, want_da = dA != nullptr, want_db = dB != nullptr;
  if (want_y && ((rc = as_mat(Y, "Y", false, &y)) || (rc = expect(y, "Y", M, N)))) return rc;
  if (want_da && ((rc = as_mat(dA, "dA", false, &da)) || (rc = expect(da, "dA", M, K)))) return rc;
  if (want_db && ((rc = as_mat(dB, "dB", false, &db)) || (rc = expect(db, "dB", K, N)))) return rc;
  for (const Mat* o : {want_y ? &y : nullptr, want_da ? &da : nullptr, want_db ? &db : nullptr})
    if (o && o->dtype != TPS_F32) return fail(TPS_ERR_DTYPE, "outputs must be f32");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);

  if (want_y) {  // Y = A B; summed over ranks for the inner split
    GemmDesc d;
    d.name = "gemm_Y";
    d.M = M; d.N = N; d.K = K; d.in_dtype = a.dtype;
    d.a = a.data; d.a_sm = a.sr; d.a_sk = a.sc;
    d.b = b.data; d.b_sk = b.sr; d.b_sn = b.sc;
    d.epi.d = y.data; d.epi.d_dtype = TPS_F32;
    d.kparts = (axis == TPS_AXIS_INNER) ? parts : 1;
    if ((rc = run_gemm(d, y.sr, y.sc, s))) return rc;
  }
  if (want_da) {  // dA = G B^T; summed over ranks for the column split
    GemmDesc d;
    d.name = "gemm_dA";
    d.M = M; d.N = K; d.K = N; d.in_dtype = a.dtype;
    d.a = g.data; d.a_sm = g.sr; d.a_sk = g.sc;
    d.b = b.data; d.b_sk = b.sc; d.b_sn = b.sr;
    d.epi.d = da.data; d.epi.d_dtype = TPS_F32;
    d.kparts = (axis == TPS_AXIS_COLUMNS) ? parts : 1;
    if ((rc = run_gemm(d, da.sr, da.sc, s))) return rc;
  }
  if (want_db) {  // dB = A^T G; summed over ranks for the row split
    GemmDesc d;
    d.name = "gemm_dB";
    d.M = K; d.N = N; d.K = M; d.in_dtype = a.dtype;
    d.a = a.data; d.a_sm = a.sc; d.a_sk = a.sr;
    d.b = g.data; d.b_sk = g.sr; d.b_sn = g.sc;
    d.epi.d = db.data; d.epi.d_dtype = TPS_F32;
    d.kparts = (axis == TPS_AXIS_ROWS) ? parts : 1;
    if ((rc = run_gemm(d, db.sr, db.sc, s))) return rc;
  }
  return TPS_OK;
}

// MLP workspace: the pre-activation, the activation and dZ, T x F each, all
// in the operand dtype.
extern "C" size_t tps_mlp_workspace_bytes(int64_t T, int64_t d, int64_t F, int32_t tp, int32_t dtype) {
  (void)d;
  (void)tp;
  if (T < 0 || F < 0) return 0;
  const size_t e = (dtype == TPS_F32) ? 4 : 2;
  const size_t n = static_cast<size_t>(T) * static_cast<size_t>(F);
  return 3 * align256(n * e);
}

// A weight's logical (in, out) strides for either layout.
static void weight_strides(const Mat& w, int layout, int64_t* s_in, int64_t* s_out) {
  if (layout == TPS_W_IN_OUT) {
    *s_in = w.sr;
    *s_out = w.sc;
  } else {
    *s_in = w.sc;
    *s_out = w.sr;
  }
}

extern "C" int tps_mlp_fwd_bwd(const tps_tensor* X, const tps_tensor* W1, const tps_tensor* W2,
                               const tps_tensor* GY, int32_t tp, int32_t act, int32_t weight_layout,
                               const tps_tensor* Y, const tps_tensor* dX, const tps_tensor* dW1,
                               const tps_tensor* dW2, void* workspace, size_t workspace_bytes,
                               void* cuda_stream) {
  t_detail.clear();
  Mat x, w1, w2, gy, y, dx, dw1, dw2;
  int rc;
  if ((rc = as_mat(X, "X", true, &x)) || (rc = as_mat(W1, "W1", false, &w1)) || (rc = as_mat(W2, "W2", false, &w2)) ||
      (rc = as_mat(GY, "GY", true, &gy)))
    return rc;
  if (weight_layout != TPS_W_IN_OUT && weight_layout != TPS_W_OUT_IN)
    return fail(TPS_ERR_ARG, "unknown weight layout %d", weight_layout);
  const bool io = weight_layout == TPS_W_IN_OUT;
  const int64_t T = x.rows, d = x.cols;
  const int64_t F = io ? w1.cols : w1.rows;
  if ((io ? w1.rows : w1.cols) != d) return fail(TPS_ERR_SHAPE, "W1 does not match X's width %lld", (long long)d);
  if ((rc = expect(w2, "W2", io ? F : d, io ? d : F))) return rc;
  if ((rc = expect(gy, "GY", T, d))) return rc;
  if (tp < 1) return fail(TPS_ERR_PARTITION, "tp must be >= 1 (got %d)", tp);
  if (act != TPS_ACT_GELU_ERF && act != TPS_ACT_GELU_TANH && act != TPS_ACT_TANH && act != TPS_ACT_SILU)
    return fail(TPS_ERR_ARG, "unknown activation %d", act);
  const int dt = x.dtype;
  if ((dt != TPS_F32 && dt != TPS_BF16) || w1.dtype != dt || w2.dtype != dt || gy.dtype != dt)
    return fail(TPS_ERR_DTYPE, "X, W1, W2, GY must all be f32 or all bf16");
  if ((rc = as_mat(Y, "Y", true, &y)) || (rc = expect(y, "Y", T, d)) || (rc = as_mat(dX, "dX", true, &dx)) ||
      (rc = expect(dx, "dX", T, d)) || (rc = as_mat(dW1, "dW1", false, &dw1)) ||
      (rc = expect(dw1, "dW1", w1.rows, w1.cols)) || (rc = as_mat(dW2, "dW2", false, &dw2)) ||
      (rc = expect(dw2, "dW2", w2.rows, w2.cols)))
    return rc;
  for (const Mat* o : {&y, &dx, &dw1, &dw2})
    if (o->dtype != TPS_F32) return fail(TPS_ERR_DTYPE, "MLP results must be f32");
  const size_t need = tps_mlp_workspace_bytes(T, d, F, tp, dt);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255)))
    return fail(TPS_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned", need);
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);

  const size_t n = static_cast<size_t>(T) * static_cast<size_t>(F);
  const size_t e = (dt == TPS_F32) ? 4 : 2;
  char* ws = static_cast<char*>(workspace);
  // T x F pre-activation, activation and dZ, each in the operand dtype.  A
  // bf16 pre-activation moves phi'(Hp) by at most phi''(x) x 2^-9 |x|,
  // which raises the relative error of dZ (one bf16 rounding already) by
  // about 5 % for GELU and SiLU, under 30 % for tanh.
  void* Hp = ws;
  void* Ha = ws + align256(n * e);
  void* dZ = ws + 2 * align256(n * e);

  int64_t w1_in, w1_out, w2_in, w2_out, dw1_in, dw1_out, dw2_in, dw2_out;
  weight_strides(w1, weight_layout, &w1_in, &w1_out);      // W1(dd, f)
  weight_strides(w2, weight_layout, &w2_in, &w2_out);      // W2(f, dd)
  weight_strides(dw1, weight_layout, &dw1_in, &dw1_out);
  weight_strides(dw2, weight_layout, &dw2_in, &dw2_out);

  {  // Hp = X W1, Ha = phi(Hp): column-parallel, each rank's columns a range of Hp
    GemmDesc g;
    g.name = "mlp_fc1_act";
    g.M = T; g.N = F; g.K = d; g.in_dtype = dt;
    g.a = x.data; g.a_sm = x.sr; g.a_sk = x.sc;
    g.b = w1.data; g.b_sk = w1_in; g.b_sn = w1_out;
    g.epi.mode = EPI_ACT_FWD; g.epi.act = act;
    g.epi.d = Hp; g.epi.d_dtype = dt;
    g.epi.d2 = Ha; g.epi.ldd2 = F; g.epi.d2_dtype = dt;
    if ((rc = run_gemm(g, F, 1, s))) return rc;
  }
  {  // Y = sum_r Ha_r W2_r: row-parallel, rank sum in the K loop
    GemmDesc g;
    g.name = "mlp_fc2";
    g.M = T; g.N = d; g.K = F; g.in_dtype = dt;
    g.a = Ha; g.a_sm = F; g.a_sk = 1;
    g.b = w2.data; g.b_sk = w2_in; g.b_sn = w2_out;
    g.epi.d = y.data; g.epi.d_dtype = TPS_F32;
    g.kparts = tp;
    if ((rc = run_gemm(g, y.sr, y.sc, s))) return rc;
  }
  {  // dZ = (GY W2^T) * phi'(Hp), per rank on its own columns
    GemmDesc g;
    g.name = "mlp_dh_act";
    g.M = T; g.N = F; g.K = d; g.in_dtype = dt;
    g.a = gy.data; g.a_sm = gy.sr; g.a_sk = gy.sc;
    g.b = w2.data; g.b_sk = w2_out; g.b_sn = w2_in;
    g.epi.mode = EPI_ACT_BWD; g.epi.act = act;
    g.epi.d = dZ; g.epi.d_dtype = dt;
    g.epi.ld_aux = F;
    if (dt == TPS_F32)
      g.epi.aux = static_cast<const float*>(Hp);
    else
      g.epi.aux_bf16 = static_cast<const uint16_t*>(Hp);
    if ((rc = run_gemm(g, F, 1, s))) return rc;
  }
  {  // dW2(f, dd) = sum_t Ha[t, f] GY[t, dd]
    GemmDesc g;
    g.name = "mlp_dW2";
    g.M = F; g.N = d; g.K = T; g.in_dtype = dt;
    g.a = Ha; g.a_sm = 1; g.a_sk = F;
    g.b = gy.data; g.b_sk = gy.sr; g.b_sn = gy.sc;
    g.epi.d = dw2.data; g.epi.d_dtype = TPS_F32;
    if ((rc = run_gemm(g, dw2_in, dw2_out, s))) return rc;
  }
  {  // dW1(dd, f) = sum_t X[t, dd] dZ[t, f]
    GemmDesc g;
    g.name = "mlp_dW1";
    g.M = d; g.N = F; g.K = T; g.in_dtype = dt;
    g.a = x.data; g.a_sm = x.sc; g.a_sk = x.sr;
    g.b = dZ; g.b_sk = F; g.b_sn = 1;
    g.epi.d = dw1.data; g.epi.d_dtype = TPS_F32;
    if ((rc = run_gemm(g, dw1_in, dw1_out, s))) return rc;
  }
  {  // dX = sum_r dZ_r W1_r^T: rank sum in the K loop
    GemmDesc g;
    g.name = "mlp_dX";
    g.M = T; g.N = d; g.K = F; g.in_dtype = dt;
    g.a = dZ; g.a_sm = F; g.a_sk = 1;
    g.b = w1.data; g.b_sk = w1_out; g.b_sn = w1_in;
    g.epi.d = dx.data; g.epi.d_dtype = TPS_F32;
    g.kparts = tp;
    if ((rc = run_gemm(g, dx.sr, dx.sc, s))) return rc;
  }
  return TPS_OK;
}

// ------------------------------------------------------------ gated MLP
// Workspace: Hg and U (T x F fp32 each), then A, dHg and dU (T x F in the
// operand dtype each).
extern "C" size_t tps_glu_mlp_workspace_bytes(int64_t T, int64_t d, int64_t F, int32_t tp, int32_t dtype) {
  (void)d;
  (void)tp;
  if (T < 0 || F < 0) return 0;
  const size_t e = (dtype == TPS_F32) ? 4 : 2;
  const size_t n = static_cast<size_t>(T) * static_cast<size_t>(F);
  return 2 * align256(n * 4) + 3 * align256(n * e);
}

extern "C" int tps_glu_mlp_fwd_bwd(const tps_tensor* X, const tps_tensor* Wg, const tps_tensor* Wu,
                                   const tps_tensor* W2, const tps_tensor* GY, int32_t tp, int32_t act,
                                   int32_t weight_layout, const tps_tensor* Y, const tps_tensor* dX,
                                   const tps_tensor* dWg, const tps_tensor* dWu, const tps_tensor* dW2,
                                   void* workspace, size_t workspace_bytes, void* cuda_stream) {
  t_detail.clear();
  Mat x, wg, wu, w2, gy, y, dx, dwg, dwu, dw2;
  int rc;
  if ((rc = as_mat(X, "X", true, &x)) || (rc = as_mat(Wg, "Wg", false, &wg)) || (rc = as_mat(Wu, "Wu", false, &wu)) ||
      (rc = as_mat(W2, "W2", false, &w2)) || (rc = as_mat(GY, "GY", true, &gy)))
    return rc;
  if (weight_layout != TPS_W_IN_OUT && weight_layout != TPS_W_OUT_IN)
    return fail(TPS_ERR_ARG, "unknown weight layout %d", weight_layout);
  const bool io = weight_layout == TPS_W_IN_OUT;
  const int64_t T = x.rows, d = x.cols;
  const int64_t F = io ? wg.cols : wg.rows;
  if ((io ? wg.rows : wg.cols) != d) return fail(TPS_ERR_SHAPE, "Wg does not match X's width %lld", (long long)d);
  if ((rc = expect(wu, "Wu", wg.rows, wg.cols))) return rc;
  if ((rc = expect(w2, "W2", io ? F : d, io ? d : F))) return rc;
  if ((rc = expect(gy, "GY", T, d))) return rc;
  if (tp < 1) return fail(TPS_ERR_PARTITION, "tp must be >= 1 (got %d)", tp);
  if (act != TPS_ACT_GELU_ERF && act != TPS_ACT_GELU_TANH && act != TPS_ACT_TANH && act != TPS_ACT_SILU)
    return fail(TPS_ERR_ARG, "unknown activation %d", act);
  const int dt = x.dtype;
  if ((dt != TPS_F32 && dt != TPS_BF16) || wg.dtype != dt || wu.dtype != dt || w2.dtype != dt || gy.dtype != dt)
    return fail(TPS_ERR_DTYPE, "X, Wg, Wu, W2, GY must all be f32 or all bf16");
  if ((rc = as_mat(Y, "Y", true, &y)) || (rc = expect(y, "Y", T, d)) || (rc = as_mat(dX, "dX", true, &dx)) ||
      (rc = expect(dx, "dX", T, d)) || (rc = as_mat(dWg, "dWg", false, &dwg)) ||
      (rc = expect(dwg, "dWg", wg.rows, wg.cols)) || (rc = as_mat(dWu, "dWu", false, &dwu)) ||
      (rc = expect(dwu, "dWu", wg.rows, wg.cols)) || (rc = as_mat(dW2, "dW2", false, &dw2)) ||
      (rc = expect(dw2, "dW2", w2.rows, w2.cols)))
    return rc;
  for (const Mat* o : {&y, &dx, &dwg, &dwu, &dw2})
    if (o->dtype != TPS_F32) return fail(TPS_ERR_DTYPE, "gated MLP results must be f32");
  const size_t need = tps_glu_mlp_workspace_bytes(T, d, F, tp, dt);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255)))
    return fail(TPS_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned", need);
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);

  const size_t n = static_cast<size_t>(T) * static_cast<size_t>(F);
  const size_t e = (dt == TPS_F32) ? 4 : 2;
  char* ws = static_cast<char*>(workspace);
  float* Hg = reinterpret_cast<float*>(ws);                          // T x F gate pre-activation
  float* U = reinterpret_cast<float*>(ws + align256(n * 4));         // T x F up projection
  void* A = ws + 2 * align256(n * 4);                                // T x F phi(Hg) * U
  void* dHg = ws + 2 * align256(n * 4) + align256(n * e);            // T x F
  void* dU = ws + 2 * align256(n * 4) + 2 * align256(n * e);         // T x F

  int64_t wg_in, wg_out, wu_in, wu_out, w2_in, w2_out;
  weight_strides(wg, weight_layout, &wg_in, &wg_out);  // Wg(dd, f)
  weight_strides(wu, weight_layout, &wu_in, &wu_out);  // Wu(dd, f)
  weight_strides(w2, weight_layout, &w2_in, &w2_out);  // W2(f, dd)
  int64_t dwg_in, dwg_out, dwu_in, dwu_out, dw2_in, dw2_out;
  weight_strides(dwg, weight_layout, &dwg_in, &dwg_out);
  weight_strides(dwu, weight_layout, &dwu_in, &dwu_out);
  weight_strides(dw2, weight_layout, &dw2_in, &dw2_out);

  {  // Hg = X Wg, U = X Wu, A = phi(Hg) * U: column-parallel, shard-local gating
    GemmDesc g;
    g.name = "glu_gate_up";
    g.M = T; g.N = F; g.K = d; g.in_dtype = dt;
    g.a = x.data; g.a_sm = x.sr; g.a_sk = x.sc;
    g.b = wg.data; g.b_sk = wg_in; g.b_sn = wg_out;
    g.b_up = wu.data;
    g.epi.mode = EPI_GLU_FWD; g.epi.act = act;
    g.epi.d = Hg; g.epi.ldd = F; g.epi.d_dtype = TPS_F32;
    g.epi.d3 = U; g.epi.ldd3 = F;
    g.epi.d2 = A; g.epi.ldd2 = F; g.epi.d2_dtype = dt;
    const bool fused = (wu_in == wg_in && wu_out == wg_out) && (T == 0 || F == 0 || d == 0 || gemm_tc_supported(g));
    if (fused) {
      if ((rc = run_gemm(g, F, 1, s))) return rc;
    } else {  // two GEMMs: Hg, then U with the gating in its epilogue
      GemmDesc h = g;
      h.name = "glu_gate";
      h.b_up = nullptr;
      h.epi = Epilogue();
      h.epi.d = Hg; h.epi.d_dtype = TPS_F32;
      if ((rc = run_gemm(h, F, 1, s))) return rc;
      GemmDesc u = h;
      u.name = "glu_up";
      u.b = wu.data; u.b_sk = wu_in; u.b_sn = wu_out;
      u.epi.mode = EPI_GLU_UP; u.epi.act = act;
      u.epi.d = U; u.epi.d_dtype = TPS_F32;
      u.epi.d2 = A; u.epi.ldd2 = F; u.epi.d2_dtype = dt;
      u.epi.aux = Hg; u.epi.ld_aux = F;
      if ((rc = run_gemm(u, F, 1, s))) return rc;
    }
  }
  {  // Y = sum_r A_r W2_r: row-parallel, rank sum in the K loop
    GemmDesc g;
    g.name = "glu_down";
    g.M = T; g.N = d; g.K = F; g.in_dtype = dt;
    g.a = A; g.a_sm = F; g.a_sk = 1;
    g.b = w2.data; g.b_sk = w2_in; g.b_sn = w2_out;
    g.epi.d = y.data; g.epi.d_dtype = TPS_F32;
    g.kparts = tp;
    if ((rc = run_gemm(g, y.sr, y.sc, s))) return rc;
  }
  {  // dA = GY W2^T; dHg = dA * U * phi'(Hg), dU = dA * phi(Hg), per rank
    GemmDesc g;
    g.name = "glu_dgate_dup";
    g.M = T; g.N = F; g.K = d; g.in_dtype = dt;
    g.a = gy.data; g.a_sm = gy.sr; g.a_sk = gy.sc;
    g.b = w2.data; g.b_sk = w2_out; g.b_sn = w2_in;
    g.epi.mode = EPI_GLU_BWD; g.epi.act = act;
    g.epi.d = dHg; g.epi.d_dtype = dt;
    g.epi.d2 = dU; g.epi.ldd2 = F; g.epi.d2_dtype = dt;
    g.epi.aux = Hg; g.epi.ld_aux = F;
    g.epi.aux2 = U; g.epi.ld_aux2 = F;
    if ((rc = run_gemm(g, F, 1, s))) return rc;
  }
  {  // dW2(f, dd) = sum_t A[t, f] GY[t, dd]
    GemmDesc g;
    g.name = "glu_dW2";
    g.M = F; g.N = d; g.K = T; g.in_dtype = dt;
    g.a = A; g.a_sm = 1; g.a_sk = F;
    g.b = gy.data; g.b_sk = gy.sr; g.b_sn = gy.sc;
    g.epi.d = dw2.data; g.epi.d_dtype = TPS_F32;
    if ((rc = run_gemm(g, dw2_in, dw2_out, s))) return rc;
  }
  {  // dWg(dd, f) = sum_t X[t, dd] dHg[t, f];  dWu likewise with dU
    GemmDesc g;
    g.name = "glu_dWg";
    g.M = d; g.N = F; g.K = T; g.in_dtype = dt;
    g.a = x.data; g.a_sm = x.sc; g.a_sk = x.sr;
    g.b = dHg; g.b_sk = F; g.b_sn = 1;
    g.epi.d = dwg.data; g.epi.d_dtype = TPS_F32;
    if ((rc = run_gemm(g, dwg_in, dwg_out, s))) return rc;
    g.name = "glu_dWu";
    g.b = dU;
    g.epi.d = dwu.data;
    if ((rc = run_gemm(g, dwu_in, dwu_out, s))) return rc;
  }
  {  // dX = sum_r (dHg_r Wg_r^T + dU_r Wu_r^T): both branches and the rank
     // sum in one K loop
    GemmDesc g;
    g.name = "glu_dX";
    g.M = T; g.N = d; g.K = F; g.in_dtype = dt;
    g.a = dHg; g.a_sm = F; g.a_sk = 1;
    g.b = wg.data; g.b_sk = wg_out; g.b_sn = wg_in;
    g.a2 = dU; g.a2_sm = F; g.a2_sk = 1;
    g.b2 = wu.data; g.b2_sk = wu_out; g.b2_sn = wu_in;
    g.K2 = F;
    g.epi.d = dx.data; g.epi.d_dtype = TPS_F32;
    g.kparts = tp;
    if ((rc = run_gemm(g, dx.sr, dx.sc, s))) return rc;
  }
  return TPS_OK;
}

// ------------------------------------------------------------ attention projections
// Head-aligned plan: query heads split evenly (H mod tp = 0); KV heads
// split evenly when H_kv mod tp = 0, else each replicated on tp / H_kv ranks
// (tp mod H_kv = 0); H mod H_kv = 0 (whole query groups per KV head).
static int plan_heads(int32_t H, int32_t Hkv, int32_t tp, int64_t* q_off, int64_t* kv_first, int32_t* kv_count,
                      int32_t* replicas) {
  if (tp < 1 || H < 1 || Hkv < 1) return fail(TPS_ERR_PARTITION, "heads and tp must be >= 1");
  if (H % tp != 0) return fail(TPS_ERR_PARTITION, "%d query heads do not split over tp=%d", H, tp);
  if (H % Hkv != 0) return fail(TPS_ERR_PARTITION, "%d query heads do not group over %d KV heads", H, Hkv);
  int32_t cnt, rep;
  if (Hkv % tp == 0) {
    cnt = Hkv / tp;
    rep = 1;
  } else if (tp % Hkv == 0) {
    cnt = 1;
    rep = tp / Hkv;
  } else {
    return fail(TPS_ERR_PARTITION, "%d KV heads neither split nor replicate evenly over tp=%d", Hkv, tp);
  }
  for (int32_t r = 0; r <= tp && q_off; ++r) q_off[r] = static_cast<int64_t>(r) * (H / tp);
  for (int32_t r = 0; r < tp && kv_first; ++r) kv_first[r] = rep > 1 ? r / rep : static_cast<int64_t>(r) * cnt;
  if (kv_count) *kv_count = cnt;
  if (replicas) *replicas = rep;
  return TPS_OK;
}

extern "C" int tps_plan_heads(int32_t n_heads, int32_t n_kv_heads, int32_t tp, int64_t* q_off, int64_t* kv_first,
                              int32_t* kv_count, int32_t* kv_replicas) {
  t_detail.clear();
  return plan_heads(n_heads, n_kv_heads, tp, q_off, kv_first, kv_count, kv_replicas);
}

// Shapes of the QKV weights: nq = H dh columns for Wq, nkv = H_kv dh for Wk
// and Wv, in either layout.
struct QkvShapes {
  int64_t T, d, nq, nkv;
  Mat x, wq, wk, wv;
};
static int qkv_shapes(const tps_tensor* X, const tps_tensor* Wq, const tps_tensor* Wk, const tps_tensor* Wv,
                      int32_t H, int32_t Hkv, int32_t tp, int32_t layout, QkvShapes* q) {
  int rc;
  if ((rc = as_mat(X, "X", true, &q->x)) || (rc = as_mat(Wq, "Wq", false, &q->wq)) ||
      (rc = as_mat(Wk, "Wk", false, &q->wk)) || (rc = as_mat(Wv, "Wv", false, &q->wv)))
    return rc;
  if (layout != TPS_W_IN_OUT && layout != TPS_W_OUT_IN) return fail(TPS_ERR_ARG, "unknown weight layout %d", layout);
  if ((rc = plan_heads(H, Hkv, tp, nullptr, nullptr, nullptr, nullptr))) return rc;
  const bool io = layout == TPS_W_IN_OUT;
  q->T = q->x.rows;
  q->d = q->x.cols;
  q->nq = io ? q->wq.cols : q->wq.rows;
  if ((io ? q->wq.rows : q->wq.cols) != q->d) return fail(TPS_ERR_SHAPE, "Wq does not match X's width");
  if (q->nq % H != 0) return fail(TPS_ERR_SHAPE, "Wq's %lld outputs are not %d whole heads", (long long)q->nq, H);
  q->nkv = (q->nq / H) * Hkv;
  if ((rc = expect(q->wk, "Wk", io ? q->d : q->nkv, io ? q->nkv : q->d)) ||
      (rc = expect(q->wv, "Wv", io ? q->d : q->nkv, io ? q->nkv : q->d)))
    return rc;
  const int dt = q->x.dtype;
  if ((dt != TPS_F32 && dt != TPS_BF16) || q->wq.dtype != dt || q->wk.dtype != dt || q->wv.dtype != dt)
    return fail(TPS_ERR_DTYPE, "X, Wq, Wk, Wv must all be f32 or all bf16");
  return TPS_OK;
}

extern "C" int tps_attn_qkv_fwd(const tps_tensor* X, const tps_tensor* Wq, const tps_tensor* Wk,
                                const tps_tensor* Wv, int32_t n_heads, int32_t n_kv_heads, int32_t tp,
                                int32_t weight_layout, const tps_tensor* Q, const tps_tensor* K, const tps_tensor* V,
                                void* cuda_stream) {
  t_detail.clear();
  QkvShapes a;
  int rc;
  if ((rc = qkv_shapes(X, Wq, Wk, Wv, n_heads, n_kv_heads, tp, weight_layout, &a))) return rc;
  Mat q, k, v;
  if ((rc = as_mat(Q, "Q", true, &q)) || (rc = expect(q, "Q", a.T, a.nq)) || (rc = as_mat(K, "K", true, &k)) ||
      (rc = expect(k, "K", a.T, a.nkv)) || (rc = as_mat(V, "V", true, &v)) || (rc = expect(v, "V", a.T, a.nkv)))
    return rc;
  if ((q.dtype != TPS_F32 && q.dtype != TPS_BF16) || k.dtype != q.dtype || v.dtype != q.dtype)
    return fail(TPS_ERR_DTYPE, "Q, K, V must share f32 or bf16");
  if ((q.sc != 1 && a.nq > 1) || (k.sc != 1 && a.nkv > 1) || (v.sc != 1 && a.nkv > 1))
    return fail(TPS_ERR_LAYOUT, "Q, K, V rows must be contiguous");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const Mat* w[3] = {&a.wq, &a.wk, &a.wv};
  const Mat* o[3] = {&q, &k, &v};
  GemmDesc g;  // Q | K | V = X [Wq | Wk | Wv]: one launch over the three column ranges
  g.name = "attn_qkv";
  g.M = a.T; g.N = a.nq + 2 * a.nkv; g.K = a.d; g.in_dtype = a.x.dtype;
  g.a = a.x.data; g.a_sm = a.x.sr; g.a_sk = a.x.sc;
  g.n_segs = 3;
  for (int i = 0; i < 3; ++i) {
    int64_t w_in, w_out;
    weight_strides(*w[i], weight_layout, &w_in, &w_out);
    g.n_cols[i] = i == 0 ? a.nq : a.nkv;
    g.nb[i] = w[i]->data; g.nb_sk[i] = w_in; g.nb_sn[i] = w_out;
    g.nd[i] = o[i]->data; g.nldd[i] = o[i]->sr;
  }
  g.b = g.nb[0]; g.b_sk = g.nb_sk[0]; g.b_sn = g.nb_sn[0];
  g.epi.d_dtype = q.dtype;
  return run_gemm(g, 0, 1, s);
}

extern "C" int tps_attn_qkv_bwd(const tps_tensor* X, const tps_tensor* Wq, const tps_tensor* Wk,
                                const tps_tensor* Wv, const tps_tensor* dQ, const tps_tensor* dK, const tps_tensor* dV,
                                int32_t n_heads, int32_t n_kv_heads, int32_t tp, int32_t weight_layout,
                                const tps_tensor* dX, const tps_tensor* dWq, const tps_tensor* dWk,
                                const tps_tensor* dWv, void* cuda_stream) {
  t_detail.clear();
  QkvShapes a;
  int rc;
  if ((rc = qkv_shapes(X, Wq, Wk, Wv, n_heads, n_kv_heads, tp, weight_layout, &a))) return rc;
  Mat dq, dk, dv, dx, dwq, dwk, dwv;
  if ((rc = as_mat(dQ, "dQ", true, &dq)) || (rc = expect(dq, "dQ", a.T, a.nq)) ||
      (rc = as_mat(dK, "dK", true, &dk)) || (rc = expect(dk, "dK", a.T, a.nkv)) ||
      (rc = as_mat(dV, "dV", true, &dv)) || (rc = expect(dv, "dV", a.T, a.nkv)) ||
      (rc = as_mat(dX, "dX", true, &dx)) || (rc = expect(dx, "dX", a.T, a.d)) ||
      (rc = as_mat(dWq, "dWq", false, &dwq)) || (rc = expect(dwq, "dWq", a.wq.rows, a.wq.cols)) ||
      (rc = as_mat(dWk, "dWk", false, &dwk)) || (rc = expect(dwk, "dWk", a.wk.rows, a.wk.cols)) ||
      (rc = as_mat(dWv, "dWv", false, &dwv)) || (rc = expect(dwv, "dWv", a.wv.rows, a.wv.cols)))
    return rc;
  const int dt = a.x.dtype;
  if (dq.dtype != dt || dk.dtype != dt || dv.dtype != dt)
    return fail(TPS_ERR_DTYPE, "dQ, dK, dV must have the operand dtype (%s)", dtname(dt));
  for (const Mat* m : {&dx, &dwq, &dwk, &dwv})
    if (m->dtype != TPS_F32) return fail(TPS_ERR_DTYPE, "projection gradients must be f32");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const Mat* w[3] = {&a.wq, &a.wk, &a.wv};
  const Mat* gr[3] = {&dq, &dk, &dv};
  const Mat* dw[3] = {&dwq, &dwk, &dwv};
  int64_t w_in[3], w_out[3];
  for (int i = 0; i < 3; ++i) weight_strides(*w[i], weight_layout, &w_in[i], &w_out[i]);
  {  // dX = sum_r (dQ_r Wq_r^T + dK_r Wk_r^T + dV_r Wv_r^T): three K segments, one K loop
    GemmDesc g;
    g.name = "attn_dX";
    g.M = a.T; g.N = a.d; g.in_dtype = dt;
    g.K = a.nq;
    g.a = dq.data; g.a_sm = dq.sr; g.a_sk = dq.sc;
    g.b = a.wq.data; g.b_sk = w_out[0]; g.b_sn = w_in[0];
    g.K2 = a.nkv;
    g.a2 = dk.data; g.a2_sm = dk.sr; g.a2_sk = dk.sc;
    g.b2 = a.wk.data; g.b2_sk = w_out[1]; g.b2_sn = w_in[1];
    g.K3 = a.nkv;
    g.a3 = dv.data; g.a3_sm = dv.sr; g.a3_sk = dv.sc;
    g.b3 = a.wv.data; g.b3_sk = w_out[2]; g.b3_sn = w_in[2];
    g.epi.d = dx.data; g.epi.d_dtype = TPS_F32;
    g.kparts = tp;
    if ((rc = run_gemm(g, dx.sr, dx.sc, s))) return rc;
  }
  // dW(dd, j) = sum_t X[t, dd] dProj[t, j]: shard-local columns.  The three
  // share A = X^T, so with row-contiguous gradients (in, out) they run as
  // one launch over the concatenated columns [dWq | dWk | dWv].
  int64_t o_in[3], o_out[3];
  bool rows_contiguous = true;
  for (int i = 0; i < 3; ++i) {
    weight_strides(*dw[i], weight_layout, &o_in[i], &o_out[i]);
    rows_contiguous = rows_contiguous && o_out[i] == 1;
  }
  if (rows_contiguous) {
    GemmDesc g;
    g.name = "attn_dWqkv";
    g.M = a.d; g.N = a.nq + 2 * a.nkv; g.K = a.T; g.in_dtype = dt;
    g.a = a.x.data; g.a_sm = a.x.sc; g.a_sk = a.x.sr;
    g.n_segs = 3;
    for (int i = 0; i < 3; ++i) {
      g.n_cols[i] = i == 0 ? a.nq : a.nkv;
      g.nb[i] = gr[i]->data; g.nb_sk[i] = gr[i]->sr; g.nb_sn[i] = gr[i]->sc;
      g.nd[i] = dw[i]->data; g.nldd[i] = o_in[i];
    }
    g.b = g.nb[0]; g.b_sk = g.nb_sk[0]; g.b_sn = g.nb_sn[0];
    g.epi.d_dtype = TPS_F32;
    return run_gemm(g, 0, 1, s);
  }
  static const char* names[3] = {"attn_dWq", "attn_dWk", "attn_dWv"};
  for (int i = 0; i < 3; ++i) {
    GemmDesc g;
    g.name = names[i];
    g.M = a.d; g.N = i == 0 ? a.nq : a.nkv; g.K = a.T; g.in_dtype = dt;
    g.a = a.x.data; g.a_sm = a.x.sc; g.a_sk = a.x.sr;
    g.b = gr[i]->data; g.b_sk = gr[i]->sr; g.b_sn = gr[i]->sc;
    g.epi.d = dw[i]->data; g.epi.d_dtype = TPS_F32;
    if ((rc = run_gemm(g, o_in[i], o_out[i], s))) return rc;
  }
  return TPS_OK;
}

extern "C" int tps_attn_out_fwd_bwd(const tps_tensor* C, const tps_tensor* Wo, const tps_tensor* GY, int32_t n_heads,
                                    int32_t tp, int32_t weight_layout, const tps_tensor* Y, const tps_tensor* dC,
                                    const tps_tensor* dWo, void* cuda_stream) {
  t_detail.clear();
  Mat c, wo, gy, y, dc, dwo;
  int rc;
  if ((rc = as_mat(C, "C", true, &c)) || (rc = as_mat(Wo, "Wo", false, &wo)) || (rc = as_mat(GY, "GY", true, &gy)))
    return rc;
  if (weight_layout != TPS_W_IN_OUT && weight_layout != TPS_W_OUT_IN)
    return fail(TPS_ERR_ARG, "unknown weight layout %d", weight_layout);
  if (tp < 1 || n_heads < 1 || n_heads % tp != 0)
    return fail(TPS_ERR_PARTITION, "%d heads do not split over tp=%d", n_heads, tp);
  const bool io = weight_layout == TPS_W_IN_OUT;
  const int64_t T = c.rows, nq = c.cols;
  const int64_t d = io ? wo.cols : wo.rows;
  if (nq % n_heads != 0) return fail(TPS_ERR_SHAPE, "C's %lld columns are not %d whole heads", (long long)nq, n_heads);
  if ((io ? wo.rows : wo.cols) != nq) return fail(TPS_ERR_SHAPE, "Wo does not match C's width");
  if ((rc = expect(gy, "GY", T, d))) return rc;
  const int dt = c.dtype;
  if ((dt != TPS_F32 && dt != TPS_BF16) || wo.dtype != dt || gy.dtype != dt)
    return fail(TPS_ERR_DTYPE, "C, Wo, GY must all be f32 or all bf16");
  if ((rc = as_mat(Y, "Y", true, &y)) || (rc = expect(y, "Y", T, d)) || (rc = as_mat(dC, "dC", true, &dc)) ||
      (rc = expect(dc, "dC", T, nq)) || (rc = as_mat(dWo, "dWo", false, &dwo)) ||
      (rc = expect(dwo, "dWo", wo.rows, wo.cols)))
    return rc;
  if (y.dtype != TPS_F32 || dwo.dtype != TPS_F32) return fail(TPS_ERR_DTYPE, "Y and dWo must be f32");
  if (dc.dtype != TPS_F32 && dc.dtype != TPS_BF16) return fail(TPS_ERR_DTYPE, "dC must be f32 or bf16");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  int64_t w_in, w_out, o_in, o_out;
  weight_strides(wo, weight_layout, &w_in, &w_out);  // Wo(j, dd)
  weight_strides(dwo, weight_layout, &o_in, &o_out);
  {  // Y = sum_r C_r Wo_r: row-parallel over the heads, rank sum in the K loop
    GemmDesc g;
    g.name = "attn_out";
    g.M = T; g.N = d; g.K = nq; g.in_dtype = dt;
    g.a = c.data; g.a_sm = c.sr; g.a_sk = c.sc;
    g.b = wo.data; g.b_sk = w_in; g.b_sn = w_out;
    g.epi.d = y.data; g.epi.d_dtype = TPS_F32;
    g.kparts = tp;
    if ((rc = run_gemm(g, y.sr, y.sc, s))) return rc;
  }
  {  // dC = GY Wo^T: each rank's head columns
    GemmDesc g;
    g.name = "attn_dC";
    g.M = T; g.N = nq; g.K = d; g.in_dtype = dt;
    g.a = gy.data; g.a_sm = gy.sr; g.a_sk = gy.sc;
    g.b = wo.data; g.b_sk = w_out; g.b_sn = w_in;
    g.epi.d = dc.data; g.epi.d_dtype = dc.dtype;
    if ((rc = run_gemm(g, dc.sr, dc.sc, s))) return rc;
  }
  {  // dWo(j, dd) = sum_t C[t, j] GY[t, dd]
    GemmDesc g;
    g.name = "attn_dWo";
    g.M = nq; g.N = d; g.K = T; g.in_dtype = dt;
    g.a = c.data; g.a_sm = c.sc; g.a_sk = c.sr;
    g.b = gy.data; g.b_sk = gy.sr; g.b_sn = gy.sc;
    g.epi.d = dwo.data; g.epi.d_dtype = TPS_F32;
    if ((rc = run_gemm(g, o_in, o_out, s))) return rc;
  }
  return TPS_OK;
}

// CE workspace: logits (T x V, fp32, or bf16 on the tensor-core path) |
// per-shard stats (T x tp x 2: the two-pass path's, or on the tensor-core
// path the statistics of tiles that straddle a shard start) | label logits
// (T) | per-tile stats (T x ceil(V/128) x 2) | per-tile shifts (T rows of
// ceil(V/128) floats, padded to a multiple of 4) | combined (m, 1/s) per
// token (T x 2)
// | 256 bytes of scalars (the count of supervised labels, int32 at +0, and
// the gradient scale, f32 at +16).
struct CeWs {
  size_t z, stats, zy, tiles, shift, ms, scal, total;
};
// Row stride of the per-tile shifts: 16-byte rows, so that a run of shifts
// starting at a multiple of 4 tiles can be copied in bulk.
static int64_t ce_shift_ld(int64_t V) { return ((V + kStatsTileN - 1) / kStatsTileN + 3) & ~int64_t(3); }
static CeWs ce_ws_layout(int64_t T, int64_t V, int32_t tp, size_t logit_bytes) {
  const size_t t = static_cast<size_t>(T);
  const size_t n_tiles = static_cast<size_t>((V + kStatsTileN - 1) / kStatsTileN);
  CeWs w;
  w.z = 0;
  w.stats = w.z + align256(t * static_cast<size_t>(V) * logit_bytes);
  w.zy = w.stats + align256(t * static_cast<size_t>(tp) * 2 * 4);
  w.tiles = w.zy + align256(t * 4);
  w.shift = w.tiles + align256(t * n_tiles * 2 * 4);
  w.ms = w.shift + align256(t * ce_shift_ld(V) * 4);
  w.scal = w.ms + align256(t * 2 * 4);
  w.total = w.scal + 256;
  return w;
}

extern "C" size_t tps_ce_workspace_bytes(int64_t T, int64_t V, int32_t tp) {
  if (T < 0 || V < 0 || tp < 1) return 0;
  return ce_ws_layout(T, V, tp, 4).total;
}

extern "C" size_t tps_ce_workspace_bytes_ex(int64_t T, int64_t V, int32_t tp, int32_t dtype) {
  if (T < 0 || V < 0 || tp < 1) return 0;
  const bool bf16_logits = dtype == TPS_BF16 && ce_tile_stats_supported(V, tp);
  return ce_ws_layout(T, V, tp, bf16_logits ? 2 : 4).total;
}

// Runs of a K split for a long-K GEMM on CTA pairs: the count (1..4, every
// run at least 256 K tiles) whose (tile, run) units fill the waves of
// resident pairs best, kept only when it fills them at least 5 % better
// than one run (the partial sums cost an extra read and write of the
// output per run).  Measured on the dHidden GEMM (V = 128256, d = 4096)
// with 256 x 256 tiles: T = 2048 (128 tiles, 1.7 waves of 76 pairs)
// 1.14-1.16 ms with four runs against 1.20-1.21 ms; T = 4096 (3.4 waves)
// 2.37 ms with two runs against 2.61 ms; T = 8192 (6.7 waves, 0.96 filled)
// 4.81-4.95 ms with one, two or four runs alike, so it keeps one.  With
// 256 x 512 tiles T = 8192 makes 256 tiles (3.4 waves): two runs, 4.34-4.40
// ms against 5.09-5.15 with one.
static int choose_ksplit(int64_t tiles, int64_t k_tiles) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 1;
  const int64_t pairs = sms / 2;
  if (pairs < 1 || tiles < 1) return 1;
  int best = 1;
  double best_fill = 0.0, one_run = 0.0;
  for (int runs = 1; runs <= 4 && k_tiles / runs >= 256; ++runs) {
    const int64_t units = tiles * runs, rounds = (units + pairs - 1) / pairs;
    const double fill = double(units) / double(rounds * pairs);
    if (runs == 1) one_run = fill;
    if (fill > best_fill + 1e-9) {
      best = runs;
      best_fill = fill;
    }
  }
  return best_fill >= 1.05 * one_run ? best : 1;
}

// Both CE entry points: `opts` NULL is the plain form (every label in
// [0, V), no reduction); `loss_reduced` and `dWhead` are nullable.
static int ce_impl(const tps_tensor* h, const tps_tensor* Whead, const tps_tensor* labels, int32_t tp,
                   int32_t weight_layout, const tps_ce_options* opts, const tps_tensor* loss,
                   const tps_tensor* loss_reduced, const tps_tensor* dlogits, const tps_tensor* dHidden,
                   const tps_tensor* dWhead, const tps_tensor* owner, void* workspace, size_t workspace_bytes,
                   void* cuda_stream) {
  t_detail.clear();
  Mat hm, w, dl, dh, dw;
  int rc;
  if ((rc = as_mat(h, "h", true, &hm)) || (rc = as_mat(Whead, "Whead", false, &w))) return rc;
  if (weight_layout != TPS_W_IN_OUT && weight_layout != TPS_W_OUT_IN)
    return fail(TPS_ERR_ARG, "unknown weight layout %d", weight_layout);
  const bool io = weight_layout == TPS_W_IN_OUT;
  const int64_t T = hm.rows, d = hm.cols;
  const int64_t V = io ? w.cols : w.rows;
  if ((io ? w.rows : w.cols) != d) return fail(TPS_ERR_SHAPE, "Whead does not match h's width %lld", (long long)d);
  if (tp < 1) return fail(TPS_ERR_PARTITION, "tp must be >= 1 (got %d)", tp);
  if (V < 1) return fail(TPS_ERR_SHAPE, "empty vocabulary");
  const int dt = hm.dtype;
  if ((dt != TPS_F32 && dt != TPS_BF16) || w.dtype != dt) return fail(TPS_ERR_DTYPE, "h and Whead must share f32 or bf16");
  // With no tokens the per-token tensors may have no storage (NULL data).
  if (labels == nullptr || (labels->data == nullptr && T > 0)) return fail(TPS_ERR_ARG, "labels missing");
  if (labels->ndim < 1 || (labels->dtype != TPS_I64 && labels->dtype != TPS_I32))
    return fail(TPS_ERR_DTYPE, "labels must be i32 or i64");
  int64_t nl = 1;
  for (int i = 0; i < labels->ndim; ++i) nl *= labels->shape[i];
  if (nl != T) return fail(TPS_ERR_SHAPE, "labels hold %lld entries for %lld tokens", (long long)nl, (long long)T);
  if (labels->stride[labels->ndim - 1] != 1 && T > 1) return fail(TPS_ERR_LAYOUT, "labels must be contiguous");
  if (loss == nullptr || (loss->data == nullptr && T > 0) || loss->dtype != TPS_F32)
    return fail(TPS_ERR_DTYPE, "loss must be f32");
  int64_t nloss = 1;
  for (int i = 0; i < loss->ndim; ++i) nloss *= loss->shape[i];
  if (nloss != T || (loss->stride[loss->ndim - 1] != 1 && T > 1)) return fail(TPS_ERR_SHAPE, "loss must be T contiguous floats");
  if ((rc = as_mat(dlogits, "dlogits", true, &dl)) || (rc = expect(dl, "dlogits", T, V))) return rc;
  if (dl.dtype != dt) return fail(TPS_ERR_DTYPE, "dlogits must have the operand dtype (%s)", dtname(dt));
  if (dl.sc != 1 && V > 1) return fail(TPS_ERR_LAYOUT, "dlogits rows must be contiguous");
  if ((rc = as_mat(dHidden, "dHidden", true, &dh)) || (rc = expect(dh, "dHidden", T, d))) return rc;
  if (dh.dtype != TPS_F32) return fail(TPS_ERR_DTYPE, "dHidden must be f32");
  int32_t* own = nullptr;
  if (owner != nullptr && owner->data != nullptr) {
    int64_t no = 1;
    for (int i = 0; i < owner->ndim; ++i) no *= owner->shape[i];
    if (owner->dtype != TPS_I32 || no != T || (owner->stride[owner->ndim - 1] != 1 && T > 1))
      return fail(TPS_ERR_SHAPE, "owner must be T contiguous i32");
    own = static_cast<int32_t*>(owner->data);
  }
  int64_t vreal = V;
  if (opts != nullptr) {
    if (opts->vocab_size < 0 || opts->vocab_size > V)
      return fail(TPS_ERR_SHAPE, "vocab_size %lld outside [0, %lld]", (long long)opts->vocab_size, (long long)V);
    if (opts->vocab_size > 0) vreal = opts->vocab_size;
    if (opts->reduction != TPS_REDUCE_NONE && opts->reduction != TPS_REDUCE_SUM && opts->reduction != TPS_REDUCE_MEAN)
      return fail(TPS_ERR_ARG, "unknown reduction %d", opts->reduction);
    if (!(opts->denominator >= 0.0) || !std::isfinite(opts->denominator))
      return fail(TPS_ERR_ARG, "denominator must be finite and >= 0");
    if (opts->reserved != 0) return fail(TPS_ERR_ARG, "reserved must be 0");
  }
  // The plain kernels serve options that change nothing.
  const bool ext = opts != nullptr && (opts->ignore_index != TPS_NO_IGNORE || vreal != V ||
                                       opts->reduction != TPS_REDUCE_NONE);
  float* red = nullptr;
  if (loss_reduced != nullptr && loss_reduced->data != nullptr) {
    int64_t n = 1;
    for (int i = 0; i < loss_reduced->ndim; ++i) n *= loss_reduced->shape[i];
    if (loss_reduced->dtype != TPS_F32 || n != 1) return fail(TPS_ERR_SHAPE, "loss_reduced must be one f32");
    red = static_cast<float*>(loss_reduced->data);
  }
  const bool want_dw = dWhead != nullptr;
  int64_t dw_in = 0, dw_out = 0;  // dWhead(dd, v) strides
  if (want_dw) {
    if ((rc = as_mat(dWhead, "dWhead", false, &dw)) || (rc = expect(dw, "dWhead", w.rows, w.cols))) return rc;
    if (dw.dtype != TPS_F32) return fail(TPS_ERR_DTYPE, "dWhead must be f32");
    weight_strides(dw, weight_layout, &dw_in, &dw_out);
  }
  int64_t w_in, w_out;
  weight_strides(w, weight_layout, &w_in, &w_out);  // W(dd, v)
  // z = h Whead: vocabulary shards are column ranges of z.  On the tensor
  // cores (shards of at least one 128-column statistics tile) the epilogue
  // also leaves each shard's partial softmax statistics per tile, and stores
  // z as bf16 relative to each tile's max, with the shifts and the fp32
  // logit at each label beside it; otherwise z is fp32.
  GemmDesc g;
  g.name = "ce_logits";
  g.M = T; g.N = V; g.K = d; g.in_dtype = dt;
  g.a = hm.data; g.a_sm = hm.sr; g.a_sk = hm.sc;
  g.b = w.data; g.b_sk = w_in; g.b_sn = w_out;
  g.epi.d_dtype = TPS_F32; g.epi.ldd = V;
  const bool fused = gemm_tc_supported(g) && ce_tile_stats_supported(V, tp);
  const CeWs lay = ce_ws_layout(T, V, tp, fused ? 2 : 4);
  if (workspace == nullptr || workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return fail(TPS_ERR_WORKSPACE, "workspace needs %zu bytes (%s logits), 256-byte aligned", lay.total,
                fused ? "bf16" : "fp32");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  if (T == 0) {  // no tokens: a zero sum and a zero head gradient
    if (red != nullptr && opts != nullptr && opts->reduction != TPS_REDUCE_NONE &&
        cudaMemsetAsync(red, 0, sizeof(float), s) != cudaSuccess)
      return fail(TPS_ERR_CUDA, "memset failed");
    if (want_dw) {
      GemmDesc gw;
      gw.name = "ce_dwhead";
      gw.M = d; gw.N = V; gw.K = 0; gw.in_dtype = dt;
      gw.epi.d = dw.data; gw.epi.d_dtype = TPS_F32;
      return run_gemm(gw, dw_in, dw_out, s);
    }
    return TPS_OK;
  }

  char* ws = static_cast<char*>(workspace);
  float* z = reinterpret_cast<float*>(ws + lay.z);
  float* stats = reinterpret_cast<float*>(ws + lay.stats);
  float* zy = reinterpret_cast<float*>(ws + lay.zy);
  float* tile_stats = reinterpret_cast<float*>(ws + lay.tiles);
  float* shift = reinterpret_cast<float*>(ws + lay.shift);
  float* ms = reinterpret_cast<float*>(ws + lay.ms);
  char* scal = ws + lay.scal;
  const int64_t n_tiles = (V + kStatsTileN - 1) / kStatsTileN;
  g.epi.d = z;
  if (fused) {
    g.epi.mode = EPI_CE_STATS;
    g.epi.d_dtype = TPS_BF16;
    g.epi.stats = tile_stats;
    g.epi.stats_b = stats;
    g.epi.n_tiles = n_tiles;
    g.epi.ce_parts = tp;
    g.epi.ce_vreal = vreal;
    g.epi.ce_shift = shift;
    g.epi.ce_shift_ld = ce_shift_ld(V);
    g.epi.ce_labels = labels->data;
    g.epi.ce_label_i64 = labels->dtype == TPS_I64 ? 1 : 0;
    g.epi.ce_zy = zy;
  }
  if ((rc = run_gemm(g, V, 1, s))) return rc;
  // dHidden = sum_r dlogits_r Whead_r^T: rank sum in the K loop
  GemmDesc gh;
  gh.name = "ce_dhidden";
  gh.M = T; gh.N = d; gh.K = V; gh.in_dtype = dt;
  gh.a = dl.data; gh.a_sm = dl.sr; gh.a_sk = 1;
  gh.b = w.data; gh.b_sk = w_out; gh.b_sn = w_in;
  gh.epi.d = dh.data; gh.epi.d_dtype = TPS_F32; gh.epi.ldd = dh.sr;
  gh.kparts = tp;
  // Wide (256 x 512) pair tiles for this long-K GEMM: 2-4 % faster than
  // 256 x 256 at T = 2048-8192 (TPS_CE_WIDE=0 keeps the 256-wide tiles).
  // TPS_CE_GRAD_IN_GEMM=1 (plain bf16 form) forms dlogits from the shifted
  // logits inside it, after the combine alone; measured 2.2 times slower
  // than the CE core and this GEMM together, so it is off by default.
  const char* wv = getenv("TPS_CE_WIDE");
  const char* gv = getenv("TPS_CE_GRAD_IN_GEMM");
  gh.wide = fused && dh.sc == 1 && (wv ? atoi(wv) != 0 : true);
  bool grad_in_gemm = gh.wide && !ext && dt == TPS_BF16 && (gv ? atoi(gv) != 0 : false);
  if (gh.wide && !gemm_wide_supported(gh)) gh.wide = grad_in_gemm = false;
  if (grad_in_gemm) {
    GemmDesc gx = gh;
    gx.a = z; gx.a_sm = V;  // the shifted bf16 logits
    gx.ce_grad.ms = ms;
    gx.ce_grad.shift = shift;
    gx.ce_grad.shift_ld = ce_shift_ld(V);
    gx.ce_grad.labels = labels->data;
    gx.ce_grad.label_i64 = labels->dtype == TPS_I64 ? 1 : 0;
    gx.ce_grad.dlogits = dl.data;
    gx.ce_grad.ldg = dl.sr;
    if (gemm_wide_supported(gx))
      gh = gx;
    else
      grad_in_gemm = false;
  }
  {
    CeDesc c;
    c.T = T; c.V = V; c.parts = tp;
    c.logits = z; c.ldz = V;
    if (fused) {
      c.logits16 = z;
      c.shift = shift;
      c.shift_ld = ce_shift_ld(V);
    }
    c.labels = labels->data; c.label_dtype = labels->dtype;
    c.loss = static_cast<float*>(loss->data);
    c.dlogits = dl.data; c.ldg = dl.sr; c.dlogits_dtype = dt;
    c.owner = own; c.stats = stats; c.zy = zy;
    if (ext) {
      c.options = true;
      c.ignore_index = opts->ignore_index;
      c.vreal = vreal;
      c.reduction = opts->reduction;
      c.denominator = opts->denominator;
      c.loss_reduced = red;
      c.count = reinterpret_cast<int32_t*>(scal);
      c.scale = reinterpret_cast<float*>(scal + 16);
    }
    uint32_t* err = dev_err_ptr();
    if (err == nullptr) return fail(TPS_ERR_CUDA, "cannot resolve the device error word");
    if (grad_in_gemm)
      rc = launch_ce_combine(c, tile_stats, n_tiles, ms, err, s);
    else
      rc = fused ? launch_ce_from_tile_stats(c, tile_stats, n_tiles, ms, err, s) : launch_ce(c, err, s, nullptr);
    if (rc) return fail(rc, "ce launch failed: %s", cudaGetErrorString(cudaGetLastError()));
  }
  {
    // The vocabulary is K here and very long, and the output has few pair
    // tiles: when they make a ragged number of waves, split K into runs
    // whose partial tiles are added into dHidden in order (the pages'
    // per-shard partial dHidden, summed) so that the (tile, run) units fill
    // the waves better.  The per-tile counters live in a region the CE
    // core has finished with: the tile statistics on the tensor-core path
    // (the GEMM that forms dlogits itself still reads the (m, 1/s) rows),
    // else the (m, 1/s) rows.
    const int64_t tiles = gh.wide ? wide_tile_count(T, d) : pair_tile_count(T, d);
    const char* ks = getenv("TPS_CE_KSPLIT");
    const int ksplit = ks ? atoi(ks) : choose_ksplit(tiles, (V + 63) / 64);
    // One more counter after the per-tile ones hands out the work units in
    // order: at T = 8192 the wide-tile GEMM took 4.35-4.40 ms against
    // 4.55-4.57 with the static round-robin, whose pairs drift apart over
    // their 2004-step tiles (TPS_CE_DYNAMIC=0 keeps the round-robin).  The
    // counter needs a zeroed word, which the fp32-logits paths' (m, 1/s)
    // region cannot spare beside the per-tile counters, so it runs on the
    // tensor-core path only.
    const char* dv = getenv("TPS_CE_DYNAMIC");
    const bool dynamic = fused && (dv ? atoi(dv) != 0 : true);
    const size_t flag_bytes = static_cast<size_t>(tiles + (dynamic ? 1 : 0)) * sizeof(uint32_t);
    uint32_t* flags = reinterpret_cast<uint32_t*>(fused ? tile_stats : ms);
    const size_t room = fused ? static_cast<size_t>(T) * static_cast<size_t>(n_tiles) * 8 : static_cast<size_t>(T) * 8;
    if ((ksplit > 1 || dynamic) && flag_bytes <= room) {
      if (cudaMemsetAsync(flags, 0, flag_bytes, s) != cudaSuccess) return fail(TPS_ERR_CUDA, "memset failed");
      if (ksplit > 1) {
        gh.ksplit = ksplit;
        gh.kflags = flags;
      }
      if (dynamic) gh.unit_counter = flags + tiles;
    }
    if ((rc = run_gemm(gh, dh.sr, dh.sc, s))) return rc;
  }
  if (want_dw) {  // dWhead = h^T dlogits; shard r's columns are its head slice
    GemmDesc g;
    g.name = "ce_dwhead";
    g.M = d; g.N = V; g.K = T; g.in_dtype = dt;
    g.a = hm.data; g.a_sm = hm.sc; g.a_sk = hm.sr;
    g.b = dl.data; g.b_sk = dl.sr; g.b_sn = 1;
    g.epi.d = dw.data; g.epi.d_dtype = TPS_F32;
    if ((rc = run_gemm(g, dw_in, dw_out, s))) return rc;
  }
  return TPS_OK;
}

extern "C" int tps_vocab_ce_fwd_bwd(const tps_tensor* h, const tps_tensor* Whead, const tps_tensor* labels,
                                    int32_t tp, int32_t weight_layout, const tps_tensor* loss,
                                    const tps_tensor* dlogits, const tps_tensor* dHidden, const tps_tensor* owner,
                                    void* workspace, size_t workspace_bytes, void* cuda_stream) {
  return ce_impl(h, Whead, labels, tp, weight_layout, nullptr, loss, nullptr, dlogits, dHidden, nullptr, owner,
                 workspace, workspace_bytes, cuda_stream);
}

extern "C" int tps_vocab_ce_fwd_bwd_ex(const tps_tensor* h, const tps_tensor* Whead, const tps_tensor* labels,
                                       int32_t tp, int32_t weight_layout, const tps_ce_options* options,
                                       const tps_tensor* loss, const tps_tensor* loss_reduced,
                                       const tps_tensor* dlogits, const tps_tensor* dHidden,
                                       const tps_tensor* dWhead, const tps_tensor* owner, void* workspace,
                                       size_t workspace_bytes, void* cuda_stream) {
  tps_ce_options defaults = {TPS_NO_IGNORE, 0, TPS_REDUCE_NONE, 0, 0.0};
  return ce_impl(h, Whead, labels, tp, weight_layout, options ? options : &defaults, loss, loss_reduced, dlogits,
                 dHidden, dWhead, owner, workspace, workspace_bytes, cuda_stream);
}

extern "C" int tps_last_device_error(void* cuda_stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
    return fail(TPS_ERR_CUDA, "stream synchronize failed: %s", cudaGetErrorString(cudaGetLastError()));
  uint32_t* p = dev_err_ptr();
  if (p == nullptr) return TPS_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_dev_err_word, sizeof(v)) != cudaSuccess) return TPS_ERR_CUDA;
  const uint32_t zero = 0;
  if (cudaMemcpyToSymbol(g_dev_err_word, &zero, sizeof(zero)) != cudaSuccess) return TPS_ERR_CUDA;
  if (v & TPS_DEVERR_TIMEOUT) return TPS_ERR_TIMEOUT;
  if (v & TPS_DEVERR_BOUNDS) return TPS_ERR_BOUNDS;
  if (v & TPS_DEVERR_LABEL) return TPS_ERR_LABEL;
  return TPS_OK;
}

extern "C" int tps_build_flags(void) { return TPS_DEBUG ? TPS_BUILD_DEBUG : 0; }

extern "C" const char* tps_strerror(int code) {
  switch (code) {
    case TPS_OK: return "ok";
    case TPS_ERR_SHAPE: return "shape";
    case TPS_ERR_PARTITION: return "partition";
    case TPS_ERR_DTYPE: return "dtype";
    case TPS_ERR_LAYOUT: return "layout";
    case TPS_ERR_LABEL: return "label out of range";
    case TPS_ERR_WORKSPACE: return "workspace";
    case TPS_ERR_CUDA: return "cuda";
    case TPS_ERR_TIMEOUT: return "device wait timed out";
    case TPS_ERR_ARG: return "argument";
    case TPS_ERR_BOUNDS: return "store outside its output (debug build)";
    default: return "unknown";
  }
}

extern "C" const char* tps_last_error_detail(void) { return t_detail.c_str(); }

extern "C" int tps_profile_reset(int enable) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& r : g_prof) {
    g_event_pool.push_back(r.start);
    g_event_pool.push_back(r.stop);
  }
  g_prof.clear();
  g_prof_on = enable != 0;
  g_launches = 0;
  return TPS_OK;
}

extern "C" int tps_profile_stop(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = false;
  return TPS_OK;
}

extern "C" int tps_profile_summary(int cap, const char** names, int64_t* launches, double* total_ms, double* flops,
                                   double* bytes) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  std::vector<std::string> fam;
  std::vector<int64_t> cnt;
  std::vector<double> ms, fl, by;
  for (auto& r : g_prof) {
    if (cudaEventSynchronize(r.stop) != cudaSuccess) return -TPS_ERR_CUDA;
    float t = 0.0f;
    if (cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess) return -TPS_ERR_CUDA;
    size_t i = 0;
    while (i < fam.size() && fam[i] != r.name) ++i;
    if (i == fam.size()) {
      fam.push_back(r.name);
      cnt.push_back(0);
      ms.push_back(0);
      fl.push_back(0);
      by.push_back(0);
    }
    cnt[i] += 1;
    ms[i] += t;
    fl[i] += r.flops;
    by[i] += r.bytes;
  }
  g_summary_names = fam;
  for (size_t i = 0; i < fam.size() && static_cast<int>(i) < cap; ++i) {
    if (names) names[i] = g_summary_names[i].c_str();
    if (launches) launches[i] = cnt[i];
    if (total_ms) total_ms[i] = ms[i];
    if (flops) flops[i] = fl[i];
    if (bytes) bytes[i] = by[i];
  }
  return static_cast<int>(fam.size());
}

extern "C" int64_t tps_launch_count(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  return g_launches;
}
