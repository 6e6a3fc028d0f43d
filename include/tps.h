/*
 * tps.h -- C ABI of the tensor-parallel sharded GEMM library for GB300
 * (sm_103a).  Built as libtps.so from backward_tcgen05_tma_gemms_gb300/csrc.
 *
 * The library computes the forward and backward of a matrix product split
 * over P logical ranks, the column-then-row tensor-parallel MLP (plain and
 * gated), the head-split attention projections and the vocabulary-sharded
 * cross-entropy.  On one GPU the logical ranks are shard
 * partitions of the same device buffers: a result the pages concatenate is a
 * range of one output buffer, and a result the pages sum over ranks is
 * accumulated inside the producing kernel (the contraction loop runs over
 * the ranks' shard segments in rank order).  No communication library is
 * used.
 *
 * Sources (web pages, cited by title and section):
 *   [SG] "Sharded GEMM与Backprop：行、列、内维三种切分"
 *   [MC] "多卡张量：拆开计算，再合回同一结果"
 *   [TP] "第 6 课：张量并行 TP"
 *
 * Conventions for every entry point:
 *   - Memory.  Every pointer in a tps_tensor is a DEVICE pointer on the
 *     current CUDA device, owned by the caller.  The library never allocates
 *     or frees device memory; scratch space comes from the caller's
 *     `workspace` (size from the *_workspace_bytes queries).
 *   - Streams.  Work is enqueued on `cuda_stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and the call returns without waiting.
 *   - Validation.  Shapes, dtypes, layouts and partition arguments are
 *     checked on the host before anything is launched; on failure nothing is
 *     enqueued and a TPS_ERR_* code is returned.  A failed CUDA launch
 *     returns TPS_ERR_CUDA.  Conditions only the device can see (a label out
 *     of range, a wait that exceeded its time limit) are recorded in a
 *     device error word read by tps_last_device_error().
 *   - Layouts.  Tensors are strided (strides in elements); a 2-D operand must
 *     have unit stride in one of its two dimensions.  Tensors described as
 *     "(..., n)" may have extra leading dimensions, which must be mutually
 *     contiguous and are flattened into rows.
 *   - Dtypes.  Operands are all TPS_F32 (true fp32 FMA arithmetic) or all
 *     TPS_BF16 (bf16 operands, fp32 accumulation on the tcgen05 tensor
 *     cores).  Results named "fp32" are always TPS_F32.
 *   - Thread safety.  Entry points may be called from several host threads;
 *     launches on one stream execute in issue order.
 *   - CUDA graphs.  tps_matmul_fwd_bwd, tps_mlp_fwd_bwd, tps_glu_mlp_fwd_bwd,
 *     tps_attn_qkv_fwd, tps_attn_qkv_bwd, tps_attn_out_fwd_bwd,
 *     tps_vocab_ce_fwd_bwd and tps_vocab_ce_fwd_bwd_ex enqueue only kernel
 *     launches and memsets on `cuda_stream`; their one-time set-up runs on
 *     the first call on a device.  After one such call they may be captured
 *     into a CUDA graph; a replay reads and writes the buffers given at
 *     capture.  tps_last_device_error synchronizes and must not be captured.
 */
#ifndef TPS_H_
#define TPS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
enum { TPS_F32 = 0, TPS_BF16 = 1, TPS_I32 = 2, TPS_I64 = 3 };

/* A strided tensor view.  `data` is a device pointer (host pointer only
 * where an entry point says so); shape/stride entries past `ndim` are
 * ignored.  Strides are in elements, not bytes. */
typedef struct tps_tensor {
  void* data;
  int32_t dtype;
  int32_t ndim; /* 1..4 */
  int64_t shape[4];
  int64_t stride[4];
} tps_tensor;

/* Status codes.  TPS_ERR_SHAPE and TPS_ERR_PARTITION are the two errors of
 * [SG] "Python 参考实现" (ValueError('shape') / ValueError('partition')). */
enum {
  TPS_OK = 0,
  TPS_ERR_SHAPE = 1,     /* wrong rank, mismatched dimensions, wrong output shape */
  TPS_ERR_PARTITION = 2, /* parts/tp < 1, unknown axis */
  TPS_ERR_DTYPE = 3,     /* unsupported or mixed element types */
  TPS_ERR_LAYOUT = 4,    /* no unit stride, or leading dims not flattenable */
  TPS_ERR_LABEL = 5,     /* a label outside [0, V) (reported by the device) */
  TPS_ERR_WORKSPACE = 6, /* workspace missing, too small or misaligned */
  TPS_ERR_CUDA = 7,      /* a CUDA runtime call failed */
  TPS_ERR_TIMEOUT = 8,   /* a device-side wait exceeded its limit */
  TPS_ERR_ARG = 9,       /* NULL where a tensor is required, bad enum */
  TPS_ERR_BOUNDS = 10    /* a kernel store fell outside its output (debug builds only) */
};

/* Split axes of tps_matmul_fwd_bwd ([SG] "解题路线" steps 2-4). */
enum { TPS_AXIS_ROWS = 0, TPS_AXIS_COLUMNS = 1, TPS_AXIS_INNER = 2 };

/* Element-wise activation phi of the MLP (and the gate of the gated MLP).
 *   GELU_ERF : x * Phi(x) -- torch's default gelu used by [TP] "参考答案".
 *   GELU_TANH: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
 *   TANH     : tanh, with phi' = 1 - H^2 as [MC] "02 / BACKWARD" writes.
 *   SILU     : x sigma(x), one of the element-wise activations [TP] core
 *              concept 2.A step 3 names (SwiGLU's gate). */
enum { TPS_ACT_GELU_ERF = 0, TPS_ACT_GELU_TANH = 1, TPS_ACT_TANH = 2, TPS_ACT_SILU = 3 };

/* Weight layouts.  IN_OUT: W1 is d x F and W2 is F x d (math notation
 * Y = phi(X W1) W2 of [MC] "01 / COLUMN THEN ROW").  OUT_IN: torch
 * nn.Linear layout, W1 is F x d and W2 is d x F ([TP] "参考答案",
 * x @ w.T).  For the CE head: IN_OUT is d x V, OUT_IN is V x d. */
enum { TPS_W_IN_OUT = 0, TPS_W_OUT_IN = 1 };

/* ------------------------------------------------------------------------
 * tps_plan_shards -- array_split shard plan ([SG] "Python 参考实现";
 * [SG] "手动走一遍": K=5, parts=2 gives 3/2; parts > dim gives empty shards).
 * Writes offsets[0..parts] (caller-owned HOST array of parts+1 entries) with
 * offsets[i] = i*floor(dim/parts) + min(i, dim mod parts): the first
 * (dim mod parts) shards get one extra element.
 * Returns TPS_ERR_PARTITION if parts < 1, TPS_ERR_SHAPE if dim < 0,
 * TPS_ERR_ARG if offsets is NULL.  Host only, no CUDA call.
 * ---------------------------------------------------------------------- */
int tps_plan_shards(int64_t dim, int32_t parts, int64_t* offsets);

/* ------------------------------------------------------------------------
 * tps_matmul_fwd_bwd -- forward and backward of L = <G, AB> split over
 * `parts` logical ranks along `axis` ([SG] "题意与假设", "解题路线" 1-4):
 *   Y = A B,  dA = G B^T,  dB = A^T G.
 *   ROWS    : A and G split by rows; Y and dA are row-concatenated layouts,
 *             dB = sum_r A_r^T G_r is reduced inside the dB kernel.
 *   COLUMNS : B and G split by columns; Y and dB are column-concatenated,
 *             dA = sum_r G_r B_r^T is reduced in-kernel.
 *   INNER   : A split by columns, B by rows; Y = sum_r A_r B_r is reduced
 *             in-kernel, dA and dB are concatenated along K.
 * A (M x K), B (K x N), G (M x N): all TPS_F32 or all TPS_BF16.
 * Y (M x N), dA (M x K), dB (K x N): TPS_F32; any may be NULL to skip it.
 * Uneven and empty shards are legal.  No division by `parts` anywhere.
 * Errors: TPS_ERR_SHAPE (non-2-D, K or G mismatch, wrong output shape),
 * TPS_ERR_PARTITION (parts < 1, unknown axis), TPS_ERR_DTYPE, TPS_ERR_LAYOUT.
 * ---------------------------------------------------------------------- */
int tps_matmul_fwd_bwd(const tps_tensor* A, const tps_tensor* B, const tps_tensor* G, int32_t parts,
                       int32_t axis, const tps_tensor* Y, const tps_tensor* dA, const tps_tensor* dB,
                       void* cuda_stream);

/* ------------------------------------------------------------------------
 * tps_mlp_fwd_bwd -- column-then-row tensor-parallel MLP, forward and
 * backward, over `tp` logical ranks that split the hidden width F
 * ([MC] "01 / COLUMN THEN ROW" and "02 / BACKWARD"; [TP] core concept 2.A):
 *   rank r owns columns F_r of W1 and rows F_r of W2 (array_split of F);
 *   H_r = phi(X W1_r) stays local, Y = sum_r H_r W2_r (one in-kernel sum);
 *   dZ_r = (G_Y W2_r^T) * phi'(X W1_r), dW2_r = H_r^T G_Y, dW1_r = X^T dZ_r,
 *   dX = sum_r dZ_r W1_r^T (in-kernel sum).  The replicated G_Y is used
 *   once per rank and never summed again.
 * X (..., d) and GY (..., d): same dtype (F32 or BF16), rows T.
 * W1, W2: layout `weight_layout` (TPS_W_IN_OUT or TPS_W_OUT_IN), same dtype.
 * Y, dX (..., d) fp32; dW1, dW2 fp32 with the shapes of W1, W2.
 * `workspace` (device, 256-byte aligned, >= tps_mlp_workspace_bytes) holds
 * the pre-activation X W1, the activation and dZ, all in the operand dtype
 * (bf16 runs keep phi'(X W1) from the bf16 pre-activation).
 * Errors as tps_matmul_fwd_bwd, plus TPS_ERR_WORKSPACE, TPS_ERR_ARG (act).
 * ---------------------------------------------------------------------- */
int tps_mlp_fwd_bwd(const tps_tensor* X, const tps_tensor* W1, const tps_tensor* W2, const tps_tensor* GY,
                    int32_t tp, int32_t act, int32_t weight_layout, const tps_tensor* Y, const tps_tensor* dX,
                    const tps_tensor* dW1, const tps_tensor* dW2, void* workspace, size_t workspace_bytes,
                    void* cuda_stream);

/* Workspace bytes tps_mlp_fwd_bwd needs for T tokens, model width d, hidden
 * width F and operand dtype `dtype` (tp does not change it). */
size_t tps_mlp_workspace_bytes(int64_t T, int64_t d, int64_t F, int32_t tp, int32_t dtype);

/* ------------------------------------------------------------------------
 * tps_mlp_fwd_bwd_noalloc -- tps_mlp_fwd_bwd for callers that cannot
 * allocate device memory.  No counterpart on the source pages: this is a
 * deployment variant.  Some callers cannot obtain a workspace: code running
 * under a framework or server that owns all device memory through its own
 * allocator and forbids side allocations, or code on a latency-critical path
 * that must not call cudaMalloc (which synchronizes the device).  This entry
 * point takes the same arguments minus the workspace and allocates nothing
 * (no cudaMalloc, no cudaFree, no allocating library call): its scratch is
 * a static device array of TPS_MLP_NOALLOC_SCRATCH_BYTES (32 MiB).
 *   - Sizes whose scratch (tps_mlp_workspace_bytes) exceeds the array are
 *     rejected with TPS_ERR_WORKSPACE before anything is launched; for bf16
 *     operands that is T x F > 5,592,320.
 *   - Every call looks up the array's device address (cudaGetSymbolAddress,
 *     with the call's device current).  Under lazy module loading (the CUDA
 *     default) the first call on a device is also when the driver loads the
 *     library's device code there and reserves the 32 MiB, which can
 *     synchronize the device; the device then holds the array until the
 *     process exits.  Make that first call, or a warm-up call, before any
 *     stream capture and before latency-critical work.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents (every byte is written before it is read, so nothing needs
 *     clearing).  Calls that overlap on the GPU race on the array: the
 *     caller must serialise them (one stream, or events between streams).
 * Results are the same as tps_mlp_fwd_bwd's for the same inputs.
 * ---------------------------------------------------------------------- */
#define TPS_MLP_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int tps_mlp_fwd_bwd_noalloc(const tps_tensor* X, const tps_tensor* W1, const tps_tensor* W2, const tps_tensor* GY,
                            int32_t tp, int32_t act, int32_t weight_layout, const tps_tensor* Y,
                            const tps_tensor* dX, const tps_tensor* dW1, const tps_tensor* dW2, void* cuda_stream);

/* ------------------------------------------------------------------------
 * tps_glu_mlp_fwd_bwd -- the gated column-then-row MLP (SwiGLU for
 * act = TPS_ACT_SILU), forward and backward, split over `tp` logical ranks
 * along the hidden width F.  [TP] reference answer Q1 puts the gate/up
 * projections and the activation in the column-parallel layer and the down
 * projection in the row-parallel one; both Wg and Wu are split along F by
 * the same array_split plan, so the gating is shard-local ([TP] core
 * concept 2.A step 3) and only the outputs Y and dX are rank sums:
 *   Hg = X Wg, U = X Wu, A = phi(Hg) * U, Y = sum_r A_r W2_r;
 *   dA = GY W2^T, dU = dA * phi(Hg), dHg = dA * U * phi'(Hg),
 *   dWg = X^T dHg, dWu = X^T dU, dW2 = A^T GY,
 *   dX = sum_r (dHg_r Wg_r^T + dU_r Wu_r^T).
 * The pages give no gating formula; this is the usual gated linear unit.
 * X, GY (..., d); Wg, Wu: d x F (TPS_W_IN_OUT) or F x d (TPS_W_OUT_IN),
 * W2: F x d or d x F; all F32 or all BF16.  Outputs Y, dX (..., d) and
 * dWg, dWu, dW2 (their weights' shapes) are F32.  For bf16 operands the
 * gate and up projections run as one tensor-core GEMM whose epilogue forms
 * A; A, dHg and dU are bf16 GEMM operands, Hg and U stay fp32.
 * `workspace` >= tps_glu_mlp_workspace_bytes bytes, 256-byte aligned.
 * ---------------------------------------------------------------------- */
int tps_glu_mlp_fwd_bwd(const tps_tensor* X, const tps_tensor* Wg, const tps_tensor* Wu, const tps_tensor* W2,
                        const tps_tensor* GY, int32_t tp, int32_t act, int32_t weight_layout, const tps_tensor* Y,
                        const tps_tensor* dX, const tps_tensor* dWg, const tps_tensor* dWu, const tps_tensor* dW2,
                        void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Workspace bytes tps_glu_mlp_fwd_bwd needs: 8 T F + 3 T F x (operand
 * element size), each part rounded up to 256 bytes. */
size_t tps_glu_mlp_workspace_bytes(int64_t T, int64_t d, int64_t F, int32_t tp, int32_t dtype);

/* ------------------------------------------------------------------------
 * Attention projections, split over `tp` logical ranks by heads
 * ([TP] core concept 2.B: W_Q, W_K, W_V column-parallel along the output
 * heads, W_O row-parallel along its input heads, one sum at the output).
 * The attention core between them is not part of this library: its context
 * C and its gradients dQ, dK, dV are inputs.
 *
 * tps_plan_heads -- the head-aligned plan ([TP] core concept 3 item 4).
 * Query heads split evenly: n_heads mod tp must be 0.  KV heads (grouped
 * query attention, n_heads mod n_kv_heads = 0) split evenly when
 * n_kv_heads mod tp = 0, else each KV head is replicated on tp / n_kv_heads
 * ranks (tp mod n_kv_heads = 0); other counts return TPS_ERR_PARTITION.
 * Writes q_off[0..tp] (rank r owns query heads [q_off[r], q_off[r+1])),
 * kv_first[0..tp-1] (first KV head of rank r), *kv_count (KV heads per
 * rank) and *kv_replicas (ranks holding each KV head).  Any output may be
 * NULL.  Host only; no device work.
 * ---------------------------------------------------------------------- */
int tps_plan_heads(int32_t n_heads, int32_t n_kv_heads, int32_t tp, int64_t* q_off, int64_t* kv_first,
                   int32_t* kv_count, int32_t* kv_replicas);

/* tps_attn_qkv_fwd -- Q = X Wq, K = X Wk, V = X Wv.  X (..., d); Wq d x nq
 * and Wk, Wv d x nkv (TPS_W_IN_OUT) or their transposes (TPS_W_OUT_IN),
 * with nq = n_heads * dh and nkv = n_kv_heads * dh; all F32 or all BF16.
 * Q (T x nq), K, V (T x nkv): F32 or BF16 (one dtype for all three), rows
 * contiguous.  Rank r's heads are a column range of each output.  For bf16
 * the three projections run as one tensor-core launch over their
 * concatenated columns when every boundary falls on 128 columns. */
int tps_attn_qkv_fwd(const tps_tensor* X, const tps_tensor* Wq, const tps_tensor* Wk, const tps_tensor* Wv,
                     int32_t n_heads, int32_t n_kv_heads, int32_t tp, int32_t weight_layout, const tps_tensor* Q,
                     const tps_tensor* K, const tps_tensor* V, void* cuda_stream);

/* tps_attn_qkv_bwd -- given dQ, dK, dV (the operand dtype; with replicated
 * KV heads dK and dV summed over the replicas): dWq = X^T dQ,
 * dWk = X^T dK, dWv = X^T dV (each rank's head columns) and
 * dX = sum_r (dQ_r Wq_r^T + dK_r Wk_r^T + dV_r Wv_r^T), one GEMM whose K
 * loop runs over the three branches.  dX (..., d) and the weight
 * gradients (their weights' shapes) are F32. */
int tps_attn_qkv_bwd(const tps_tensor* X, const tps_tensor* Wq, const tps_tensor* Wk, const tps_tensor* Wv,
                     const tps_tensor* dQ, const tps_tensor* dK, const tps_tensor* dV, int32_t n_heads,
                     int32_t n_kv_heads, int32_t tp, int32_t weight_layout, const tps_tensor* dX,
                     const tps_tensor* dWq, const tps_tensor* dWk, const tps_tensor* dWv, void* cuda_stream);

/* tps_attn_out_fwd_bwd -- the output projection: Y = sum_r C_r Wo_r (the
 * row-parallel sum over the ranks' heads), dC = GY Wo^T, dWo = C^T GY.
 * C (T x nq) and GY (..., d) in the operand dtype, Wo nq x d (IN_OUT) or
 * d x nq (OUT_IN); n_heads mod tp must be 0.  Y and dWo F32; dC F32 or
 * BF16 (the attention core's backward input). */
int tps_attn_out_fwd_bwd(const tps_tensor* C, const tps_tensor* Wo, const tps_tensor* GY, int32_t n_heads,
                         int32_t tp, int32_t weight_layout, const tps_tensor* Y, const tps_tensor* dC,
                         const tps_tensor* dWo, void* cuda_stream);

/* ------------------------------------------------------------------------
 * tps_vocab_ce_fwd_bwd -- cross-entropy over a vocabulary split into `tp`
 * contiguous shards (array_split of V), forward and backward
 * ([MC] "04 / VOCABULARY SHARDS"; single supervised position per token, no
 * label smoothing, no ignore index):
 *   z = h Whead (T x V, kept in the workspace: on the tensor-core path --
 *   bf16 operands, shards of at least 128 columns -- as bf16 relative to
 *   the max of each row's 128-column tile, with those maxima and the fp32
 *   logit at each label beside it; otherwise fp32);
 *   per token and shard r: m_r = max_{j in V_r} z_j, s_r = sum e^{z_j - m_r};
 *   combined: m = max_r m_r, s = sum_r s_r e^{m_r - m},
 *   loss = log s + m - z_y;  dlogits_j = e^{z_j - m}/s - 1[j = y];
 *   dHidden = dlogits Whead^T, summed over all shards (no division by tp).
 * h (..., d): F32 or BF16.  Whead: d x V (TPS_W_IN_OUT) or V x d
 * (TPS_W_OUT_IN), same dtype.  labels (T): TPS_I64 or TPS_I32 in [0, V).
 * loss (T) fp32.  dlogits (T x V): the operand dtype (bf16 for bf16 runs).
 * dHidden (..., d) fp32.  owner (T) TPS_I32 or NULL: the rank whose shard
 * holds the label.  `workspace`: 256-B aligned, at least
 * tps_ce_workspace_bytes (enough for every path), or
 * tps_ce_workspace_bytes_ex for the operand dtype when the call takes the
 * tensor-core path; a smaller workspace fails with TPS_ERR_WORKSPACE before
 * anything is launched.
 * A label outside [0, V) makes that token's loss NaN and its owner -1, and
 * sets TPS_ERR_LABEL in the device error word.
 * ---------------------------------------------------------------------- */
int tps_vocab_ce_fwd_bwd(const tps_tensor* h, const tps_tensor* Whead, const tps_tensor* labels, int32_t tp,
                         int32_t weight_layout, const tps_tensor* loss, const tps_tensor* dlogits,
                         const tps_tensor* dHidden, const tps_tensor* owner, void* workspace,
                         size_t workspace_bytes, void* cuda_stream);

/* Workspace bytes tps_vocab_ce_fwd_bwd and tps_vocab_ce_fwd_bwd_ex need for
 * T tokens, vocabulary V and `tp` shards on any path (fp32 logits). */
size_t tps_ce_workspace_bytes(int64_t T, int64_t V, int32_t tp);

/* Workspace bytes for operands of `dtype` (TPS_F32 or TPS_BF16).  With bf16
 * operands and shards of at least 128 columns (V / tp >= 128) the logits
 * are kept as bf16, which halves their T x V region (4.2 GB -> 2.1 GB at
 * T = 8192, V = 128256).  That size assumes the tensor-core path: h and
 * Whead 16-byte aligned, unit stride along their rows and row pitches that
 * are multiples of 16 bytes.  Operands that do not qualify run the fp32
 * path and need tps_ce_workspace_bytes.  Returns 0 for T < 0, V < 0 or
 * tp < 1. */
size_t tps_ce_workspace_bytes_ex(int64_t T, int64_t V, int32_t tp, int32_t dtype);

/* ------------------------------------------------------------------------
 * tps_vocab_ce_fwd_bwd_ex -- tps_vocab_ce_fwd_bwd with the extensions a
 * production loss needs, which [MC] "04 / VOCABULARY SHARDS" names after its
 * worked example (a vocabulary padded to a shardable size, an ignore_index)
 * and [SG] "易错点与追问" raises (a mean whose denominator is the same on every
 * rank even when ranks hold different numbers of supervised tokens), plus
 * the head's own gradient dWhead = h^T dlogits, the other half of the
 * backward of z = h Whead ([SG] "解题路线" step 1: dB = A^T G).
 *   options->vocab_size (0 = V): columns [vocab_size, V) of Whead are
 *     padding.  They are left out of every softmax, their dlogits are 0,
 *     and a label there is an error.  Shards stay the array_split of the
 *     padded V (so `owner` is the rank of the padded plan).
 *   options->ignore_index (TPS_NO_IGNORE = none): a token whose label
 *     equals it has loss 0, dlogits row 0, owner -1, and is not counted.
 *   options->reduction: TPS_REDUCE_NONE, _SUM or _MEAN.  `loss` always
 *     holds the per-token losses; `loss_reduced` (one f32, may be NULL)
 *     receives sum_t loss_t (SUM) or sum_t loss_t / D (MEAN), where D =
 *     options->denominator if > 0 (e.g. the job-wide count of supervised
 *     tokens, summed over data-parallel ranks by the caller), else the
 *     number of supervised tokens of this call (1 if none).  dlogits,
 *     dHidden and dWhead are the gradients of sum_t loss_t (NONE, SUM) or
 *     of the mean (MEAN, i.e. divided by D).
 *   dWhead (Whead's shape, f32, may be NULL): the head's gradient, a
 *     tensor-core GEMM over the T tokens for bf16 operands.
 * options == NULL means all defaults (no padding, no ignore, NONE).
 * Other arguments, workspace size and errors as tps_vocab_ce_fwd_bwd;
 * additionally TPS_ERR_SHAPE for vocab_size outside [0, V] and TPS_ERR_ARG
 * for an unknown reduction or a negative / non-finite denominator.
 * ---------------------------------------------------------------------- */
#define TPS_NO_IGNORE INT64_MIN
enum { TPS_REDUCE_NONE = 0, TPS_REDUCE_SUM = 1, TPS_REDUCE_MEAN = 2 };
typedef struct tps_ce_options {
  int64_t ignore_index;
  int64_t vocab_size;
  int32_t reduction;
  int32_t reserved; /* must be 0 */
  double denominator;
} tps_ce_options;
int tps_vocab_ce_fwd_bwd_ex(const tps_tensor* h, const tps_tensor* Whead, const tps_tensor* labels, int32_t tp,
                            int32_t weight_layout, const tps_ce_options* options, const tps_tensor* loss,
                            const tps_tensor* loss_reduced, const tps_tensor* dlogits, const tps_tensor* dHidden,
                            const tps_tensor* dWhead, const tps_tensor* owner, void* workspace,
                            size_t workspace_bytes, void* cuda_stream);

/* ------------------------------------------------------------------------
 * tps_last_device_error -- synchronizes `cuda_stream`, then reads and clears
 * the current device's error word.  Returns TPS_OK, TPS_ERR_TIMEOUT (a
 * kernel gave up waiting and exited early; its outputs are invalid),
 * TPS_ERR_LABEL, TPS_ERR_BOUNDS (debug builds: a store outside its output
 * was skipped), or TPS_ERR_CUDA if the synchronization itself failed.
 * ---------------------------------------------------------------------- */
int tps_last_device_error(void* cuda_stream);

/* ------------------------------------------------------------------------
 * tps_build_flags -- how this library was built: TPS_BUILD_DEBUG is set in
 * the debug build (compiled with TPS_DEBUG=1), whose kernels check every
 * direct epilogue store, every CE statistics store and every store of the
 * CE core against the bounds of its output -- the stand-in for a memory
 * sanitizer (TMA stores need no check: the hardware clips each box to its
 * tensor map, built with the output's extent).  A store outside its output is skipped
 * and recorded as TPS_ERR_BOUNDS in the device error word; nothing traps.
 * No counterpart on the source pages.
 * ---------------------------------------------------------------------- */
#define TPS_BUILD_DEBUG 1
int tps_build_flags(void);

/* ------------------------------------------------------------------------
 * tps_selftest_wait_timeout -- failure-detection self test.  Launches one
 * thread that waits on a barrier nothing arrives on, with the same bounded
 * wait the pipelined kernels use, giving up after `limit_ns` (1 ns .. 2 s).
 * The kernel then returns normally and the next tps_last_device_error()
 * reports TPS_ERR_TIMEOUT; the CUDA context stays usable.  Returns
 * TPS_ERR_ARG for a limit outside that range.
 * ---------------------------------------------------------------------- */
int tps_selftest_wait_timeout(uint64_t limit_ns, void* cuda_stream);

/* Static description of a status code. */
const char* tps_strerror(int code);

/* Detail of the last failure on the calling host thread ("" if none). */
const char* tps_last_error_detail(void);

/* ------------------------------------------------------------------------
 * Launch profiler.  While enabled, every kernel the library launches is
 * bracketed by two CUDA events recorded on its own stream.
 * tps_profile_reset clears the records and enables recording;
 * tps_profile_stop disables it.  tps_profile_summary synchronizes the
 * recorded events and writes, for kernel family i < n (host arrays of
 * `cap` entries, NULL to skip): its name, number of launches, total device
 * milliseconds, total algorithmic FLOPs and bytes.  Returns n, or a
 * negative TPS_ERR_* code.  tps_launch_count returns the number of kernels
 * launched since the last reset, whether or not profiling is enabled.
 * ---------------------------------------------------------------------- */
int tps_profile_reset(int enable);
int tps_profile_stop(void);
int tps_profile_summary(int cap, const char** names, int64_t* launches, double* total_ms, double* flops,
                        double* bytes);
int64_t tps_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* TPS_H_ */
