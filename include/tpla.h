/*
 * tpla.h -- tensor-parallel linear algebra on one GPU (B300, sm_103a).
 *
 * The Megatron-style split of a transformer layer's linear algebra, with every
 * tensor-parallel shard materialised on ONE device and the all-reduce's sum
 * done inside the kernel:
 *
 *   column-parallel linear   Y_i = act(X . W_i^T + b_i)   (W split on outputs)
 *   row-parallel linear      Y   = sum_i X_i . W_i^T + b  (W split on inputs,
 *                                                           bias added once)
 *   FFN block                column -> act per shard -> row
 *   attention projections    QKV column-split by head group, O row-split by
 *                            head
 *
 * Sources (page title -- section):
 *   [P3] "Understanding Tensor Parallelism for Multi-GPU LLM Serving" --
 *        "How Tensor Parallelism Works Under the Hood" and the
 *        ColumnParallelLinear / RowParallelLinear modules of "Implementing
 *        Tensor Parallelism with Hugging Face Accelerate".
 *   [P4] "What is tensor parallelism?" -- "How a layer is split", "Why it
 *        helps when serving".
 *   [P5] "Tensor parallel serving" -- "Simulating the split, and proving it is
 *        correct", "Column-parallel and row-parallel layers, paired".
 *
 * Conventions shared by every entry point
 *   - Weights are stored like nn.Linear: [out_features, in_features],
 *     row-major.  Activations are row-major [tokens, features].
 *   - Every data pointer is DEVICE memory owned by the caller; host arrays of
 *     shard pointers (w_shards, b_shards) are read during the call only.  The
 *     library never allocates, frees or retains caller memory.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream).  Outputs must not alias inputs.
 *   - Arguments are validated before anything is launched.  On any error the
 *     call returns a status, writes nothing and launches nothing.  No C++
 *     exception crosses this boundary.
 *   - Alignment: X, weight shards and the FFN workspace are 16-byte aligned,
 *     and every input row stride (ld * element size) and weight row length
 *     (in_features * element size, per shard) is a multiple of 16 bytes, as
 *     128-bit and TMA loads need.  Outputs and biases need only their natural
 *     alignment.  Otherwise TP_ERR_ALIGNMENT.
 *   - 1 <= tp <= TP_MAX_TP.  tp = 1 is the unsharded layer.
 *   - M = 0 (no tokens) is a valid empty call: TP_OK, nothing launched.
 *   - Arithmetic: bf16 inputs are multiplied exactly and accumulated in fp32;
 *     bias, activation and the shard sum are fp32; the result is rounded once
 *     to the output dtype (round to nearest even for bf16).  fp32 inputs use
 *     fp32 FMA on CUDA cores (no TF32).
 *   - Determinism: the summation order of a column-parallel output depends
 *     only on (M, K, the total output count N, dtype, act) and the device's
 *     SM count, never on tp or the shard widths, so a sharded run is
 *     bit-identical to the same call with tp = 1.  (Decode-shaped calls whose
 *     outputs would give each SM fewer than 128 weight rows split K over a
 *     cluster and add the partials in a fixed order; whether they do depends
 *     on N, K and M.)
 */
#ifndef TPLA_H
#define TPLA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the same underlying type). */
typedef struct CUstream_st* tp_stream_t;

typedef enum {
  TP_OK = 0,
  TP_ERR_NULL = 1,            /* a required pointer is NULL */
  TP_ERR_NOT_DIVISIBLE = 2,   /* tp does not divide a split dimension */
  TP_ERR_BAD_SHAPE = 3,       /* negative/zero size, tp out of range, ld too small */
  TP_ERR_DTYPE = 4,           /* unsupported dtype combination */
  TP_ERR_ALIGNMENT = 5,       /* pointer or stride not 16-byte aligned */
  TP_ERR_CUDA = 6,            /* a CUDA runtime/driver call failed */
  TP_ERR_DEVICE_TIMEOUT = 7,  /* a bounded device-side wait gave up */
  TP_ERR_UNSUPPORTED = 8,     /* valid but not offered (e.g. a bias where none is defined) */
  TP_ERR_DEVICE_CHECK = 9     /* checked build only: a kernel's index check failed (access skipped) */
} tp_status;

typedef enum { TP_F32 = 0, TP_BF16 = 1 } tp_dtype;

typedef enum {
  TP_ACT_NONE = 0,
  TP_ACT_GELU_ERF = 1, /* 0.5 z (1 + erf(z / sqrt 2)), the torch F.gelu default */
  TP_ACT_SWIGLU = 2    /* silu(x.Wg^T) * (x.Wu^T); packed gate/up shards, no bias */
} tp_act;

typedef enum {
  TP_SPLIT_COLUMN = 0,    /* rows [i*out/tp, (i+1)*out/tp) of W  -> [out/tp, in]  */
  TP_SPLIT_ROW = 1,       /* cols [i*in/tp,  (i+1)*in/tp)  of W  -> [out, in/tp]  */
  TP_SPLIT_QKV_HEADS = 2, /* head group i of a [Q;K;V] weight    -> [(H+2Hkv)/tp*hd, in] */
  TP_SPLIT_GATE_UP = 3    /* gate/up rows of shard i, packed     -> [2*G*ceil(out/tp/G), in] */
} tp_split;

/* Largest tensor-parallel size accepted. */
#define TP_MAX_TP 16

/*
 * Row-group size G of a packed gate/up (SwiGLU) shard.  Packed shard i holds,
 * for each group j = 0, 1, ...: gate rows i*out/tp + j*G + [0, G) followed by
 * up rows i*out/tp + j*G + [0, G).  Rows past out/tp in the last group are
 * zero.  One GEMM tile therefore holds matching gate and up outputs.
 */
#define TP_GATE_UP_GROUP 128

/* Human-readable name of a status; never NULL. */
const char* tp_status_string(tp_status status);

/*
 * tp_shard_shape -- rows and columns of one weight shard produced by
 * tp_shard_weights for this split.
 *
 * Defined by the shard shapes of ColumnParallelLinear ([out/tp, in]) and
 * RowParallelLinear ([out, in/tp]) in [P3], the head split of [P4], and the
 * gate/up packing above.  out_f/in_f are the unsharded weight's dimensions;
 * n_heads, n_kv_heads, head_dim are read for TP_SPLIT_QKV_HEADS only (then
 * out_f must equal (n_heads + 2*n_kv_heads) * head_dim).
 * Errors: TP_ERR_NULL (rows or cols NULL), TP_ERR_BAD_SHAPE, TP_ERR_NOT_DIVISIBLE.
 */
tp_status tp_shard_shape(tp_split split, int tp, int64_t out_f, int64_t in_f,
                         int n_heads, int n_kv_heads, int head_dim,
                         int64_t* rows, int64_t* cols);

/*
 * tp_shard_weights -- cut an unsharded weight (and bias) into tp contiguous
 * shards on the device.  A bit-preserving copy; one-time setup.
 *
 * [P3] ColumnParallelLinear / RowParallelLinear (shard shapes, the asserts
 * out_features % tp == 0 and in_features % tp == 0); [P5] "Simulating the
 * split" (W[:split], W[split:] and b likewise); [P4] (heads to different
 * GPUs; tp divides the head count).
 *
 *   split        which cut (tp_split).
 *   wdt          element type of W, W_up and the shards (TP_F32 or TP_BF16).
 *   W            [out_f, in_f] unsharded weight (gate weight for GATE_UP),
 *                device memory.
 *   W_up         [out_f, in_f] up weight for TP_SPLIT_GATE_UP, else NULL.
 *   b            fp32 [out_f] bias or NULL.  Sharded for COLUMN and
 *                QKV_HEADS.  ROW and GATE_UP take no bias here
 *                (TP_ERR_UNSUPPORTED): a row-parallel bias is added once,
 *                after the shard sum, and is passed whole to
 *                row_parallel_linear.
 *   n_heads, n_kv_heads, head_dim   QKV_HEADS only; W's rows are
 *                [Q heads 0..H-1; K heads 0..Hkv-1; V heads 0..Hkv-1], each
 *                head_dim rows.  Shard i gets Q heads [i*H/tp, (i+1)*H/tp),
 *                then K and V heads [i*Hkv/tp, (i+1)*Hkv/tp).
 *   w_shards     host array of tp device pointers, each to a buffer of
 *                tp_shard_shape() rows x cols elements (row-major, contiguous).
 *   b_shards     host array of tp device pointers to fp32 [rows] buffers, or
 *                NULL; required exactly when b is given.
 * Errors: TP_ERR_NULL, TP_ERR_BAD_SHAPE, TP_ERR_NOT_DIVISIBLE (tp must divide
 * out_f, in_f, H or Hkv as the split needs), TP_ERR_ALIGNMENT, TP_ERR_DTYPE,
 * TP_ERR_UNSUPPORTED, TP_ERR_CUDA.
 */
tp_status tp_shard_weights(tp_split split, int tp, tp_dtype wdt, const void* W,
                           const void* W_up, int64_t out_f, int64_t in_f,
                           const float* b, int n_heads, int n_kv_heads,
                           int head_dim, void* const* w_shards,
                           float* const* b_shards, tp_stream_t stream);

/*
 * column_parallel_linear -- Y_i = act(X . W_i^T + b_i) for every shard i, in
 * one launch; shard i writes columns [i*N/tp, (i+1)*N/tp) of Y, so the
 * concatenation of [P5] is the output layout itself.
 *
 * [P3] "How Tensor Parallelism Works Under the Hood" (column parallelism: the
 * full input X is shared, each shard computes a slice of the output) and
 * ColumnParallelLinear.forward; the nonlinearity applied per shard follows
 * the FFN demo of [P3] (h = gelu(ffn_up(x))).
 *
 *   M, K, N      tokens, input features, output features of the UNSHARDED
 *                layer (N % tp == 0).
 *   X            [M, K] (row stride ldx >= K), dtype xdt.
 *   w_shards     host array of tp device pointers; shard i is [N/tp, K]
 *                (TP_SPLIT_COLUMN) or, for TP_ACT_SWIGLU, the packed gate/up
 *                shard of TP_SPLIT_GATE_UP.  Same dtype as X.
 *   b_shards     host array of tp fp32 [N/tp] device pointers, or NULL for
 *                no bias.  Must be NULL for TP_ACT_SWIGLU.
 *   act          TP_ACT_NONE, TP_ACT_GELU_ERF or TP_ACT_SWIGLU.
 *   Y            [M, N] (row stride ldy >= N), dtype ydt.
 *   xdt / ydt    TP_BF16 in with TP_BF16 or TP_F32 out; TP_F32 in with
 *                TP_F32 out.
 * Errors: TP_ERR_NULL, TP_ERR_BAD_SHAPE, TP_ERR_NOT_DIVISIBLE, TP_ERR_DTYPE,
 * TP_ERR_ALIGNMENT, TP_ERR_UNSUPPORTED, TP_ERR_CUDA.
 */
tp_status column_parallel_linear(int tp, int64_t M, int64_t K, int64_t N,
                                 const void* X, int64_t ldx, tp_dtype xdt,
                                 const void* const* w_shards,
                                 const float* const* b_shards, tp_act act,
                                 void* Y, int64_t ldy, tp_dtype ydt,
                                 tp_stream_t stream);

/*
 * row_parallel_linear -- Y = sum_{i=0}^{tp-1} X_i . W_i^T + b, one fp32
 * accumulator walking the shards in order 0..tp-1, the bias added once after
 * the sum.  This is the all-reduce's arithmetic, done inside the kernel.
 *
 * [P3] "How Tensor Parallelism Works Under the Hood" (row parallelism: each
 * shard computes a partial sum, an all-reduce adds them) and
 * RowParallelLinear.forward (all_reduce SUM, then + bias); [P5] (sum, not
 * concatenate).  X_i is the shard-local input, i.e. columns
 * [i*K/tp, (i+1)*K/tp) of X (the output of the preceding column-parallel
 * layer needs no re-slicing).
 *
 *   M, K, N      tokens, input features, output features of the UNSHARDED
 *                layer (K % tp == 0).
 *   X            [M, K] (row stride ldx >= K), dtype xdt.
 *   w_shards     host array of tp device pointers; shard i is [N, K/tp]
 *                (TP_SPLIT_ROW), same dtype as X.
 *   b            fp32 [N] or NULL.
 *   Y            [M, N] (row stride ldy >= N), dtype ydt.
 * Errors: as column_parallel_linear.
 */
tp_status row_parallel_linear(int tp, int64_t M, int64_t K, int64_t N,
                              const void* X, int64_t ldx, tp_dtype xdt,
                              const void* const* w_shards, const float* b,
                              void* Y, int64_t ldy, tp_dtype ydt,
                              tp_stream_t stream);

/*
 * row_parallel_linear_ring -- row_parallel_linear with the shard sum done the
 * way a ring all-reduce adds the partials on real devices, instead of in one
 * fp32 accumulator.
 *
 * [P5] "Communication cost" (the ring all-reduce: the message is cut into tp
 * chunks; in the reduce-scatter each chunk's running sum travels once around
 * the ring, gaining one rank's partial per hop; the all-gather copies the
 * finished chunks); [P3] RowParallelLinear (all_reduce SUM of each rank's
 * local partial, then + bias).  Readings where the pages leave the arithmetic
 * open:
 *   - rank i's partial X_i . W_i^T is accumulated in fp32 and held in the
 *     wire dtype (bf16 rounded to nearest even, or fp32);
 *   - the flattened [M, N] message of L = M*N elements is cut into chunks
 *     c = [c*L/tp, (c+1)*L/tp) (integer division);
 *   - chunk c's sum starts with rank c's partial and adds ranks c+1, ...,
 *     c+tp-1 (mod tp), each addition in fp32 rounded to the wire dtype (every
 *     hop transmits the running sum in that dtype);
 *   - the bias is added once, after the all-reduce, in fp32; the result is
 *     rounded once to ydt.
 * With a bf16 wire this shows the rounding that a real bf16 all-reduce adds
 * on top of the fused single-accumulator sum.
 *
 *   M, K, N, X, ldx, xdt, w_shards, b, Y, ldy, ydt   as row_parallel_linear.
 *   wire_dt      TP_BF16 or TP_F32 (TP_F32 needs xdt == TP_F32 or TP_BF16;
 *                TP_BF16 needs xdt == TP_BF16).
 *   partials     caller-provided workspace [tp][M][N], contiguous, of dtype
 *                wire_dt; on return (stream order) it holds the partials.
 * Launches tp partial GEMMs and one reduction kernel.
 * Errors: as row_parallel_linear, and TP_ERR_NULL for partials.
 */
tp_status row_parallel_linear_ring(int tp, int64_t M, int64_t K, int64_t N,
                                   const void* X, int64_t ldx, tp_dtype xdt,
                                   const void* const* w_shards, const float* b,
                                   tp_dtype wire_dt, void* partials, void* Y,
                                   int64_t ldy, tp_dtype ydt,
                                   tp_stream_t stream);

/*
 * tp_shard_weights_uneven / column_parallel_linear_uneven -- the column split
 * with explicit per-shard output widths, e.g. 9 outputs as 5 + 4.
 *
 * [P5] "Try it yourself" (split 9 output features unevenly, 5 + 4; the
 * concatenation still equals the full product).  This relaxes the equal-width
 * assert of [P3]'s ColumnParallelLinear for the column side only.
 *
 *   widths       host array of tp widths, each >= 1; sum = out_f (= N).
 *   Sharding: shard i = rows [w_0 + ... + w_{i-1}, ... + w_i) of W, a
 *   contiguous [widths[i], in_f] buffer (and fp32 bias slice [widths[i]]).
 *   Compute: shard i writes columns [w_0 + ... + w_{i-1}, ...) of Y, with
 *   act TP_ACT_NONE or TP_ACT_GELU_ERF (TP_ACT_SWIGLU: TP_ERR_UNSUPPORTED).
 *   Each shard runs as a one-shard column call, so the result is bit-identical
 *   to the same call with tp = 1.
 *   Other arguments as tp_shard_weights / column_parallel_linear.
 * Errors: TP_ERR_NULL, TP_ERR_BAD_SHAPE (a width < 1, widths not summing to
 * out_f), TP_ERR_DTYPE, TP_ERR_ALIGNMENT, TP_ERR_UNSUPPORTED, TP_ERR_CUDA.
 */
tp_status tp_shard_weights_uneven(int tp, const int64_t* widths, tp_dtype wdt,
                                  const void* W, int64_t out_f, int64_t in_f,
                                  const float* b, void* const* w_shards,
                                  float* const* b_shards, tp_stream_t stream);
tp_status column_parallel_linear_uneven(int tp, const int64_t* widths, int64_t M,
                                        int64_t K, const void* X, int64_t ldx,
                                        tp_dtype xdt,
                                        const void* const* w_shards,
                                        const float* const* b_shards, tp_act act,
                                        void* Y, int64_t ldy, tp_dtype ydt,
                                        tp_stream_t stream);

/*
 * FP8 (e4m3) weights for decode-shaped calls -- half the weight bytes of bf16.
 *
 * "Model Parallelism" (statistical-learning-notes) sizes weights at about one
 * byte per parameter in FP8.  No page fixes the format or the scaling; this
 * library's reading:
 *   - e4m3 codes (4 exponent bits, bias 7, 3 mantissa bits, no infinities,
 *     largest finite value 448), one byte per weight, row-major like W;
 *   - one fp32 scale per weight row, s = max_k |W[r,k]| / 448 (1 for a row of
 *     zeros); code = W[r,k] / s rounded to nearest even, saturating at 448;
 *     the scale and the quotient are computed in fp32;
 *   - y = s * (x . q): the dot product runs in fp32 over the e4m3 values and is
 *     then multiplied by the row's scale; a row-parallel shard is quantized as
 *     its own [N, K/tp] matrix, so each shard's partial is scaled by its own s
 *     before the in-kernel shard sum, and the bias is added once.
 * Quantize the shards tp_shard_weights produces (for SwiGLU, the packed
 * gate/up shard: every packed row gets its own scale).  The compute calls take
 * bf16 activations and at most TP_FP8_MAX_TOKENS tokens (decode shapes: a
 * weight-streaming GEMV for one token; up to 32 tokens a tensor-core kernel
 * that multiplies the e4m3 codes by an exact three-plane e4m3 split of each
 * token; tensor-core kernels that widen the codes exactly to bf16 on chip for
 * more -- into tensor memory up to 64 tokens, into shared memory above;
 * larger M: TP_ERR_UNSUPPORTED); K (per shard for the row split) must be a
 * multiple of 16.  The column split stays
 * bit-identical to tp = 1.
 */
#define TP_FP8_MAX_TOKENS 128

/*
 * tp_quantize_fp8 -- per-row e4m3 quantization of a bf16 [rows, cols] device
 * matrix W (contiguous): Q[rows, cols] (uint8 e4m3 codes), scales[rows]
 * (fp32).  All device memory owned by the caller.
 * Errors: TP_ERR_BAD_SHAPE, TP_ERR_NULL, TP_ERR_ALIGNMENT, TP_ERR_CUDA.
 */
tp_status tp_quantize_fp8(int64_t rows, int64_t cols, const void* W, void* Q,
                          float* scales, tp_stream_t stream);

/*
 * column_parallel_linear_fp8 / row_parallel_linear_fp8 / tp_mlp_block_fp8 --
 * column_parallel_linear, row_parallel_linear and tp_mlp_block with FP8 weight
 * shards: q_shards[i] holds shard i's e4m3 codes (same shape as the bf16
 * shard), scale_shards[i] its fp32 row scales.  xdt must be TP_BF16 (X, and
 * h of the FFN block, are bf16); other arguments as the bf16 calls.
 * Errors: as the bf16 calls, TP_ERR_UNSUPPORTED for M > TP_FP8_MAX_TOKENS.
 */
tp_status column_parallel_linear_fp8(int tp, int64_t M, int64_t K, int64_t N,
                                     const void* X, int64_t ldx, tp_dtype xdt,
                                     const void* const* q_shards,
                                     const float* const* scale_shards,
                                     const float* const* b_shards, tp_act act,
                                     void* Y, int64_t ldy, tp_dtype ydt,
                                     tp_stream_t stream);
tp_status row_parallel_linear_fp8(int tp, int64_t M, int64_t K, int64_t N,
                                  const void* X, int64_t ldx, tp_dtype xdt,
                                  const void* const* q_shards,
                                  const float* const* scale_shards,
                                  const float* b, void* Y, int64_t ldy,
                                  tp_dtype ydt, tp_stream_t stream);
tp_status tp_mlp_block_fp8(int tp, int64_t M, int64_t d_model, int64_t d_ff,
                           tp_act act, const void* X,
                           const void* const* q1_shards,
                           const float* const* s1_shards,
                           const float* const* b1_shards,
                           const void* const* q2_shards,
                           const float* const* s2_shards, const float* b2,
                           void* h, void* Y, tp_dtype ydt, tp_stream_t stream);

/*
 * tp_mlp_block -- the tensor-parallel FFN block: column-parallel first linear
 * with the activation applied per shard, then row-parallel second linear whose
 * shard-i input is h_i, summed in the kernel, + b2 once.
 *
 * [P3] "How Tensor Parallelism Works Under the Hood" (the first FFN linear is
 * column-parallel, the second row-parallel, one synchronisation per block)
 * and its FFN demo; [P5] "Column-parallel and row-parallel layers, paired"
 * (the intermediate activation is never exchanged).
 *
 *   d_model, d_ff  layer widths; d_ff % tp == 0.
 *   act          TP_ACT_GELU_ERF (w1 shards from TP_SPLIT_COLUMN, optional
 *                b1 shards) or TP_ACT_SWIGLU (w1 shards from
 *                TP_SPLIT_GATE_UP, b1 must be NULL) or TP_ACT_NONE.
 *   X            [M, d_model] contiguous, dtype xdt.
 *   w2_shards    shard i is [d_model, d_ff/tp] (TP_SPLIT_ROW).
 *   b2           fp32 [d_model] or NULL.
 *   h            caller-provided workspace [M, d_ff] contiguous, dtype xdt
 *                (bf16 for bf16 inputs: the intermediate is stored in bf16).
 *                On return (stream order) it holds the activation.
 *   Y            [M, d_model] contiguous, dtype ydt.
 * Errors: as column_parallel_linear.
 */
tp_status tp_mlp_block(int tp, int64_t M, int64_t d_model, int64_t d_ff,
                       tp_act act, tp_dtype xdt, const void* X,
                       const void* const* w1_shards,
                       const float* const* b1_shards,
                       const void* const* w2_shards, const float* b2, void* h,
                       void* Y, tp_dtype ydt, tp_stream_t stream);

/*
 * tp_attn_proj -- the head-split attention projections: QKV column-parallel
 * by head group, O row-parallel by head with the shard sum in the kernel.
 * The attention core between them is not part of this call: ctx, the
 * attention output [M, n_heads*head_dim], is an input.
 *
 * [P4] "How a layer is split" (different attention heads go to different
 * GPUs) and "Why it helps when serving" (tp divides the head count); [P3]
 * "What Is Tensor Parallelism?" (one exchange after the attention
 * concatenation); [P5] "Column-parallel and row-parallel layers, paired" (one
 * all-reduce per attention block).
 *
 *   n_heads, n_kv_heads, head_dim   tp divides both head counts.
 *   X            [M, d_model] contiguous, dtype xdt.
 *   wqkv_shards  shard i from TP_SPLIT_QKV_HEADS: [(H+2Hkv)/tp*hd, d_model].
 *   bqkv_shards  host array of tp fp32 device pointers, or NULL.
 *   qkv_out      [tp][M][(H+2Hkv)/tp*hd] shard-major (what device i would
 *                hold: its Q heads, then its K head(s), then its V head(s)),
 *                dtype qkv_dt.
 *   ctx          [M, H*hd] contiguous, dtype xdt; shard i reads head columns
 *                [i*H/tp*hd, (i+1)*H/tp*hd).
 *   wo_shards    shard i from TP_SPLIT_ROW of W_o [d_model, H*hd]:
 *                [d_model, H/tp*hd].
 *   bo           fp32 [d_model] or NULL.
 *   Y            [M, d_model] contiguous, dtype ydt.
 * Errors: as column_parallel_linear.
 */
tp_status tp_attn_proj(int tp, int64_t M, int64_t d_model, int n_heads,
                       int n_kv_heads, int head_dim, tp_dtype xdt,
                       const void* X, const void* const* wqkv_shards,
                       const float* const* bqkv_shards, void* qkv_out,
                       tp_dtype qkv_dt, const void* ctx,
                       const void* const* wo_shards, const float* bo, void* Y,
                       tp_dtype ydt, tp_stream_t stream);

/*
 * tp_layer_args / tp_layer_forward -- the linear algebra of one transformer
 * layer in one call: the attention projections (QKV column-parallel by head
 * group, O row-parallel by head with the shard sum in the kernel), then the FFN
 * block (column-parallel with the activation per shard, row-parallel with the
 * shard sum).  Four launches on one stream, in that order; every argument of
 * all four is validated before the first one.
 *
 * [P4] "How a layer is split" and "Why it helps when serving" (the attention
 * heads and the FFN are split the same way in every layer; two all-reduces
 * per layer, one after each block); [P3] "How Tensor Parallelism Works Under
 * the Hood"; [P5] "Column-parallel and row-parallel layers, paired".
 *
 * The steps between the two blocks -- the attention core, residual additions,
 * normalisation -- are not part of this library, so their results are inputs:
 * ctx is the attention output, X_ffn the FFN block's input.  X_ffn may be
 * Y_attn itself (the FFN then reads the attention block's output; Y_attn must
 * then have dtype xdt).  The call captures into a CUDA graph like any other
 * sequence of launches (call it once before capturing, so that one-time set-up
 * happens outside the capture).
 *
 * Fields have the meaning, layout and alignment of the same arguments of
 * tp_attn_proj (tp .. attn_ydt) and tp_mlp_block (d_ff .. ffn_ydt); X and X_ffn
 * are [M, d_model].  Errors: as tp_attn_proj and tp_mlp_block, and
 * TP_ERR_NULL for a NULL args pointer.
 */
typedef struct {
  int tp;
  int64_t M, d_model;
  tp_dtype xdt;
  /* attention projections */
  int n_heads, n_kv_heads, head_dim;
  const void* X;
  const void* const* wqkv_shards;
  const float* const* bqkv_shards;
  void* qkv_out;
  tp_dtype qkv_dt;
  const void* ctx;
  const void* const* wo_shards;
  const float* bo;
  void* Y_attn;
  tp_dtype attn_ydt;
  /* FFN block */
  int64_t d_ff;
  tp_act ffn_act;
  const void* X_ffn;
  const void* const* w1_shards;
  const float* const* b1_shards;
  const void* const* w2_shards;
  const float* b2;
  void* h;
  void* Y_ffn;
  tp_dtype ffn_ydt;
} tp_layer_args;

tp_status tp_layer_forward(const tp_layer_args* args, tp_stream_t stream);

/*
 * Size in bytes of the workspace built into the library for
 * tp_mlp_block_noalloc (8 MiB).
 */
#define TP_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/*
 * tp_mlp_block_noalloc -- tp_mlp_block without a caller-provided workspace.
 *
 * No passage of the pages has a counterpart to this call; it exists for users
 * of this library.  tp_mlp_block needs a [M, d_ff] device workspace for the
 * intermediate activation h.  Some callers cannot allocate one: their device
 * memory belongs to another allocator (a serving engine that reserves the
 * GPU at start-up, a plugin whose host application hands out no device
 * memory), or cudaMalloc is off limits on their path because it can
 * synchronise the device and stall unrelated work.  This call keeps h in a
 * fixed buffer of TP_NOALLOC_SCRATCH_BYTES that is part of the library image:
 * every GPU that loads the library holds it until the process exits.  The call
 * itself allocates nothing (no cudaMalloc, no cudaFree).
 *
 *   Limit       M * d_ff * (2 for TP_BF16, 4 for TP_F32) <= TP_NOALLOC_SCRATCH_BYTES,
 *               e.g. up to 146 tokens at d_ff = 28672 in bf16.  Larger calls
 *               return TP_ERR_UNSUPPORTED and launch nothing.
 *   Set-up      every call looks up the buffer's device address on the
 *               current device (nothing is cached, so a device reset leaves
 *               no stale address behind).  The first call on a device may
 *               load the library's device code there: make that first call
 *               before any stream capture on the device.
 *   Sharing     every call on a device uses the same buffer, which keeps the
 *               last call's contents.  Nothing in it needs to start at zero:
 *               each call writes all of its h before reading it.  Calls that
 *               can run at the same time on the GPU (different streams with no
 *               ordering between them) race on the buffer and give wrong
 *               results: order them.
 *   Arguments, results and other errors: as tp_mlp_block, without h.
 */
tp_status tp_mlp_block_noalloc(int tp, int64_t M, int64_t d_model, int64_t d_ff,
                               tp_act act, tp_dtype xdt, const void* X,
                               const void* const* w1_shards,
                               const float* const* b1_shards,
                               const void* const* w2_shards, const float* b2,
                               void* Y, tp_dtype ydt, tp_stream_t stream);

/*
 * tp_device_status -- synchronise `stream`, then report and clear the
 * library's device-side error word on the current device.  Every spin-wait
 * inside the library's kernels is bounded; a wait that runs out sets this
 * word and the kernel returns early (its output is then incomplete).
 * Returns TP_OK, TP_ERR_DEVICE_TIMEOUT, or TP_ERR_CUDA if the stream itself
 * reports an error.  A checked build of the library (libtpla_checked.so,
 * compiled with TPLA_CHECKED) also checks the kernels' computed shared-memory,
 * tensor-memory and weight-row indices; a failed check skips the access and
 * is reported here as TP_ERR_DEVICE_CHECK.
 */
tp_status tp_device_status(tp_stream_t stream);

/*
 * tp_selftest_bounded_wait -- exercise the bounded-wait path: launch one
 * kernel that waits on a barrier nothing will ever complete, with a limit of
 * `limit_ns` nanoseconds (1 .. 10^10).  The kernel gives up, sets the device
 * error word and returns; tp_device_status then reports
 * TP_ERR_DEVICE_TIMEOUT and the context stays usable.  For tests.
 */
tp_status tp_selftest_bounded_wait(int64_t limit_ns, tp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TPLA_H */
